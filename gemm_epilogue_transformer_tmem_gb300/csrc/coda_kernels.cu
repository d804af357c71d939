// Small kernels around the fused GEMM: the deterministic finish of the
// cross-tile row reductions, the gamma fold of the commuted RMSNorm, and the
// unfused memory-bound kernels (RMSNorm, epilogue applied to a stored C) that
// the fused kernel replaces.
#include <cuda.h>
#include <cuda_runtime.h>

#include "coda_internal.h"
#include "coda_launch.h"
#include "coda_ops.cuh"
#include "coda_ptx.cuh"

namespace coda {

// Launch a kernel as the programmatic dependent of the previous kernel on the
// stream: it may be scheduled once that grid has signalled
// (griddepcontrol.launch_dependents) and begins with griddepcontrol.wait,
// which holds it until that grid has completed and its writes are visible.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), unsigned blocks, unsigned threads, cudaStream_t st,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- finalize
// row_stats[slot][i] = sum over column tiles of the partials, in tile order
// (deterministic), divided by the row width for ROW_MEAN; keep counts likewise.
__global__ void finalize_rows_kernel(const float* __restrict__ ws_red, const uint32_t* __restrict__ ws_keep,
                                     int M, int num_n_tiles, int n_red, RedInfo info, float inv_width,
                                     float* __restrict__ row_stats, uint32_t* __restrict__ keep_count) {
  griddep_wait();   // the fused kernel's partials (launched as its programmatic dependent)
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= M) return;
  const size_t Ms = static_cast<size_t>(M);
  for (int r = 0; r < n_red; ++r) {
    float s = 0.0f;
    const float* src = ws_red + static_cast<size_t>(r) * num_n_tiles * Ms + row;
    for (int t = 0; t < num_n_tiles; ++t) s += src[static_cast<size_t>(t) * Ms];
    if (info.is_mean[r]) s *= inv_width;
    row_stats[static_cast<size_t>(info.slot[r]) * Ms + row] = s;
  }
  if (keep_count != nullptr) {
    uint32_t k = 0;
    for (int t = 0; t < num_n_tiles; ++t) k += ws_keep[static_cast<size_t>(t) * Ms + row];
    keep_count[row] = k;
  }
}

cudaError_t launch_finalize(const float* ws_red, const uint32_t* ws_keep, int M, int num_n_tiles, int n_red,
                            const RedInfo& info, float inv_width, float* row_stats, uint32_t* keep_count,
                            cudaStream_t st) {
  const int threads = 256;
  const int blocks = (M + threads - 1) / threads;
  return launch_dependent(finalize_rows_kernel, blocks, threads, st, ws_red, ws_keep, M, num_n_tiles, n_red, info,
                          inv_width, row_stats, keep_count);
}

// Column reductions: col_stats[slot][j] = sum over the 32-row blocks of the
// partials (block order, deterministic); a thread per column, coalesced in j.
struct ColSlots {
  int32_t s[CODA_MAX_COL_REDUCTIONS];
};

__global__ void finalize_cols_kernel(const float* __restrict__ ws_col, int n_colred, int num_rb, int64_t n_out,
                                     ColSlots slots, float* __restrict__ col_stats) {
  griddep_wait();   // the fused kernel's partials (launched as its programmatic dependent)
  const int64_t j = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (j >= n_out) return;
  for (int r = 0; r < n_colred; ++r) {
    const float* src = ws_col + static_cast<size_t>(r) * num_rb * n_out + j;
    float acc = 0.0f;
    for (int b = 0; b < num_rb; ++b) acc += src[static_cast<size_t>(b) * n_out];
    col_stats[static_cast<size_t>(slots.s[r]) * n_out + j] = acc;
  }
}

cudaError_t launch_finalize_cols(const float* ws_col, int n_colred, int num_rb, int64_t n_out, const int32_t* slots,
                                 float* col_stats, cudaStream_t st) {
  ColSlots cs{};
  for (int r = 0; r < n_colred && r < CODA_MAX_COL_REDUCTIONS; ++r) cs.s[r] = slots[r];
  const int threads = 256;
  return launch_dependent(finalize_cols_kernel, static_cast<unsigned>((n_out + threads - 1) / threads), threads, st,
                          ws_col, n_colred, num_rb, n_out, cs, col_stats);
}

// ------------------------------------------------- commuted-norm row scales
// Row statistics of A for the commuted norms: the side path for CTA-pair tiles,
// run just before the GEMM as a full grid at memory bandwidth (a warp per row,
// eight 16-byte loads in flight per lane).  The GEMM is launched as its
// programmatic dependent, so its launch overlaps this kernel's tail and only
// its epilogue waits for the statistics.
//   RMSNorm:   r_i = rsqrt(sum_k a_ik^2 / K + eps)
//   LayerNorm: mu_i = sum_k a_ik / K,  r_i = rsqrt(sum_k (a_ik - mu_i)^2 / K + eps),
//              in one pass over data shifted by the row's first element
//              (the shifted-data variance of Chan, Golub & LeVeque, 1983):
//              with d = a - a_i0, var = sum d^2 / K - (sum d / K)^2, which
//              cancels only as far as the row's spread, not its mean.
// K % 8 == 0.
__device__ __forceinline__ float warp_row_sum(const uint4* ar, int64_t n8, int lane, float shift, bool squares) {
  float acc = 0.0f;
  int64_t i = lane;
  for (; i + 224 < n8; i += 256) {
    uint4 q[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) q[u] = __ldg(ar + i + 32 * u);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      float x[8];
      unpack8(q[u], x);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float d = x[j] - shift;
        acc = squares ? fmaf(d, d, acc) : acc + d;
      }
    }
  }
  for (; i < n8; i += 32) {
    float x[8];
    unpack8(__ldg(ar + i), x);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float d = x[j] - shift;
      acc = squares ? fmaf(d, d, acc) : acc + d;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  return acc;
}

// sum_k (a_k - shift) and sum_k (a_k - shift)^2 over one row, reduced over the warp
__device__ __forceinline__ void warp_row_moments(const uint4* ar, int64_t n8, int lane, float shift, float& s1,
                                                 float& s2) {
  float a1 = 0.0f, a2 = 0.0f;
  int64_t i = lane;
  for (; i + 224 < n8; i += 256) {
    uint4 q[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) q[u] = __ldg(ar + i + 32 * u);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      float x[8];
      unpack8(q[u], x);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float d = x[j] - shift;
        a1 += d;
        a2 = fmaf(d, d, a2);
      }
    }
  }
  for (; i < n8; i += 32) {
    float x[8];
    unpack8(__ldg(ar + i), x);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float d = x[j] - shift;
      a1 += d;
      a2 = fmaf(d, d, a2);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a1 += __shfl_xor_sync(0xFFFFFFFFu, a1, o);
    a2 += __shfl_xor_sync(0xFFFFFFFFu, a2, o);
  }
  s1 = a1;
  s2 = a2;
}

__global__ void __launch_bounds__(256) rms_rowscale_kernel(const uint16_t* __restrict__ A, int64_t M, int64_t K,
                                                           float inv_K, float eps, int layernorm,
                                                           float* __restrict__ r, float* __restrict__ r_copy,
                                                           float* __restrict__ mu, float* __restrict__ mu_copy) {
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t n8 = K >> 3;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); row < M;
       row += stride) {
    const uint4* ar = reinterpret_cast<const uint4*>(A + row * K);
    float m = 0.0f, ss;
    if (layernorm) {
      const float shift = __uint_as_float(static_cast<uint32_t>(__ldg(A + row * K)) << 16);
      float s1, s2;
      warp_row_moments(ar, n8, lane, shift, s1, s2);
      const float d = s1 * inv_K;
      m = shift + d;
      ss = fmaxf(s2 - s1 * d, 0.0f);   // sum (a - mu)^2
    } else {
      ss = warp_row_sum(ar, n8, lane, 0.0f, true);
    }
    if (lane == 0) {
      const float v = rsqrtf(fmaf(ss, inv_K, eps));
      r[row] = v;
      if (r_copy != nullptr) r_copy[row] = v;
      if (layernorm) {
        mu[row] = m;
        if (mu_copy != nullptr) mu_copy[row] = m;
      }
    }
  }
}

cudaError_t launch_rms_rowscale(const void* A, int64_t M, int64_t K, float inv_K, float eps, bool layernorm, float* r,
                                float* r_copy, float* mu, float* mu_copy, cudaStream_t st) {
  const int threads = 256;
  const int64_t blocks = (M + threads / 32 - 1) / (threads / 32);
  rms_rowscale_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(
      static_cast<const uint16_t*>(A), M, K, inv_K, eps, layernorm ? 1 : 0, r, r_copy, mu, mu_copy);
  return cudaGetLastError();
}

// ---------------------------------------------------- FP8 quantisation
// One warp per row: amax over the row, inv = 448 / amax and scale = amax / 448
// (IEEE fp32 divisions), then each element x * inv (fp32 product) converted
// to E4M3 with round-to-nearest-even and saturation (cvt.rn.satfinite).
// Sixteen elements (two 16-byte loads, one 16-byte store) per lane step.
__global__ void quantize_e4m3_rows_kernel(const uint16_t* __restrict__ X, int64_t M, int64_t K,
                                          uint8_t* __restrict__ Q, float* __restrict__ scale) {
  const int64_t row = blockIdx.x * static_cast<int64_t>(blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const uint4* xr = reinterpret_cast<const uint4*>(X + row * K);
  const int64_t n8 = K >> 3;
  float amax = 0.0f;
  for (int64_t i = lane; i < n8; i += 32) {
    float x[8];
    unpack8(__ldg(xr + i), x);
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(x[j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  const float inv = amax > 0.0f ? __fdiv_rn(448.0f, amax) : 0.0f;
  if (lane == 0) scale[row] = __fdiv_rn(amax, 448.0f);
  uint4* qr = reinterpret_cast<uint4*>(Q + row * K);
  for (int64_t i = lane; 2 * i < n8; i += 32) {
    float x[16];
    unpack8(__ldg(xr + 2 * i), x);
    unpack8(__ldg(xr + 2 * i + 1), x + 8);
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t lo = cvt_e4m3x2(__fmul_rn(x[4 * q], inv), __fmul_rn(x[4 * q + 1], inv));
      const uint32_t hi = cvt_e4m3x2(__fmul_rn(x[4 * q + 2], inv), __fmul_rn(x[4 * q + 3], inv));
      w[q] = lo | (hi << 16);
    }
    qr[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

cudaError_t launch_quantize_e4m3_rows(const void* X, int64_t M, int64_t K, void* Q, float* scale, cudaStream_t st) {
  const int threads = 256;
  const int64_t blocks = (M + threads / 32 - 1) / (threads / 32);
  quantize_e4m3_rows_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(
      static_cast<const uint16_t*>(X), M, K, static_cast<uint8_t*>(Q), scale);
  return cudaGetLastError();
}

// ------------------------------------------------------ MX E4M3 quantiser
// OCP Microscaling Formats (MX) v1.0: each block of 32 elements along K shares
// an E8M0 scale X = 2^(e - 127).  The shared exponent is floor(log2 amax) - 8
// (E4M3's largest normal is 1.75 * 2^8), clamped to the scale's range: with E
// the biased fp32 exponent field of the block maximum, e = max(E - 8, 0) (0 for
// a zero or subnormal-range maximum).  Codes e4m3(x * 2^(127 - e)), rounded to
// nearest even and saturated at 448; the product is exact wherever the code is
// not zero.  One thread per block of 32 (64 bytes in, 32 code bytes and one
// scale byte out); scales go to the tiled storage of coda.h, whose padding the
// caller set to 127 first.
__global__ void quantize_mx_e4m3_kernel(const uint16_t* __restrict__ X, int64_t R, int64_t K,
                                        uint8_t* __restrict__ Q, uint8_t* __restrict__ S) {
  const int64_t nb = K >> 5;
  const int64_t kbt = (nb + 3) >> 2;
  const int64_t total = R * nb;
  for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = t / nb;
    const int64_t j = t - r * nb;
    const uint4* src = reinterpret_cast<const uint4*>(X + r * K + j * 32);
    float x[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) unpack8(__ldg(src + q), x + 8 * q);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
    int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 8;
    if (e < 0) e = 0;
    const float mul = __uint_as_float(static_cast<uint32_t>(254 - e) << 23);   // 2^(127 - e), e <= 247
    uint32_t w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t lo = cvt_e4m3x2(__fmul_rn(x[4 * q], mul), __fmul_rn(x[4 * q + 1], mul));
      const uint32_t hi = cvt_e4m3x2(__fmul_rn(x[4 * q + 2], mul), __fmul_rn(x[4 * q + 3], mul));
      w[q] = lo | (hi << 16);
    }
    uint4* dst = reinterpret_cast<uint4*>(Q + r * K + j * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    S[((r >> 7) * kbt + (j >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (j & 3)] = static_cast<uint8_t>(e);
  }
}

cudaError_t launch_quantize_mx_e4m3(const void* X, int64_t R, int64_t K, void* Q, void* S, size_t s_bytes, int num_sms,
                                    cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(S, 127, s_bytes, st);   // padding: scale 1
  if (e != cudaSuccess) return e;
  const int threads = 256;
  const int64_t total = R * (K >> 5);
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  quantize_mx_e4m3_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(
      static_cast<const uint16_t*>(X), R, K, static_cast<uint8_t*>(Q), static_cast<uint8_t*>(S));
  return cudaGetLastError();
}

// --------------------------------------------------------- norm backward
// dX = r (g - sum_g / K - x_hat S / K), x_hat = (x - mu) r, S = r (sum_gx - mu sum_g);
// RMSNorm: mu = sum_g = null.  Eight elements per thread, grid-stride over the
// [M, K] tensors (K % 8 == 0), 16-byte loads and stores.
__global__ void norm_backward_kernel(const uint4* __restrict__ g, const uint4* __restrict__ X,
                                     const float* __restrict__ r, const float* __restrict__ mu,
                                     const float* __restrict__ sum_g, const float* __restrict__ sum_gx, int64_t M,
                                     int64_t K, float inv_K, uint4* __restrict__ dX) {
  const int64_t k8 = K >> 3;
  const int64_t total = M * k8;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = i / k8;
    const float rr = __ldg(r + row);
    const float m = mu ? __ldg(mu + row) : 0.0f;
    const float s1 = sum_g ? __ldg(sum_g + row) : 0.0f;
    const float S = rr * (__ldg(sum_gx + row) - m * s1);
    float gv[8], xv[8], out[8];
    unpack8(__ldg(g + i), gv);
    unpack8(__ldg(X + i), xv);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float xh = (xv[j] - m) * rr;
      out[j] = rr * (gv[j] - s1 * inv_K - xh * S * inv_K);
    }
    dX[i] = pack8(out);
  }
}

cudaError_t launch_norm_backward(const void* g, const void* X, const float* r, const float* mu, const float* sum_g,
                                 const float* sum_gx, int64_t M, int64_t K, void* dX, int num_sms, cudaStream_t st) {
  const int threads = 256;
  const int64_t work = M * (K >> 3);
  int64_t blocks = (work + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  norm_backward_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(
      static_cast<const uint4*>(g), static_cast<const uint4*>(X), r, mu, sum_g, sum_gx, M, K,
      static_cast<float>(1.0 / static_cast<double>(K)), static_cast<uint4*>(dX));
  return cudaGetLastError();
}

// ------------------------------------------------------ LayerNorm fold
// c_n = sum_k W'[k,n] over the folded bf16 weight, b_n = sum_k beta_k W[k,n]
// (fp32).  [K,N] layout: a thread per column n, coalesced along n.  [N,K]
// layout: a warp per row n.
__global__ void ln_colsum_kn_kernel(const uint16_t* __restrict__ Wf, const uint16_t* __restrict__ W,
                                    const uint16_t* __restrict__ beta, int64_t K, int64_t N, float* __restrict__ c,
                                    float* __restrict__ b) {
  const int64_t n = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (n >= N) return;
  float sc = 0.0f, sb = 0.0f;
  for (int64_t k = 0; k < K; ++k) {
    sc += __uint_as_float(static_cast<uint32_t>(__ldg(Wf + k * N + n)) << 16);
    if (beta != nullptr)
      sb = fmaf(__uint_as_float(static_cast<uint32_t>(__ldg(beta + k)) << 16),
                __uint_as_float(static_cast<uint32_t>(__ldg(W + k * N + n)) << 16), sb);
  }
  c[n] = sc;
  b[n] = sb;
}

__global__ void ln_colsum_nk_kernel(const uint16_t* __restrict__ Wf, const uint16_t* __restrict__ W,
                                    const uint16_t* __restrict__ beta, int64_t K, int64_t N, float* __restrict__ c,
                                    float* __restrict__ b) {
  const int64_t n = blockIdx.x * static_cast<int64_t>(blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (n >= N) return;
  const uint4* wf = reinterpret_cast<const uint4*>(Wf + n * K);
  const uint4* w = reinterpret_cast<const uint4*>(W + n * K);
  const uint4* bt = reinterpret_cast<const uint4*>(beta);
  float sc = 0.0f, sb = 0.0f;
  for (int64_t i = lane; i < (K >> 3); i += 32) {
    float x[8];
    unpack8(__ldg(wf + i), x);
#pragma unroll
    for (int j = 0; j < 8; ++j) sc += x[j];
    if (beta != nullptr) {
      float y[8], g[8];
      unpack8(__ldg(w + i), y);
      unpack8(__ldg(bt + i), g);
#pragma unroll
      for (int j = 0; j < 8; ++j) sb = fmaf(g[j], y[j], sb);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sc += __shfl_xor_sync(0xFFFFFFFFu, sc, o);
    sb += __shfl_xor_sync(0xFFFFFFFFu, sb, o);
  }
  if (lane == 0) {
    c[n] = sc;
    b[n] = sb;
  }
}

cudaError_t launch_ln_colsum(const void* W_folded, const void* W, const void* beta, int64_t K, int64_t N, bool kn,
                             float* c, float* b, cudaStream_t st) {
  if (kn) {
    const int threads = 256;
    ln_colsum_kn_kernel<<<static_cast<unsigned>((N + threads - 1) / threads), threads, 0, st>>>(
        static_cast<const uint16_t*>(W_folded), static_cast<const uint16_t*>(W), static_cast<const uint16_t*>(beta),
        K, N, c, b);
  } else {
    const int threads = 256;
    ln_colsum_nk_kernel<<<static_cast<unsigned>((N + 7) / 8), threads, 0, st>>>(
        static_cast<const uint16_t*>(W_folded), static_cast<const uint16_t*>(W), static_cast<const uint16_t*>(beta),
        K, N, c, b);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------- unfused LayerNorm
// One warp per row: mean, centred variance (two passes), then
// Xn = bf16(gamma * (x - mu) * r + beta).  K % 8 == 0.
__global__ void layernorm_kernel(const uint16_t* __restrict__ X, const uint16_t* __restrict__ gamma,
                                 const uint16_t* __restrict__ beta, int64_t M, int64_t K, float eps,
                                 uint16_t* __restrict__ Xn) {
  const int64_t row = blockIdx.x * static_cast<int64_t>(blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const uint4* xr = reinterpret_cast<const uint4*>(X + row * K);
  const int64_t n8 = K >> 3;
  const float inv_K = 1.0f / static_cast<float>(K);
  const float m = warp_row_sum(xr, n8, lane, 0.0f, false) * inv_K;
  const float r = rsqrtf(fmaf(warp_row_sum(xr, n8, lane, m, true), inv_K, eps));
  uint4* yr = reinterpret_cast<uint4*>(Xn + row * K);
  const uint4* gr = reinterpret_cast<const uint4*>(gamma);
  const uint4* br = reinterpret_cast<const uint4*>(beta);
  for (int64_t i = lane; i < n8; i += 32) {
    float x[8], g[8], bb[8], y[8];
    unpack8(__ldg(xr + i), x);
    unpack8(__ldg(gr + i), g);
    if (beta != nullptr) {
      unpack8(__ldg(br + i), bb);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) bb[j] = 0.0f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] = fmaf(g[j] * (x[j] - m), r, bb[j]);
    yr[i] = pack8(y);
  }
}

cudaError_t launch_layernorm(const void* X, const void* gamma, const void* beta, int64_t M, int64_t K, float eps,
                             void* Xn, cudaStream_t st) {
  const int threads = 256;
  const int64_t blocks = (M + 7) / 8;
  layernorm_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(
      static_cast<const uint16_t*>(X), static_cast<const uint16_t*>(gamma), static_cast<const uint16_t*>(beta), M, K,
      eps, static_cast<uint16_t*>(Xn));
  return cudaGetLastError();
}

// -------------------------------------------------------------- gamma fold
// W_out[k,n] = bf16(gamma[k] * W[k,n]) ([K,N] layout) or W_out[n,k] = bf16(gamma[k]
// * W[n,k]) ([N,K] layout); 8 elements (16 bytes) per thread, grid-stride.
template <bool kKN>
__global__ void fold_gamma_kernel(const uint16_t* __restrict__ W, const uint16_t* __restrict__ gamma,
                                  uint16_t* __restrict__ W_out, int64_t K, int64_t N) {
  const int64_t total8 = (K * N) >> 3;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = i << 3;
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(W) + i);
    float w[8], o[8];
    unpack8(q, w);
    if (kKN) {
      const int64_t k = e / N;   // N % 8 == 0: the 8 elements share a row k
      const float g = __uint_as_float(static_cast<uint32_t>(__ldg(gamma + k)) << 16);
#pragma unroll
      for (int j = 0; j < 8; ++j) o[j] = w[j] * g;
    } else {
      const int64_t k0 = e % K;  // K % 8 == 0: columns k0 .. k0+7 of one row n
      float g[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(gamma + k0)), g);
#pragma unroll
      for (int j = 0; j < 8; ++j) o[j] = w[j] * g[j];
    }
    reinterpret_cast<uint4*>(W_out)[i] = pack8(o);
  }
}

cudaError_t launch_fold_gamma(const void* W, const void* gamma, void* W_out, int64_t K, int64_t N, bool kn,
                              int num_sms, cudaStream_t st) {
  const int threads = 256;
  const int64_t total8 = (K * N) >> 3;
  int64_t blocks = (total8 + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (kn)
    fold_gamma_kernel<true><<<static_cast<int>(blocks), threads, 0, st>>>(
        static_cast<const uint16_t*>(W), static_cast<const uint16_t*>(gamma), static_cast<uint16_t*>(W_out), K, N);
  else
    fold_gamma_kernel<false><<<static_cast<int>(blocks), threads, 0, st>>>(
        static_cast<const uint16_t*>(W), static_cast<const uint16_t*>(gamma), static_cast<uint16_t*>(W_out), K, N);
  return cudaGetLastError();
}

// ------------------------------------------------------- unfused RMSNorm
// One warp per row: sum of squares in fp32, r = rsqrt(ss/K + eps), then
// Xn = bf16(r * x * gamma).  K % 8 == 0.
__global__ void rmsnorm_kernel(const uint16_t* __restrict__ X, const uint16_t* __restrict__ gamma, int64_t M,
                               int64_t K, float eps, uint16_t* __restrict__ Xn, float* __restrict__ rstd) {
  const int64_t row = blockIdx.x * static_cast<int64_t>(blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const uint4* xr = reinterpret_cast<const uint4*>(X + row * K);
  const int64_t n8 = K >> 3;
  float ss = 0.0f;
  for (int64_t i = lane; i < n8; i += 32) {
    float x[8];
    unpack8(__ldg(xr + i), x);
#pragma unroll
    for (int j = 0; j < 8; ++j) ss = fmaf(x[j], x[j], ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  const float r = rsqrtf(ss / static_cast<float>(K) + eps);
  if (lane == 0 && rstd != nullptr) rstd[row] = r;
  uint4* yr = reinterpret_cast<uint4*>(Xn + row * K);
  const uint4* gr = reinterpret_cast<const uint4*>(gamma);
  for (int64_t i = lane; i < n8; i += 32) {
    float x[8], g[8], y[8];
    unpack8(__ldg(xr + i), x);
    unpack8(__ldg(gr + i), g);
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] = r * x[j] * g[j];
    yr[i] = pack8(y);
  }
}

cudaError_t launch_rmsnorm(const void* X, const void* gamma, int64_t M, int64_t K, float eps, void* Xn,
                           float* rstd, cudaStream_t st) {
  const int threads = 256;
  const int64_t blocks = (M + 7) / 8;
  rmsnorm_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(
      static_cast<const uint16_t*>(X), static_cast<const uint16_t*>(gamma), M, K, eps, static_cast<uint16_t*>(Xn),
      rstd);
  return cudaGetLastError();
}

// ------------------------------------------- unfused epilogue application
// Aux values for 8 consecutive columns straight from global memory.
struct GmemAux {
  const uint16_t* const* ptr;   // aux tensors by staging index
  size_t off;                   // element offset of (row, col)
  __device__ __forceinline__ void load(int k, float (&out)[8]) const {
    unpack8(__ldg(reinterpret_cast<const uint4*>(ptr[k] + off)), out);
  }
};

struct ApplyParams {
  int64_t M;
  int32_t N;       // input width
  int32_t N_out;   // output width
  int32_t half;    // SwiGLU: U offset in the input
  const uint16_t* aux[kMaxAux];
  float* row_stats;
  uint32_t* keep_count;
  EpiProgram prog;
};

// One warp per row; each lane handles 8 consecutive columns per step (16-byte
// loads and stores), row reductions finished by warp shuffles.
template <bool kGLU>
__global__ void epilogue_apply_kernel(const uint16_t* __restrict__ C, uint16_t* __restrict__ D,
                                      const __grid_constant__ ApplyParams ap) {
  const int64_t row = blockIdx.x * static_cast<int64_t>(blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= ap.M) return;
  float red[CODA_MAX_REDUCTIONS] = {0.0f, 0.0f, 0.0f, 0.0f};
  uint32_t keep = 0;
  const uint16_t* crow = C + row * ap.N;
  uint16_t* drow = D + row * ap.N_out;
  for (int col = lane * 8; col < ap.N_out; col += 256) {
    float v[8], u[8];
    unpack8(__ldg(reinterpret_cast<const uint4*>(crow + col)), v);
    if (kGLU) unpack8(__ldg(reinterpret_cast<const uint4*>(crow + ap.half + col)), u);
    const RowCtx rc{static_cast<int>(row), true, col, 8, ap.half, ap.N_out, static_cast<int>(ap.M), 1.0f};
    const GmemAux ax{ap.aux, static_cast<size_t>(row) * ap.N_out + col};
    run_ops<8, kGLU>(ap.prog, v, u, rc, ax, red, keep);
    *reinterpret_cast<uint4*>(drow + col) = pack8(v);
  }
  for (int r = 0; r < ap.prog.n_red; ++r) {
    float s = red[0];
    if (r == 1) s = red[1];
    if (r == 2) s = red[2];
    if (r == 3) s = red[3];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    if (lane == 0) {
      if (ap.prog.red.is_mean[r]) s /= static_cast<float>(ap.N_out);
      ap.row_stats[static_cast<size_t>(ap.prog.red.slot[r]) * ap.M + row] = s;
    }
  }
  if (ap.keep_count != nullptr) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) keep += __shfl_xor_sync(0xFFFFFFFFu, keep, o);
    if (lane == 0) ap.keep_count[row] = keep;
  }
}

cudaError_t launch_epilogue_apply(const void* C, void* D, int64_t M, int N, int N_out, int half,
                                  const void* const* aux, float* row_stats, uint32_t* keep_count,
                                  const EpiProgram& prog, cudaStream_t st) {
  ApplyParams ap{};
  ap.M = M;
  ap.N = N;
  ap.N_out = N_out;
  ap.half = half;
  for (int k = 0; k < kMaxAux; ++k) ap.aux[k] = static_cast<const uint16_t*>(aux[k]);
  ap.row_stats = row_stats;
  ap.keep_count = keep_count;
  ap.prog = prog;
  const int threads = 256;
  const int64_t blocks = (M + 7) / 8;
  if (prog.glu_pos >= 0)
    epilogue_apply_kernel<true><<<static_cast<unsigned>(blocks), threads, 0, st>>>(
        static_cast<const uint16_t*>(C), static_cast<uint16_t*>(D), ap);
  else
    epilogue_apply_kernel<false><<<static_cast<unsigned>(blocks), threads, 0, st>>>(
        static_cast<const uint16_t*>(C), static_cast<uint16_t*>(D), ap);
  return cudaGetLastError();
}

}  // namespace coda
