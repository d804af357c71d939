// Device-side epilogue op interpreter.
//
// The CODA article (d9bl.com, §3.1) applies an epilogue f elementwise or row by
// row to the GEMM output tile before it is written; agentlenshq.com ("仕組み")
// builds f from scaling, reduction, elementwise-transform and accumulation
// primitives.  Here f is an op list run in order on NE consecutive fp32 values
// of one output row held in registers.  With SwiGLU the thread also holds the U
// values paired with its G values; ops before the SWIGLU op act on both.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "coda_internal.h"

namespace coda {

constexpr float kSqrt2OverPi = 0.7978845608028654f;
constexpr float kGeluC = 0.044715f;
constexpr uint64_t kSplitmixGamma = 0x9E3779B97F4A7C15ull;

// The logistic function and the activations built on it.  The epilogue has one
// warp per scheduler and little to hide latency behind, and the special-function
// unit is its busiest pipe (SiLU and GELU took two of its operations per element
// with an exponential and a reciprocal).  So the logistic function is taken from
// the hardware tanh (PTX tanh.approx.f32, one operation, relative error about
// 2^-11):  sigmoid(x) = (1 + tanh(x/2)) / 2,  1 - sigmoid(x) = (1 - tanh(x/2)) / 2.
// Its absolute error is at most 2^-12 (about 2.4e-4): SiLU and GELU carry at
// most 2.4e-4 |x|, below the bf16 rounding of the output (2^-9 to 2^-8) where
// the output is not near zero; in the negative tail, where sigmoid(x) itself is
// below 1e-3, the error is absolute, not relative.  tanh saturates to +-1, so
// no argument overflows.
__device__ __forceinline__ float tanh_hw(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float sigmoid_f(float x, float& one_minus) {
  const float t = tanh_hw(0.5f * x);
  one_minus = fmaf(-0.5f, t, 0.5f);
  return fmaf(0.5f, t, 0.5f);
}

__device__ __forceinline__ float silu_f(float x) {
  float om;
  return x * sigmoid_f(x, om);
}

// tanh-form GELU: 0.5 x (1 + tanh(u)) with u = sqrt(2/pi) (x + 0.044715 x^3);
// since (1 + tanh(u)) / 2 = sigmoid(2u), this is x sigmoid(2u)
__device__ __forceinline__ float gelu_tanh_f(float x) {
  const float u = kSqrt2OverPi * fmaf(kGeluC * x * x, x, x);
  float om;
  return x * sigmoid_f(2.0f * u, om);
}

// derivative of gelu_tanh_f: 0.5 (1 + t) + 0.5 z (1 - t^2) u'(z) with t = tanh(u);
// with s = sigmoid(2u): (1 + t) / 2 = s and 1 - t^2 = 4 s (1 - s), so the
// derivative is s + 2 z s (1 - s) u'(z), free of the cancellation in 1 - t^2
__device__ __forceinline__ float gelu_tanh_grad_f(float z) {
  // constants folded: u = z (c + c k z^2), 2 u'(z) = 2 c + 6 c k z^2 (c = sqrt(2/pi), k = 0.044715)
  constexpr float kC1 = kSqrt2OverPi * kGeluC;
  const float z2 = z * z;
  const float u = z * fmaf(kC1, z2, kSqrt2OverPi);
  const float du2 = fmaf(6.0f * kC1, z2, 2.0f * kSqrt2OverPi);
  const float t = tanh_hw(u);                    // sigmoid(2u) = (1 + tanh(u)) / 2
  const float s = fmaf(0.5f, t, 0.5f);
  const float om = fmaf(-0.5f, t, 0.5f);
  return fmaf(z * du2, s * om, s);
}

// exact GELU: x * Phi(x), Phi the standard normal distribution function
__device__ __forceinline__ float gelu_erf_f(float x) { return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f)); }

// its derivative: Phi(z) + z * phi(z)
__device__ __forceinline__ float gelu_erf_grad_f(float z) {
  const float cdf = 0.5f * (1.0f + erff(z * 0.70710678118654752f));
  const float pdf = 0.39894228040143268f * expf(-0.5f * z * z);
  return fmaf(z, pdf, cdf);
}

// splitmix64 output function (Steele, Lea & Flood, OOPSLA 2014)
__device__ __forceinline__ uint64_t splitmix_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4 q, float* out) {
  out[0] = bf16_lo(q.x); out[1] = bf16_hi(q.x);
  out[2] = bf16_lo(q.y); out[3] = bf16_hi(q.y);
  out[4] = bf16_lo(q.z); out[5] = bf16_hi(q.z);
  out[6] = bf16_lo(q.w); out[7] = bf16_hi(q.w);
}

// round-to-nearest-even pack of two floats into a bf16x2 word
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint4 pack8(const float* v) {
  uint4 q;
  q.x = pack_bf16x2(v[0], v[1]);
  q.y = pack_bf16x2(v[2], v[3]);
  q.z = pack_bf16x2(v[4], v[5]);
  q.w = pack_bf16x2(v[6], v[7]);
  return q;
}

// NE values of a bf16 vector starting at `col`; entries at or past `width` read 0.
template <int NE>
__device__ __forceinline__ void load_colvec(const uint16_t* vec, int col, int width, float (&out)[NE]) {
  if (col + NE <= width) {
#pragma unroll
    for (int i = 0; i < NE / 8; ++i) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(vec + col) + i);
      unpack8(q, out + 8 * i);
    }
  } else {
#pragma unroll
    for (int j = 0; j < NE; ++j)
      out[j] = (col + j < width) ? __uint_as_float(static_cast<uint32_t>(__ldg(vec + col + j)) << 16) : 0.0f;
  }
}

// NE values of an fp32 vector starting at `col` (0 past `width` or for a null vector).
template <int NE>
__device__ __forceinline__ void load_colvec_f32(const float* vec, int col, int width, float (&out)[NE]) {
  if (vec == nullptr) {
#pragma unroll
    for (int j = 0; j < NE; ++j) out[j] = 0.0f;
  } else if (col + NE <= width) {
#pragma unroll
    for (int i = 0; i < NE / 4; ++i) {
      const float4 q = __ldg(reinterpret_cast<const float4*>(vec + col) + i);
      out[4 * i] = q.x;
      out[4 * i + 1] = q.y;
      out[4 * i + 2] = q.z;
      out[4 * i + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < NE; ++j) out[j] = (col + j < width) ? __ldg(vec + col + j) : 0.0f;
  }
}

template <int NE>
__device__ __forceinline__ void store_row_bf16(uint16_t* dst, int col, int width, const float (&v)[NE]) {
  if (col + NE <= width) {
#pragma unroll
    for (int i = 0; i < NE / 8; ++i) reinterpret_cast<uint4*>(dst + col)[i] = pack8(v + 8 * i);
  } else {
#pragma unroll
    for (int j = 0; j < NE; ++j)
      if (col + j < width) {
        const __nv_bfloat16 h = __float2bfloat16_rn(v[j]);
        dst[col + j] = *reinterpret_cast<const uint16_t*>(&h);
      }
  }
}

__device__ __forceinline__ void add_red(float (&red)[CODA_MAX_REDUCTIONS], int idx, float s) {
  if (idx == 0) red[0] += s;
  else if (idx == 1) red[1] += s;
  else if (idx == 2) red[2] += s;
  else red[3] += s;
}

// Sums of 32 columns over the 32 rows (lanes) of a warp: after five rounds of
// exchanging half of the remaining columns with the lane `s` apart and adding,
// a[0] of lane l holds the sum over all lanes of column l (31 shuffles).
__device__ __forceinline__ void warp_column_sums(float (&a)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = upper ? a[i] : a[i + s];
      const float keep = upper ? a[i + s] : a[i];
      a[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, s);
    }
  }
}

// Where the row values of one output row live for this run of NE columns.
struct RowCtx {
  int row;          // absolute output row
  bool row_ok;      // row < M
  int col;          // first output column of the run
  int nvalid;       // columns of the run that are < N_out (0..NE)
  int half;         // SwiGLU: column offset of U in the GEMM output (N/2)
  int n_out;        // output width
  int M;
  float r_rms;      // commuted-norm row scale of this row
  float mu;         // commuted-LayerNorm row mean of this row
  const float* cvs; // this run's first column in the warp's staged column-vector slices
                    // (slice k at cvs + k * cv_stride), or null: read them from global memory
  int cv_stride;
};

// NE staged fp32 values (shared memory, 16-byte aligned; the same address in
// every lane, so each load is a broadcast)
template <int NE>
__device__ __forceinline__ void load_staged(const float* s, float (&out)[NE]) {
#pragma unroll
  for (int i = 0; i < NE / 4; ++i) {
    const float4 q = reinterpret_cast<const float4*>(s)[i];
    out[4 * i] = q.x;
    out[4 * i + 1] = q.y;
    out[4 * i + 2] = q.z;
    out[4 * i + 3] = q.w;
  }
}

// One op of the list applied to v (and, before SWIGLU, to u: `pre`), with the
// opcode fixed at compile time.  Both the op-list interpreter below and the
// fixed op sequences call this, so every op has one implementation.
// `aux.load(k, out)` fills NE values of aux tensor k for this run.
template <uint32_t CODE, int NE, bool kGLU, class Aux>
__device__ __forceinline__ void op_apply(const EpiProgram& P, const DevOp& op, bool pre, float (&v)[NE], float (&u)[NE],
                                         const RowCtx& c, const Aux& aux, float (&red)[CODA_MAX_REDUCTIONS],
                                         uint32_t& keep_cnt) {
  switch (CODE) {
    case CODA_OP_SCALE: {
#pragma unroll
      for (int j = 0; j < NE; ++j) v[j] *= op.f0;
      if (pre) {
#pragma unroll
        for (int j = 0; j < NE; ++j) u[j] *= op.f0;
      }
      break;
    }
    case CODA_OP_COL_SCALE:
    case CODA_OP_BIAS: {
      const uint16_t* vec = P.col_vec[op.slot];
      const bool staged = c.cvs != nullptr && op.cv >= 0;
      float cv[NE];
      if (staged)
        load_staged<NE>(c.cvs + op.cv * c.cv_stride, cv);
      else
        load_colvec<NE>(vec, c.col, c.n_out, cv);
      constexpr bool is_bias = CODE == CODA_OP_BIAS;
      if constexpr (is_bias) {
#pragma unroll
        for (int j = 0; j < NE; ++j) v[j] += cv[j];
      } else {
#pragma unroll
        for (int j = 0; j < NE; ++j) v[j] *= cv[j];
      }
      if (pre) {
        if (staged)
          load_staged<NE>(c.cvs + (op.cv + 1) * c.cv_stride, cv);
        else
          load_colvec<NE>(vec + c.half, c.col, c.n_out, cv);
        if constexpr (is_bias) {
#pragma unroll
          for (int j = 0; j < NE; ++j) u[j] += cv[j];
        } else {
#pragma unroll
          for (int j = 0; j < NE; ++j) u[j] *= cv[j];
        }
      }
      break;
    }
    case CODA_OP_COL_SCALE_F32: {
      const bool staged = c.cvs != nullptr && op.cv >= 0;
      float cv[NE];
      if (staged)
        load_staged<NE>(c.cvs + op.cv * c.cv_stride, cv);
      else
        load_colvec_f32<NE>(P.col_scale_f32, c.col, c.n_out, cv);
#pragma unroll
      for (int j = 0; j < NE; ++j) v[j] *= cv[j];
      if (pre) {
        if (staged)
          load_staged<NE>(c.cvs + (op.cv + 1) * c.cv_stride, cv);
        else
          load_colvec_f32<NE>(P.col_scale_f32 + c.half, c.col, c.n_out, cv);
#pragma unroll
        for (int j = 0; j < NE; ++j) u[j] *= cv[j];
      }
      break;
    }
    case CODA_OP_ROW_SCALE:
    case CODA_OP_RMS_ROWSCALE: {
      const float s = (CODE == CODA_OP_RMS_ROWSCALE) ? c.r_rms
                      : (c.row_ok ? __ldg(P.row_vec[op.slot] + c.row) : 0.0f);
#pragma unroll
      for (int j = 0; j < NE; ++j) v[j] *= s;
      if (pre) {
#pragma unroll
        for (int j = 0; j < NE; ++j) u[j] *= s;
      }
      break;
    }
    case CODA_OP_LN_ROWSCALE: {
      // r (x - mu c_j) + b_j; staged slices: c (and its up half before
      // SWIGLU), then b (likewise) where the op has one
      const bool staged = c.cvs != nullptr && op.cv >= 0;
      const int nc = pre ? 2 : 1;
      float cv[NE], bv[NE];
      if (staged) {
        load_staged<NE>(c.cvs + op.cv * c.cv_stride, cv);
        if (P.ln_bias != nullptr) {
          load_staged<NE>(c.cvs + (op.cv + nc) * c.cv_stride, bv);
        } else {
#pragma unroll
          for (int j = 0; j < NE; ++j) bv[j] = 0.0f;
        }
      } else {
        load_colvec_f32<NE>(P.ln_colsum, c.col, c.n_out, cv);
        load_colvec_f32<NE>(P.ln_bias, c.col, c.n_out, bv);
      }
#pragma unroll
      for (int j = 0; j < NE; ++j) v[j] = fmaf(c.r_rms, fmaf(-c.mu, cv[j], v[j]), bv[j]);
      if (pre) {
        if (staged) {
          load_staged<NE>(c.cvs + (op.cv + 1) * c.cv_stride, cv);
          if (P.ln_bias != nullptr) load_staged<NE>(c.cvs + (op.cv + 3) * c.cv_stride, bv);
        } else {
          load_colvec_f32<NE>(P.ln_colsum ? P.ln_colsum + c.half : nullptr, c.col, c.n_out, cv);
          load_colvec_f32<NE>(P.ln_bias ? P.ln_bias + c.half : nullptr, c.col, c.n_out, bv);
        }
#pragma unroll
        for (int j = 0; j < NE; ++j) u[j] = fmaf(c.r_rms, fmaf(-c.mu, cv[j], u[j]), bv[j]);
      }
      break;
    }
    case CODA_OP_GELU_TANH: {
#pragma unroll
      for (int j = 0; j < NE; ++j) v[j] = gelu_tanh_f(v[j]);
      if (pre) {
#pragma unroll
        for (int j = 0; j < NE; ++j) u[j] = gelu_tanh_f(u[j]);
      }
      break;
    }
    case CODA_OP_GELU_ERF: {
#pragma unroll
      for (int j = 0; j < NE; ++j) v[j] = gelu_erf_f(v[j]);
      if (pre) {
#pragma unroll
        for (int j = 0; j < NE; ++j) u[j] = gelu_erf_f(u[j]);
      }
      break;
    }
    case CODA_OP_GELU_ERF_GRAD: {
      float z[NE];
      aux.load(op.aux, z);
#pragma unroll
      for (int j = 0; j < NE; ++j) v[j] *= gelu_erf_grad_f(z[j]);
      break;
    }
    case CODA_OP_SILU: {
#pragma unroll
      for (int j = 0; j < NE; ++j) v[j] = silu_f(v[j]);
      if (pre) {
#pragma unroll
        for (int j = 0; j < NE; ++j) u[j] = silu_f(u[j]);
      }
      break;
    }
    case CODA_OP_SWIGLU: {
      if (kGLU) {
#pragma unroll
        for (int j = 0; j < NE; ++j) v[j] = silu_f(v[j]) * u[j];
      }
      break;
    }
    case CODA_OP_GELU_TANH_GRAD: {
      float z[NE];
      aux.load(op.aux, z);
#pragma unroll
      for (int j = 0; j < NE; ++j) v[j] *= gelu_tanh_grad_f(z[j]);
      break;
    }
    case CODA_OP_DROPOUT: {
      // element (row, col + j) is output n = row*N_out + col + j of the stream
      const uint64_t n0 = static_cast<uint64_t>(c.row) * static_cast<uint64_t>(c.n_out) +
                          static_cast<uint64_t>(c.col);
      uint64_t state = P.seed + (n0 + 1ull) * kSplitmixGamma;
      const bool keep_all = op.f0 == 0.0f;
      uint32_t kc = 0;
#pragma unroll
      for (int j = 0; j < NE; ++j) {
        const bool keep = keep_all || (splitmix_mix(state) < op.u);
        state += kSplitmixGamma;
        v[j] = keep ? v[j] * op.f1 : 0.0f;
        kc += (keep && j < c.nvalid) ? 1u : 0u;
      }
      keep_cnt += kc;
      break;
    }
    case CODA_OP_RESIDUAL: {
      float r[NE];
      aux.load(op.aux, r);
#pragma unroll
      for (int j = 0; j < NE; ++j) v[j] = fmaf(op.f0, r[j], v[j]);
      break;
    }
    case CODA_OP_STORE_PREACT: {
      if (c.row_ok) {
        uint16_t* base = P.preact + static_cast<size_t>(c.row) * static_cast<size_t>(P.preact_width);
        store_row_bf16<NE>(base, c.col, c.n_out, v);
        if (pre) store_row_bf16<NE>(base + c.half, c.col, c.n_out, u);
      }
      break;
    }
    case CODA_OP_ROW_SUM:
    case CODA_OP_ROW_MEAN: {
      float s = 0.0f;
      if (c.nvalid >= NE) {   // a whole chunk: no per-element masks
#pragma unroll
        for (int j = 0; j < NE; ++j) s += v[j];
      } else {
#pragma unroll
        for (int j = 0; j < NE; ++j) s += (j < c.nvalid) ? v[j] : 0.0f;
      }
      add_red(red, op.red, s);
      break;
    }
    case CODA_OP_ROW_SUMSQ: {
      float s = 0.0f;
      if (c.nvalid >= NE) {
#pragma unroll
        for (int j = 0; j < NE; ++j) s += v[j] * v[j];
      } else {
#pragma unroll
        for (int j = 0; j < NE; ++j) s += (j < c.nvalid) ? v[j] * v[j] : 0.0f;
      }
      add_red(red, op.red, s);
      break;
    }
    case CODA_OP_ROW_DOT_AUX: {
      float x[NE];
      aux.load(op.aux, x);
      float s = 0.0f;
      if (c.nvalid >= NE) {
#pragma unroll
        for (int j = 0; j < NE; ++j) s += v[j] * x[j];
      } else {
#pragma unroll
        for (int j = 0; j < NE; ++j) s += (j < c.nvalid) ? v[j] * x[j] : 0.0f;
      }
      add_red(red, op.red, s);
      break;
    }
    case CODA_OP_COL_SUM:
    case CODA_OP_COL_SUMSQ:
    case CODA_OP_COL_DOT_AUX:
    case CODA_OP_COL_DOT_NORM: {
      // the warp's 32 rows of NE = 32 columns: per-column partial over this
      // 32-row block, finished over the row blocks by a second kernel
      if constexpr (NE == 32) {
        float x[NE];
        if constexpr (CODE == CODA_OP_COL_DOT_AUX || CODE == CODA_OP_COL_DOT_NORM) aux.load(op.aux, x);
        if constexpr (CODE == CODA_OP_COL_DOT_NORM) {
          // x_hat = r (aux - mu) with r = rowvec[0], mu = rowvec[1] (or 0)
          const float rr = c.row_ok ? __ldg(P.row_vec[0] + c.row) : 0.0f;
          const float mm = (c.row_ok && P.row_vec[1] != nullptr) ? __ldg(P.row_vec[1] + c.row) : 0.0f;
#pragma unroll
          for (int j = 0; j < NE; ++j) x[j] = rr * (x[j] - mm);
        }
        float a[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float t = (CODE == CODA_OP_COL_SUM) ? v[j] : (CODE == CODA_OP_COL_SUMSQ) ? v[j] * v[j] : v[j] * x[j];
          a[j] = c.row_ok ? t : 0.0f;
        }
        warp_column_sums(a);
        const int lane = threadIdx.x & 31;
        const int rb = c.row >> 5;
        if (rb < P.num_rb && lane < c.nvalid)
          P.ws_col[(static_cast<size_t>(op.red) * P.num_rb + rb) * c.n_out + c.col + lane] = a[0];
      }
      break;
    }
    default:
      break;
  }
}

// Run the op list on v (and, before SWIGLU, on u): the interpreter, for any
// list the library has no fixed sequence for.
template <int NE, bool kGLU, class Aux>
__device__ __forceinline__ void run_ops(const EpiProgram& P, float (&v)[NE], float (&u)[NE], const RowCtx& c,
                                        const Aux& aux, float (&red)[CODA_MAX_REDUCTIONS], uint32_t& keep_cnt) {
  const int n_ops = P.n_ops;
  for (int o = 0; o < n_ops; ++o) {
    const DevOp op = P.ops[o];
    const bool pre = kGLU && (o < P.glu_pos);
    switch (op.code) {
      case CODA_OP_SCALE:
        op_apply<CODA_OP_SCALE, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_COL_SCALE:
        op_apply<CODA_OP_COL_SCALE, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_BIAS:
        op_apply<CODA_OP_BIAS, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_ROW_SCALE:
        op_apply<CODA_OP_ROW_SCALE, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_RMS_ROWSCALE:
        op_apply<CODA_OP_RMS_ROWSCALE, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_LN_ROWSCALE:
        op_apply<CODA_OP_LN_ROWSCALE, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_GELU_TANH:
        op_apply<CODA_OP_GELU_TANH, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_GELU_ERF:
        op_apply<CODA_OP_GELU_ERF, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_GELU_ERF_GRAD:
        op_apply<CODA_OP_GELU_ERF_GRAD, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_SILU:
        op_apply<CODA_OP_SILU, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_SWIGLU:
        op_apply<CODA_OP_SWIGLU, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_GELU_TANH_GRAD:
        op_apply<CODA_OP_GELU_TANH_GRAD, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_DROPOUT:
        op_apply<CODA_OP_DROPOUT, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_RESIDUAL:
        op_apply<CODA_OP_RESIDUAL, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_STORE_PREACT:
        op_apply<CODA_OP_STORE_PREACT, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_ROW_SUM:
        op_apply<CODA_OP_ROW_SUM, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_ROW_MEAN:
        op_apply<CODA_OP_ROW_MEAN, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_ROW_SUMSQ:
        op_apply<CODA_OP_ROW_SUMSQ, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_ROW_DOT_AUX:
        op_apply<CODA_OP_ROW_DOT_AUX, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_COL_SUM:
        op_apply<CODA_OP_COL_SUM, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_COL_SUMSQ:
        op_apply<CODA_OP_COL_SUMSQ, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_COL_DOT_AUX:
        op_apply<CODA_OP_COL_DOT_AUX, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_COL_DOT_NORM:
        op_apply<CODA_OP_COL_DOT_NORM, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      case CODA_OP_COL_SCALE_F32:
        op_apply<CODA_OP_COL_SCALE_F32, NE, kGLU>(P, op, pre, v, u, c, aux, red, keep_cnt);
        break;
      default:
        break;
    }
  }
}

// A fixed op sequence (the opcodes of a hot op list, known at compile time):
// straight-line code without the interpreter's per-op dispatch.  The op
// parameters (scalars, slots, aux indices) still come from the op list.
template <uint32_t... Codes>
struct OpSeq {
  static constexpr int size = sizeof...(Codes);
};

template <int NE, bool kGLU, class Aux, uint32_t... Codes>
__device__ __forceinline__ void run_seq(OpSeq<Codes...>, const EpiProgram& P, float (&v)[NE], float (&u)[NE],
                                        const RowCtx& c, const Aux& aux, float (&red)[CODA_MAX_REDUCTIONS],
                                        uint32_t& keep_cnt) {
  int o = 0;
  ((op_apply<Codes, NE, kGLU>(P, P.ops[o], kGLU && (o < P.glu_pos), v, u, c, aux, red, keep_cnt), ++o), ...);
}

// Epilogue policies for the fused kernel: the interpreter, or one fixed sequence.
struct EpiInterp {
  template <int NE, bool kGLU, class Aux>
  __device__ __forceinline__ static void run(const EpiProgram& P, float (&v)[NE], float (&u)[NE], const RowCtx& c,
                                             const Aux& aux, float (&red)[CODA_MAX_REDUCTIONS], uint32_t& keep_cnt) {
    run_ops<NE, kGLU>(P, v, u, c, aux, red, keep_cnt);
  }
};

template <uint32_t... Codes>
struct EpiFixed {
  template <int NE, bool kGLU, class Aux>
  __device__ __forceinline__ static void run(const EpiProgram& P, float (&v)[NE], float (&u)[NE], const RowCtx& c,
                                             const Aux& aux, float (&red)[CODA_MAX_REDUCTIONS], uint32_t& keep_cnt) {
    run_seq<NE, kGLU>(OpSeq<Codes...>{}, P, v, u, c, aux, red, keep_cnt);
  }
};

}  // namespace coda
