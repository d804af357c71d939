// Host-side launchers of the library's kernels (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "coda_internal.h"

namespace coda {

// fused GEMM + epilogue; maps = {A, B, D, aux0, aux1, aux2}
// pair: cta_group::2 on clusters of two CTAs (grid counts CTAs and is even)
// the op-list interpreter (any op list); SwiGLU-paired outputs in their own unit
cudaError_t launch_gemm_interp(bool glu, bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                             const CUtensorMap* maps,
                               const GemmParams& p, int grid, size_t smem, cudaStream_t st);
cudaError_t launch_gemm_interp_glu(bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                                   const CUtensorMap* maps, const GemmParams& p, int grid, size_t smem,
                                   cudaStream_t st);
cudaError_t launch_gemm_interp_glu_amn(bool b_mn_major, bool row_stats, bool pair, const CUtensorMap* maps,
                                       const GemmParams& p, int grid, size_t smem, cudaStream_t st);
// fixed op sequences (coda_sequences.h); cudaErrorNotSupported for a sequence
// or variant a translation unit does not hold
cudaError_t launch_gemm_norm(int seq, bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                             const CUtensorMap* maps,
                             const GemmParams& p, int grid, size_t smem, cudaStream_t st);
cudaError_t launch_gemm_norm_glu(int seq, bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                             const CUtensorMap* maps,
                                 const GemmParams& p, int grid, size_t smem, cudaStream_t st);
cudaError_t launch_gemm_fwd(int seq, bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                             const CUtensorMap* maps,
                            const GemmParams& p, int grid, size_t smem, cudaStream_t st);
cudaError_t launch_gemm_fwd_glu(int seq, bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                             const CUtensorMap* maps,
                                const GemmParams& p, int grid, size_t smem, cudaStream_t st);
cudaError_t launch_gemm_bwd(int seq, bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                             const CUtensorMap* maps,
                            const GemmParams& p, int grid, size_t smem, cudaStream_t st);
cudaError_t launch_gemm_gpt(int seq, bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                            const CUtensorMap* maps, const GemmParams& p, int grid, size_t smem, cudaStream_t st);
// FP8 E4M3 operands: the interpreter and the FP8 fixed sequences
cudaError_t launch_gemm_fp8(int seq, bool glu, bool pair, const CUtensorMap* maps, const GemmParams& p, int grid,
                            size_t smem, cudaStream_t st);
// MX block-scaled E4M3 operands (maps[6], maps[7]: the scale tiles): the
// interpreter, the plain GEMM and SwiGLU
cudaError_t launch_gemm_mx(int seq, bool glu, bool pair, const CUtensorMap* maps, const GemmParams& p, int grid,
                           size_t smem, cudaStream_t st);
// how many CTA pairs of the pair kernel fit on the device at once
cudaError_t max_pairs(bool glu, bool b_mn_major, size_t smem, int* pairs);
cudaError_t max_pairs_glu(bool b_mn_major, size_t smem, int* pairs);

cudaError_t launch_finalize(const float* ws_red, const uint32_t* ws_keep, int M, int num_n_tiles, int n_red,
                            const RedInfo& info, float inv_width, float* row_stats, uint32_t* keep_count,
                            cudaStream_t st);
// col_stats[slot[r]][j] = sum over the 32-row blocks of the partials, in block order
cudaError_t launch_finalize_cols(const float* ws_col, int n_colred, int num_rb, int64_t n_out, const int32_t* slots,
                                 float* col_stats, cudaStream_t st);
cudaError_t launch_rms_rowscale(const void* A, int64_t M, int64_t K, float inv_K, float eps, bool layernorm, float* r,
                                float* r_copy, float* mu, float* mu_copy, cudaStream_t st);
cudaError_t launch_ln_colsum(const void* W_folded, const void* W, const void* beta, int64_t K, int64_t N, bool kn,
                             float* c, float* b, cudaStream_t st);
cudaError_t launch_norm_backward(const void* g, const void* X, const float* r, const float* mu, const float* sum_g,
                                 const float* sum_gx, int64_t M, int64_t K, void* dX, int num_sms, cudaStream_t st);
cudaError_t launch_quantize_e4m3_rows(const void* X, int64_t M, int64_t K, void* Q, float* scale, cudaStream_t st);
// MX E4M3: codes [R, K] and E8M0 scales in the tiled storage (s_bytes, padding set to 127 first)
cudaError_t launch_quantize_mx_e4m3(const void* X, int64_t R, int64_t K, void* Q, void* S, size_t s_bytes, int num_sms,
                                    cudaStream_t st);
cudaError_t launch_layernorm(const void* X, const void* gamma, const void* beta, int64_t M, int64_t K, float eps,
                             void* Xn, cudaStream_t st);
cudaError_t launch_fold_gamma(const void* W, const void* gamma, void* W_out, int64_t K, int64_t N, bool kn,
                              int num_sms, cudaStream_t st);
cudaError_t launch_rmsnorm(const void* X, const void* gamma, int64_t M, int64_t K, float eps, void* Xn,
                           float* rstd, cudaStream_t st);
cudaError_t launch_epilogue_apply(const void* C, void* D, int64_t M, int N, int N_out, int half,
                                  const void* const* aux, float* row_stats, uint32_t* keep_count,
                                  const EpiProgram& prog, cudaStream_t st);

// Workspace bytes for coda_gemm_epilogue: with_split = the size that allows the
// split over K (what coda_workspace_size reports), else the minimum.
coda_status workspace_need(int64_t M, int64_t N, int64_t K, const coda_epilogue* epi, bool with_split,
                           size_t* bytes);

}  // namespace coda
