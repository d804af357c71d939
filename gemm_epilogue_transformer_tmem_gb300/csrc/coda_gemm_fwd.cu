// Fused kernels for forward op lists without a norm or SwiGLU (fixed op sequences).
#include "coda_gemm_kernel.cuh"
#include "coda_launch.h"
#include "coda_sequences.h"

namespace coda {

cudaError_t launch_gemm_fwd(int seq, bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                             const CUtensorMap* maps,
                            const GemmParams& p, int grid, size_t smem, cudaStream_t st) {
  switch (seq) {
    case SEQ_NONE:
      return launch_variant<EpiFixed<>, false, false, true>(a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
    case SEQ_RESIDUAL:
      return launch_variant<EpiFixed<CODA_OP_RESIDUAL>, false, false, true>(a_mn_major, b_mn_major, row_stats, pair, maps, p,
                                                                      grid, smem, st);
    case SEQ_BIAS_GELU_RESIDUAL:
      return launch_variant<EpiFixed<CODA_OP_BIAS, CODA_OP_GELU_TANH, CODA_OP_RESIDUAL>, false, false>(
          a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
    case SEQ_RESIDUAL_SUMSQ:
      return launch_variant<EpiFixed<CODA_OP_RESIDUAL, CODA_OP_ROW_SUMSQ>, false, false>(
          a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
    default:
      return cudaErrorNotSupported;
  }
}

}  // namespace coda
