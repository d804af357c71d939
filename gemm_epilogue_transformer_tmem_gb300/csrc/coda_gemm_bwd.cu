// Fused kernels for the backward op lists (fixed op sequences): the data
// gradient through GELU, and the weight gradient accumulated in place.
#include "coda_gemm_kernel.cuh"
#include "coda_launch.h"
#include "coda_sequences.h"

namespace coda {

cudaError_t launch_gemm_bwd(int seq, bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                             const CUtensorMap* maps,
                            const GemmParams& p, int grid, size_t smem, cudaStream_t st) {
  switch (seq) {
    case SEQ_DGRAD:
      return launch_variant<EpiFixed<CODA_OP_GELU_TANH_GRAD, CODA_OP_ROW_DOT_AUX, CODA_OP_ROW_SUM>, false, false>(
          a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
    case SEQ_WGRAD:   // A as [K, M] (the stored activations) or [M, K]
      return launch_variant<EpiFixed<CODA_OP_SCALE, CODA_OP_RESIDUAL, CODA_OP_ROW_SUMSQ>, false, false, true>(
          a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
    default:
      return cudaErrorNotSupported;
  }
}

}  // namespace coda
