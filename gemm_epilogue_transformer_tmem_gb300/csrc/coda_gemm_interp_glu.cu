// Instantiations of the fused kernel with the op-list interpreter for
// SwiGLU-paired outputs (G and U halves) with A given as [M, K], and their
// CTA-pair occupancy query; A given as [K, M] is compiled in
// coda_gemm_interp_glu_amn.cu.
#include "coda_gemm_kernel.cuh"
#include "coda_launch.h"

namespace coda {

cudaError_t launch_gemm_interp_glu(bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                                   const CUtensorMap* maps, const GemmParams& p, int grid, size_t smem,
                                   cudaStream_t st) {
  if (a_mn_major) return launch_gemm_interp_glu_amn(b_mn_major, row_stats, pair, maps, p, grid, smem, st);
  return launch_variant<EpiInterp, true, true, false>(false, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
}

cudaError_t max_pairs_glu(bool b_mn_major, size_t smem, int* pairs) {
  return b_mn_major ? max_active_pairs_t<true, true, false>(smem, pairs)
                    : max_active_pairs_t<true, false, false>(smem, pairs);
}

}  // namespace coda
