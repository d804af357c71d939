// Instantiations of the fused kernel with the op-list interpreter (any op list),
// plain and SwiGLU-paired, and the CTA-pair occupancy queries.
#include "coda_gemm_kernel.cuh"
#include "coda_launch.h"

namespace coda {

cudaError_t launch_gemm_interp(bool glu, bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                             const CUtensorMap* maps,
                               const GemmParams& p, int grid, size_t smem, cudaStream_t st) {
  return glu ? launch_variant<EpiInterp, true, true, true>(a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st)
             : launch_variant<EpiInterp, false, true, true>(a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
}

cudaError_t max_pairs(bool glu, bool b_mn_major, size_t smem, int* pairs) {
  if (glu)
    return b_mn_major ? max_active_pairs_t<true, true, false>(smem, pairs)
                      : max_active_pairs_t<true, false, false>(smem, pairs);
  return b_mn_major ? max_active_pairs_t<false, true, false>(smem, pairs)
                    : max_active_pairs_t<false, false, false>(smem, pairs);
}

}  // namespace coda
