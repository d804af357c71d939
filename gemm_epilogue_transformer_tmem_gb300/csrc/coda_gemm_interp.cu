// Instantiations of the fused kernel with the op-list interpreter (any op list)
// for plain (unpaired) outputs, and the CTA-pair occupancy queries; the
// SwiGLU-paired instantiations are compiled in coda_gemm_interp_glu.cu.
#include "coda_gemm_kernel.cuh"
#include "coda_launch.h"

namespace coda {

cudaError_t launch_gemm_interp(bool glu, bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                               const CUtensorMap* maps, const GemmParams& p, int grid, size_t smem, cudaStream_t st) {
  if (glu) return launch_gemm_interp_glu(a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
  return launch_variant<EpiInterp, false, true, true>(a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
}

cudaError_t max_pairs(bool glu, bool b_mn_major, size_t smem, int* pairs) {
  if (glu) return max_pairs_glu(b_mn_major, smem, pairs);
  return b_mn_major ? max_active_pairs_t<false, true, false>(smem, pairs)
                    : max_active_pairs_t<false, false, false>(smem, pairs);
}

}  // namespace coda
