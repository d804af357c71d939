// Instantiations of the fused kernel with the SwiGLU pairing (B tile = G half | U half).
#include "coda_gemm_kernel.cuh"
#include "coda_launch.h"

namespace coda {

cudaError_t launch_gemm_glu(bool b_mn_major, bool row_stats, bool pair, const CUtensorMap* maps, const GemmParams& p,
                        int grid, size_t smem, cudaStream_t st) {
  if (pair) {
    if (b_mn_major)
      return row_stats ? launch_gemm_t<true, true, true, true>(maps, p, grid, smem, st)
                       : launch_gemm_t<true, true, false, true>(maps, p, grid, smem, st);
    return row_stats ? launch_gemm_t<true, false, true, true>(maps, p, grid, smem, st)
                     : launch_gemm_t<true, false, false, true>(maps, p, grid, smem, st);
  }
  if (b_mn_major)
    return row_stats ? launch_gemm_t<true, true, true, false>(maps, p, grid, smem, st)
                     : launch_gemm_t<true, true, false, false>(maps, p, grid, smem, st);
  return row_stats ? launch_gemm_t<true, false, true, false>(maps, p, grid, smem, st)
                   : launch_gemm_t<true, false, false, false>(maps, p, grid, smem, st);
}

cudaError_t max_pairs_glu(bool b_mn_major, bool row_stats, size_t smem, int* pairs) {
  if (b_mn_major)
    return row_stats ? max_active_pairs_t<true, true, true>(smem, pairs)
                     : max_active_pairs_t<true, true, false>(smem, pairs);
  return row_stats ? max_active_pairs_t<true, false, true>(smem, pairs)
                   : max_active_pairs_t<true, false, false>(smem, pairs);
}

}  // namespace coda
