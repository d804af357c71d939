// Instantiations of the fused kernel without SwiGLU pairing (256 output columns per tile).
#include "coda_gemm_kernel.cuh"
#include "coda_launch.h"

namespace coda {

cudaError_t launch_gemm_plain(bool b_mn_major, bool row_stats, bool pair, const CUtensorMap* maps, const GemmParams& p,
                        int grid, size_t smem, cudaStream_t st) {
  if (pair) {
    if (b_mn_major)
      return row_stats ? launch_gemm_t<false, true, true, true>(maps, p, grid, smem, st)
                       : launch_gemm_t<false, true, false, true>(maps, p, grid, smem, st);
    return row_stats ? launch_gemm_t<false, false, true, true>(maps, p, grid, smem, st)
                     : launch_gemm_t<false, false, false, true>(maps, p, grid, smem, st);
  }
  if (b_mn_major)
    return row_stats ? launch_gemm_t<false, true, true, false>(maps, p, grid, smem, st)
                     : launch_gemm_t<false, true, false, false>(maps, p, grid, smem, st);
  return row_stats ? launch_gemm_t<false, false, true, false>(maps, p, grid, smem, st)
                   : launch_gemm_t<false, false, false, false>(maps, p, grid, smem, st);
}

cudaError_t max_pairs_plain(bool b_mn_major, bool row_stats, size_t smem, int* pairs) {
  if (b_mn_major)
    return row_stats ? max_active_pairs_t<false, true, true>(smem, pairs)
                     : max_active_pairs_t<false, true, false>(smem, pairs);
  return row_stats ? max_active_pairs_t<false, false, true>(smem, pairs)
                   : max_active_pairs_t<false, false, false>(smem, pairs);
}

}  // namespace coda
