// Instantiations of the fused kernel without SwiGLU pairing (256 output columns per tile).
#include "coda_gemm_kernel.cuh"
#include "coda_launch.h"

namespace coda {

cudaError_t launch_gemm_plain(bool b_mn_major, bool row_stats, const CUtensorMap* maps, const GemmParams& p,
                              int grid, size_t smem, cudaStream_t st) {
  if (b_mn_major)
    return row_stats ? launch_gemm_t<false, true, true>(maps, p, grid, smem, st)
                     : launch_gemm_t<false, true, false>(maps, p, grid, smem, st);
  return row_stats ? launch_gemm_t<false, false, true>(maps, p, grid, smem, st)
                   : launch_gemm_t<false, false, false>(maps, p, grid, smem, st);
}

}  // namespace coda
