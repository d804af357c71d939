// Instantiations of the fused kernel with the SwiGLU pairing (B tile = G half | U half).
#include "coda_gemm_kernel.cuh"
#include "coda_launch.h"

namespace coda {

cudaError_t launch_gemm_glu(bool b_mn_major, bool row_stats, const CUtensorMap* maps, const GemmParams& p,
                            int grid, size_t smem, cudaStream_t st) {
  if (b_mn_major)
    return row_stats ? launch_gemm_t<true, true, true>(maps, p, grid, smem, st)
                     : launch_gemm_t<true, true, false>(maps, p, grid, smem, st);
  return row_stats ? launch_gemm_t<true, false, true>(maps, p, grid, smem, st)
                   : launch_gemm_t<true, false, false>(maps, p, grid, smem, st);
}

}  // namespace coda
