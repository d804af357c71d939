// Instantiations of the fused kernel with the op-list interpreter for
// SwiGLU-paired outputs with A given as [K, M] (no row-statistics warps).
#include "coda_gemm_kernel.cuh"
#include "coda_launch.h"

namespace coda {

cudaError_t launch_gemm_interp_glu_amn(bool b_mn_major, bool row_stats, bool pair, const CUtensorMap* maps,
                                       const GemmParams& p, int grid, size_t smem, cudaStream_t st) {
  if (row_stats) return cudaErrorNotSupported;
  if (pair)
    return b_mn_major ? launch_gemm_t<true, true, false, true, EpiInterp, true>(maps, p, grid, smem, st)
                      : launch_gemm_t<true, false, false, true, EpiInterp, true>(maps, p, grid, smem, st);
  return b_mn_major ? launch_gemm_t<true, true, false, false, EpiInterp, true>(maps, p, grid, smem, st)
                    : launch_gemm_t<true, false, false, false, EpiInterp, true>(maps, p, grid, smem, st);
}

}  // namespace coda
