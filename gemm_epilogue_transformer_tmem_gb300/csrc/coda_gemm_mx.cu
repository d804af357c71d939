// Fused kernels with MX block-scaled E4M3 operands (tcgen05 kind::mxf8f6f4):
// the op-list interpreter, the plain GEMM and SwiGLU.
#include "coda_gemm_kernel.cuh"
#include "coda_launch.h"
#include "coda_sequences.h"

namespace coda {

cudaError_t launch_gemm_mx(int seq, bool glu, bool pair, const CUtensorMap* maps, const GemmParams& p, int grid,
                           size_t smem, cudaStream_t st) {
  switch (seq) {
    case SEQ_INTERP:
      return glu ? launch_variant_mx<EpiInterp, true>(pair, maps, p, grid, smem, st)
                 : launch_variant_mx<EpiInterp, false>(pair, maps, p, grid, smem, st);
    case SEQ_NONE:
      return launch_variant_mx<EpiFixed<>, false>(pair, maps, p, grid, smem, st);
    case SEQ_SWIGLU:
      return launch_variant_mx<EpiFixed<CODA_OP_SWIGLU>, true>(pair, maps, p, grid, smem, st);
    default:
      return cudaErrorNotSupported;
  }
}

}  // namespace coda
