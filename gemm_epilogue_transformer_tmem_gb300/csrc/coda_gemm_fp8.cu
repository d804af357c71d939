// Fused kernels with FP8 E4M3 operands: the op-list interpreter and the
// dequantisation sequences (row scale x column scale, optionally into SwiGLU).
#include "coda_gemm_kernel.cuh"
#include "coda_launch.h"
#include "coda_sequences.h"

namespace coda {

cudaError_t launch_gemm_fp8(int seq, bool glu, bool pair, const CUtensorMap* maps, const GemmParams& p, int grid,
                            size_t smem, cudaStream_t st) {
  switch (seq) {
    case SEQ_INTERP:
      return glu ? launch_variant_fp8<EpiInterp, true>(pair, maps, p, grid, smem, st)
                 : launch_variant_fp8<EpiInterp, false>(pair, maps, p, grid, smem, st);
    case SEQ_DEQUANT:
      return launch_variant_fp8<EpiFixed<CODA_OP_ROW_SCALE, CODA_OP_COL_SCALE_F32>, false>(pair, maps, p, grid,
                                                                                          smem, st);
    case SEQ_DEQUANT_SWIGLU:
      return launch_variant_fp8<EpiFixed<CODA_OP_ROW_SCALE, CODA_OP_COL_SCALE_F32, CODA_OP_SWIGLU>, true>(
          pair, maps, p, grid, smem, st);
    default:
      return cudaErrorNotSupported;
  }
}

}  // namespace coda
