// Fused kernel for the commuted RMSNorm into a SwiGLU projection (fixed op sequence).
#include "coda_gemm_kernel.cuh"
#include "coda_launch.h"
#include "coda_sequences.h"

namespace coda {

cudaError_t launch_gemm_norm_glu(int seq, bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                             const CUtensorMap* maps,
                                 const GemmParams& p, int grid, size_t smem, cudaStream_t st) {
  if (seq != SEQ_RMS_SWIGLU) return cudaErrorNotSupported;
  return launch_variant<EpiFixed<CODA_OP_RMS_ROWSCALE, CODA_OP_SWIGLU>, true, true>(a_mn_major, b_mn_major, row_stats, pair,
                                                                                    maps, p, grid, smem, st);
}

}  // namespace coda
