// Fused kernels for SwiGLU projections (fixed op sequences).
#include "coda_gemm_kernel.cuh"
#include "coda_launch.h"
#include "coda_sequences.h"

namespace coda {

cudaError_t launch_gemm_fwd_glu(int seq, bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                             const CUtensorMap* maps,
                                const GemmParams& p, int grid, size_t smem, cudaStream_t st) {
  switch (seq) {
    case SEQ_SWIGLU:
      return launch_variant<EpiFixed<CODA_OP_SWIGLU>, true, false>(a_mn_major, b_mn_major, row_stats, pair, maps, p,
                                                                   grid, smem, st);
    case SEQ_SWIGLU_DROPOUT:
      return launch_variant<EpiFixed<CODA_OP_SWIGLU, CODA_OP_DROPOUT>, true, false>(a_mn_major, b_mn_major, row_stats, pair,
                                                                                    maps, p, grid, smem, st);
    default:
      return cudaErrorNotSupported;
  }
}

}  // namespace coda
