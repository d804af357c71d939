// Fused kernels for the GPT-2 / BERT-style op lists (fixed op sequences):
// bias, bias -> GELU (tanh or erf), bias -> residual, GELU alone.
#include "coda_gemm_kernel.cuh"
#include "coda_launch.h"
#include "coda_sequences.h"

namespace coda {

cudaError_t launch_gemm_gpt(int seq, bool a_mn_major, bool b_mn_major, bool row_stats, bool pair,
                            const CUtensorMap* maps, const GemmParams& p, int grid, size_t smem, cudaStream_t st) {
  switch (seq) {
    case SEQ_BIAS:
      return launch_variant<EpiFixed<CODA_OP_BIAS>, false, false>(a_mn_major, b_mn_major, row_stats, pair, maps, p,
                                                                  grid, smem, st);
    case SEQ_BIAS_GELU:
      return launch_variant<EpiFixed<CODA_OP_BIAS, CODA_OP_GELU_TANH>, false, false>(
          a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
    case SEQ_BIAS_GELU_ERF:
      return launch_variant<EpiFixed<CODA_OP_BIAS, CODA_OP_GELU_ERF>, false, false>(
          a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
    case SEQ_BIAS_RESIDUAL:
      return launch_variant<EpiFixed<CODA_OP_BIAS, CODA_OP_RESIDUAL>, false, false>(
          a_mn_major, b_mn_major, row_stats, pair, maps, p, grid, smem, st);
    case SEQ_GELU:
      return launch_variant<EpiFixed<CODA_OP_GELU_TANH>, false, false>(a_mn_major, b_mn_major, row_stats, pair,
                                                                       maps, p, grid, smem, st);
    default:
      return cudaErrorNotSupported;
  }
}

}  // namespace coda
