// Fixed op sequences of the fused kernel (internal).
//
// The CODA article (d9bl.com, §3.3) compiles each epilogue program into its own
// specialised kernel.  Here the op list is interpreted at run time, except for
// the op lists below: for these the kernel is instantiated with the opcodes
// fixed at compile time (straight-line epilogue code, no per-op dispatch; the
// op parameters still come from the op list).  A list that matches none of
// them, or a kernel variant a sequence is not built for, runs the interpreter.
#pragma once

#include <cstdint>

#include "../../include/coda.h"

namespace coda {

enum SeqId : int {
  SEQ_INTERP = 0,         // interpreter
  SEQ_NONE,               // plain GEMM
  SEQ_RMS,                // commuted RMSNorm projection
  SEQ_LN,                 // commuted LayerNorm projection
  SEQ_RESIDUAL,           // projection + residual
  SEQ_BIAS_GELU_RESIDUAL, // bias -> GELU(tanh) -> + residual
  SEQ_DGRAD,              // dX = dY W^T * GELU'(Z), row sums of dX*Xhat and dX
  SEQ_SWIGLU,             // SwiGLU up-projection
  SEQ_RMS_SWIGLU,         // commuted RMSNorm -> SwiGLU
  SEQ_SWIGLU_DROPOUT,     // SwiGLU -> dropout
  SEQ_DEQUANT,            // FP8 dequantisation: row scale x column scale
  SEQ_DEQUANT_SWIGLU,     // FP8 dequantisation -> SwiGLU
  SEQ_BIAS,               // projection + bias
  SEQ_BIAS_GELU,          // bias -> GELU(tanh): GPT-2 MLP up-projection
  SEQ_BIAS_GELU_ERF,      // bias -> GELU(erf): BERT MLP up-projection
  SEQ_BIAS_RESIDUAL,      // bias -> + residual: attention out / MLP down-projection
  SEQ_GELU,               // GELU(tanh) without bias
  SEQ_RESIDUAL_SUMSQ,     // + residual, row sums of squares (the next norm's statistics)
  SEQ_WGRAD,              // s * X^T dY + dW (in place), row sums of squares of the new dW
  SEQ_COUNT_
};

struct SeqDef {
  int id;
  bool glu;
  int n;
  uint32_t codes[4];
};

constexpr SeqDef kSeqDefs[] = {
    {SEQ_NONE, false, 0, {0, 0, 0, 0}},
    {SEQ_RMS, false, 1, {CODA_OP_RMS_ROWSCALE, 0, 0, 0}},
    {SEQ_LN, false, 1, {CODA_OP_LN_ROWSCALE, 0, 0, 0}},
    {SEQ_RESIDUAL, false, 1, {CODA_OP_RESIDUAL, 0, 0, 0}},
    {SEQ_BIAS_GELU_RESIDUAL, false, 3, {CODA_OP_BIAS, CODA_OP_GELU_TANH, CODA_OP_RESIDUAL, 0}},
    {SEQ_DGRAD, false, 3, {CODA_OP_GELU_TANH_GRAD, CODA_OP_ROW_DOT_AUX, CODA_OP_ROW_SUM, 0}},
    {SEQ_SWIGLU, true, 1, {CODA_OP_SWIGLU, 0, 0, 0}},
    {SEQ_RMS_SWIGLU, true, 2, {CODA_OP_RMS_ROWSCALE, CODA_OP_SWIGLU, 0, 0}},
    {SEQ_SWIGLU_DROPOUT, true, 2, {CODA_OP_SWIGLU, CODA_OP_DROPOUT, 0, 0}},
    {SEQ_DEQUANT, false, 2, {CODA_OP_ROW_SCALE, CODA_OP_COL_SCALE_F32, 0, 0}},
    {SEQ_DEQUANT_SWIGLU, true, 3, {CODA_OP_ROW_SCALE, CODA_OP_COL_SCALE_F32, CODA_OP_SWIGLU, 0}},
    {SEQ_BIAS, false, 1, {CODA_OP_BIAS, 0, 0, 0}},
    {SEQ_BIAS_GELU, false, 2, {CODA_OP_BIAS, CODA_OP_GELU_TANH, 0, 0}},
    {SEQ_BIAS_GELU_ERF, false, 2, {CODA_OP_BIAS, CODA_OP_GELU_ERF, 0, 0}},
    {SEQ_BIAS_RESIDUAL, false, 2, {CODA_OP_BIAS, CODA_OP_RESIDUAL, 0, 0}},
    {SEQ_GELU, false, 1, {CODA_OP_GELU_TANH, 0, 0, 0}},
    {SEQ_RESIDUAL_SUMSQ, false, 2, {CODA_OP_RESIDUAL, CODA_OP_ROW_SUMSQ, 0, 0}},
    {SEQ_WGRAD, false, 3, {CODA_OP_SCALE, CODA_OP_RESIDUAL, CODA_OP_ROW_SUMSQ, 0}},
};

}  // namespace coda
