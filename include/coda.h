/*
 * coda.h -- C ABI of the GB300 (sm_103a) GEMM + on-chip epilogue library.
 *
 * The operation.  The CODA article (d9bl.com, "CODA：将 Transformer 模块重新
 * 表达为 GEMM+Epilogue 程序", §3.1 "GEMM+Epilogue 分解", Fig. 1 and Fig. 4)
 * writes the fused kernel as a GEMM  C = alpha*A*B + beta*C_prev  followed by an
 * epilogue  D = f(C)  that is applied elementwise or row by row while the output
 * tile is still on chip, before the single global write of D.  The
 * agentlenshq.com summary ("CODA: GEMM-Epilogue FusionによるTransformer
 * トレーニングの最適化", section "仕組み") keeps the GEMM mainloop fixed and
 * builds f from a small set of composable primitives: scaling (by a constant or
 * a vector), reductions (sum or mean along a dimension), pairwise/elementwise
 * transforms (activations) and accumulation (residual).  The zeli.app page
 * ("CODA: Wie Transformer-Blöcke als GEMM-Epilogue-Programme neu geschrieben
 * werden", augment_me's comment) adds the commuted RMSNorm: the norm's row
 * scale r_i is pulled past the projection,
 *     rmsnorm(X) @ W  ==  r (.)_row ( X @ (gamma (.)_row W) ),
 * with r_i = 1/sqrt(mean_k x_ik^2 + eps) gathered over the K tiles of X.
 *
 * Here f is an op list (coda_epilogue) interpreted on the fp32 accumulator tile
 * after it is drained from tensor memory; the pages' DSL and compiler are not
 * reproduced.  alpha is the SCALE op; beta*C_prev is the RESIDUAL op.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     keeps no reference after the call returns and allocates no device memory.
 *   - Matrices are dense row-major with the row stride equal to the row width.
 *   - A, B, D, residual, Z, Xhat, column vectors, gamma and the pre-activation
 *     output are bf16 (stored as 16-bit words); row vectors, row statistics and
 *     the accumulator are fp32; keep counts are uint32.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous: they validate, enqueue and return.  A returned CODA_OK means
 *     the work was enqueued, not that it finished.
 *   - Argument, alignment and op-list checks happen on the host before anything
 *     is enqueued; on failure nothing is enqueued and no output is touched.
 *   - Device-side failures (a pipeline wait that exceeded its time limit) are
 *     recorded in a per-device error word and reported by
 *     coda_check_device_error().  Kernels never trap.
 *   - No function prints, throws or aborts.  Functions are thread-safe except
 *     that concurrent launches on one device share the device error word.
 */
#ifndef CODA_H
#define CODA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CODA_API __attribute__((visibility("default")))
#else
#define CODA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CODA_OK = 0,
  CODA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad op list         */
  CODA_ERR_UNSUPPORTED = 2,   /* valid request the library does not support  */
  CODA_ERR_ALIGNMENT = 3,     /* pointer or row stride not 16-byte aligned   */
  CODA_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed           */
  CODA_ERR_TIMEOUT = 5,       /* a device-side wait exceeded its time limit  */
  CODA_ERR_WORKSPACE = 6      /* workspace missing or too small              */
} coda_status;

/* Storage of the B operand. */
typedef enum {
  CODA_B_KN = 0,   /* B is [K, N] row-major: C = A @ B   (weights as x @ W)    */
  CODA_B_NK = 1,   /* B is [N, K] row-major: C = A @ B^T (dgrad dY @ W^T, or an
                      nn.Linear weight stored [out, in])                        */
  CODA_A_KM = 2,   /* flag, OR-ed with either of the above: A is given as [K, M]
                      row-major, C = A^T @ B (the weight gradient X^T @ dY from
                      the stored activations X [tokens, features]); M must be a
                      multiple of 8; not with RMS_ROWSCALE / LN_ROWSCALE        */
  CODA_AB_E4M3 = 4 /* flag: A [M, K] and B [N, K] (CODA_B_NK) are FP8 E4M3 bytes
                      (tcgen05 kind::f8f6f4, fp32 accumulation); K must be a
                      multiple of 16; the dequantisation scales are epilogue ops
                      (ROW_SCALE for A's rows, COL_SCALE_F32 for B's); not with
                      CODA_A_KM, RMS_ROWSCALE or LN_ROWSCALE                    */
} coda_b_layout;

/*
 * Epilogue opcodes.  Ops run in list order on the fp32 value x of each output
 * element (row i, column j).  "width" is the current row width: N before a
 * SWIGLU op, N/2 after it (N_out = N/2 when the list has SWIGLU, else N).
 *
 * Scaling (agentlenshq.com "Scaling"; alpha of CODA §3.1):
 *   SCALE          x *= f0
 *   COL_SCALE      x *= colvec[slot][j]         (bf16 vector of `width` entries)
 *   BIAS           x += colvec[slot][j]         (bf16 vector of `width` entries)
 *   ROW_SCALE      x *= rowvec[slot][i]         (fp32 vector of M entries)
 *   COL_SCALE_F32  x *= aux.col_scale_f32[j]    (fp32 vector of `width` entries: e.g.
 *                  the per-channel dequantisation scale of an FP8 weight)
 *   RMS_ROWSCALE   x *= r_i, r_i = 1/sqrt(sum_k A[i,k]^2 / K + f0) gathered from
 *                  the A tiles the mainloop streams (commuted RMSNorm, zeli.app);
 *                  f0 = eps.  If slot != CODA_NO_SLOT, r_i is also written to
 *                  row_stats[slot*M + i].  With B = bf16(gamma (.)_row W) (see
 *                  coda_fold_gamma) the result is rmsnorm(A; gamma) @ W.
 *   LN_ROWSCALE    commuted LayerNorm: x = r_i * (x - mu_i * c_j) + b_j, with
 *                  mu_i = mean_k A[i,k], r_i = 1/sqrt(mean_k (A[i,k]-mu_i)^2 + f0)
 *                  gathered from A like RMS_ROWSCALE (f0 = eps), c = aux.ln_colsum
 *                  and b = aux.ln_bias (fp32 vectors of `width` entries, b may be
 *                  NULL).  With B, c and b from coda_fold_layernorm the result is
 *                  layernorm(A; gamma, beta) @ W.  At most one RMS_ROWSCALE,
 *                  RMS_SUMSQ_ROWSCALE or LN_ROWSCALE per list.
 *   RMS_SUMSQ_ROWSCALE  x *= r_i, r_i = 1/sqrt(rowvec[slot][i] / K + f0): the
 *                  commuted RMSNorm with the row sums of squares of A supplied
 *                  (fp32 [M], sum_k A[i,k]^2), f0 = eps.  When A is the output
 *                  of an earlier call whose epilogue ended in RESIDUAL (a
 *                  Transformer block's hidden state), that call's ROW_SUMSQ gives
 *                  these sums while the tile is on chip, so the norm costs no
 *                  pass over A at all: the row statistics of the zeli.app
 *                  comment's commuted norm, gathered one call earlier.  With
 *                  B = bf16(gamma (.)_row W) the result is rmsnorm(A; gamma) @ W.
 * Elementwise transforms (agentlenshq.com "Pairwise Transformations"):
 *   GELU_TANH      x = 0.5 x (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3)))
 *   SILU           x = x / (1 + exp(-x))
 *   SWIGLU         pairs output column j < N/2 (G) with column j + N/2 (U):
 *                  x_j = silu(G_j) * U_j; width becomes N/2.  At most once.
 *   GELU_TANH_GRAD x *= GELU_TANH'(z[i,j])      (z: bf16 [M, N_out], aux.z)
 *   GELU_ERF       x = x * Phi(x) = 0.5 x (1 + erf(x / sqrt(2)))   (exact GELU)
 *   GELU_ERF_GRAD  x *= Phi(z) + z phi(z), phi the standard normal density
 *                  (z: bf16 [M, N_out], aux.z)
 *   DROPOUT        f0 = p in [0,1).  keep iff splitmix64(seed, i*N_out + j) < T,
 *                  T = floor(ldexp(1-p, 64)) in fp64; kept x *= 1/(1-p), dropped
 *                  x = 0.  splitmix64(seed, n) is output n (0-based) of the
 *                  splitmix64 generator seeded with `seed` (Steele, Lea & Flood,
 *                  OOPSLA 2014).  At most once.  Per-row keep counts go to
 *                  row_keep_count when it is non-NULL.
 * Accumulation (agentlenshq.com "Accumulation"; beta*C_prev of CODA §3.1):
 *   RESIDUAL       x += f0 * residual[i,j]      (bf16 [M, N_out], aux.residual; it may
 *                  be D itself, for accumulation in place)
 *   STORE_PREACT   writes bf16(x) to aux.preact_out[i, j] ([M, width]); at most once
 * Reductions over the row's `width` columns (agentlenshq.com "Reductions"):
 *   ROW_SUM        row_stats[slot*M + i] = sum_j x
 *   ROW_MEAN       row_stats[slot*M + i] = sum_j x / width
 *   ROW_SUMSQ      row_stats[slot*M + i] = sum_j x^2
 *   ROW_DOT_AUX    row_stats[slot*M + i] = sum_j x * xhat[i,j]  (aux.xhat [M,N_out])
 * Reductions over the M rows of each output column (agentlenshq.com
 * "Reductions", along the other dimension; the bias and norm-parameter
 * gradients of a backward pass), fused kernel only:
 *   COL_SUM        col_stats[slot*N_out + j] = sum_i x
 *   COL_SUMSQ      col_stats[slot*N_out + j] = sum_i x^2
 *   COL_DOT_AUX    col_stats[slot*N_out + j] = sum_i x * xhat[i,j]
 *   COL_DOT_NORM   col_stats[slot*N_out + j] = sum_i x * r_i (xhat[i,j] - mu_i), with
 *                  r = rowvec[0] and mu = rowvec[1] (NULL: 0): with xhat = the norm's
 *                  input X and x = dL/d(norm output), this is dL/dgamma
 *                  (col_stats = aux.col_stats, fp32; at most CODA_MAX_COL_REDUCTIONS)
 *
 * Ops that read an [M, N_out] aux tensor, reductions and DROPOUT must come
 * after SWIGLU when the list has one.  At most CODA_MAX_REDUCTIONS reductions.
 */
typedef enum {
  CODA_OP_SCALE = 0,
  CODA_OP_COL_SCALE = 1,
  CODA_OP_BIAS = 2,
  CODA_OP_ROW_SCALE = 3,
  CODA_OP_RMS_ROWSCALE = 4,
  CODA_OP_GELU_TANH = 5,
  CODA_OP_SILU = 6,
  CODA_OP_SWIGLU = 7,
  CODA_OP_GELU_TANH_GRAD = 8,
  CODA_OP_DROPOUT = 9,
  CODA_OP_RESIDUAL = 10,
  CODA_OP_STORE_PREACT = 11,
  CODA_OP_ROW_SUM = 12,
  CODA_OP_ROW_MEAN = 13,
  CODA_OP_ROW_SUMSQ = 14,
  CODA_OP_ROW_DOT_AUX = 15,
  CODA_OP_GELU_ERF = 16,
  CODA_OP_GELU_ERF_GRAD = 17,
  CODA_OP_LN_ROWSCALE = 18,
  CODA_OP_COL_SUM = 19,
  CODA_OP_COL_SUMSQ = 20,
  CODA_OP_COL_DOT_AUX = 21,
  CODA_OP_COL_DOT_NORM = 22,
  CODA_OP_COL_SCALE_F32 = 23,
  CODA_OP_RMS_SUMSQ_ROWSCALE = 24,
  CODA_OP_COUNT_ = 25
} coda_opcode;

#define CODA_MAX_OPS 16
#define CODA_MAX_COL_VECS 4
#define CODA_MAX_ROW_VECS 2
#define CODA_MAX_STAT_SLOTS 8
#define CODA_MAX_REDUCTIONS 4
#define CODA_MAX_COL_REDUCTIONS 2
#define CODA_NO_SLOT 0xFFFFFFFFu

typedef struct {
  uint32_t opcode;   /* coda_opcode                                   */
  uint32_t slot;     /* vector slot or row-stat slot, per opcode      */
  float f0;          /* scalar parameter, per opcode                  */
  float f1;          /* reserved, must be 0                           */
} coda_op;

typedef struct {
  uint32_t n_ops;                 /* 0 .. CODA_MAX_OPS; 0 = plain GEMM      */
  uint32_t reserved;              /* must be 0                              */
  uint64_t seed;                  /* dropout seed                           */
  coda_op ops[CODA_MAX_OPS];
} coda_epilogue;

typedef struct {
  const void* col_vec[CODA_MAX_COL_VECS];  /* bf16 [width at the op]        */
  const float* row_vec[CODA_MAX_ROW_VECS]; /* fp32 [M]                      */
  const void* residual;                    /* bf16 [M, N_out]               */
  const void* z;                           /* bf16 [M, N_out]               */
  const void* xhat;                        /* bf16 [M, N_out]               */
  void* preact_out;                        /* bf16 [M, width at the op]     */
  const float* ln_colsum;                  /* fp32 [width], LN_ROWSCALE     */
  const float* ln_bias;                    /* fp32 [width], LN_ROWSCALE     */
  float* col_stats;                        /* fp32 [slots][N_out], COL_* ops (output) */
  const float* col_scale_f32;              /* fp32 [width], COL_SCALE_F32   */
} coda_aux;

/*
 * coda_gemm_epilogue -- D = f(A @ B) in one persistent kernel on the calling
 * stream: TMA-staged bf16 operands, tcgen05 MMA into fp32 tensor memory, the
 * op list applied to the drained tile, bf16 (round-to-nearest-even) TMA store.
 * Row reductions and keep counts are finished by a second small kernel.
 *
 *   A        bf16 [M, K], or [K, M] with the CODA_A_KM flag in b_layout
 *   B        bf16 [K, N] (CODA_B_KN) or [N, K] (CODA_B_NK)
 *   M, N, K  M >= 0, N >= 0, K >= 0, each < 2^31.  N and K must be multiples of
 *            8 (16-byte rows); with SWIGLU, N must be a multiple of 16.  M == 0
 *            or N == 0 enqueues nothing.  K == 0 means C = 0.
 *   epi      op list (may be NULL: plain GEMM)
 *   aux      aux tensors the op list names (may be NULL if it names none)
 *   D        bf16 [M, N_out] output
 *   row_stats fp32 [CODA_MAX_STAT_SLOTS or fewer][M], slot-major; required if
 *            the list has a reduction or an RMS_ROWSCALE with a slot
 *   row_keep_count uint32 [M] or NULL
 *   workspace / workspace_bytes: device scratch of at least
 *            coda_workspace_size() bytes (may be NULL when that size is 0);
 *            the call overwrites it; it must not be shared by calls that can
 *            run at the same time.
 * All pointers must be 16-byte aligned.  Returns CODA_OK once enqueued.
 */
CODA_API coda_status coda_gemm_epilogue(const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                               int32_t b_layout, const coda_epilogue* epi, const coda_aux* aux,
                               void* D, float* row_stats, uint32_t* row_keep_count,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * coda_gemm_epilogue_noalloc -- coda_gemm_epilogue without a caller-supplied
 * workspace.  The paper has no counterpart: this entry point exists for callers
 * that cannot allocate device memory when they call the library, such as a
 * serving loop that fixes its memory footprint at start-up (cudaMalloc can
 * synchronise the device and has no latency bound) or a runtime whose device
 * memory belongs entirely to another allocator.
 *
 * The row-reduction and keep-count partials go to one scratch buffer of
 * CODA_NOALLOC_SCRATCH_BYTES that the library holds on every GPU it is loaded
 * on, for the life of the process.  Arguments, results and errors are those of
 * coda_gemm_epilogue, plus CODA_ERR_WORKSPACE when the problem needs more
 * scratch than the buffer holds (coda_workspace_size tells how much it needs,
 * less its split-K part: the split over K runs only when its partials fit as
 * well; problems without reductions, keep counts or a commuted norm need none).  It calls no
 * allocating routine.  The first call on a device looks up the buffer's device
 * address (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture.  All calls share the buffer: calls whose
 * kernels can run at the same time on one device (different streams or host
 * threads) race on it.
 */
#define CODA_NOALLOC_SCRATCH_BYTES (8u << 20)
CODA_API coda_status coda_gemm_epilogue_noalloc(const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                                                int32_t b_layout, const coda_epilogue* epi, const coda_aux* aux,
                                                void* D, float* row_stats, uint32_t* row_keep_count,
                                                void* stream);

/* Scratch bytes coda_gemm_epilogue wants for these sizes and this op list:
 * row-reduction and keep-count partials (one per 128/256-column tile), the
 * commuted-norm row statistics, and the split-K partial accumulators (3 x 128
 * KB per slot) and arrival counters (4 bytes per slot): one slot per tile for a
 * problem of at most 76 tiles of 128 rows with K >= 1024, which leaves most SMs
 * idle; 160 slots (one per CTA of the grid) for a problem of at least 128
 * tiles, whose last, partly filled wave may be split.  A workspace that holds
 * everything but the split-K part is accepted and runs without the split.
 * The answer depends on coda_set_cta_pair / coda_set_split_k, not on the device. */
CODA_API coda_status coda_workspace_size(int64_t M, int64_t N, int64_t K, const coda_epilogue* epi,
                                size_t* bytes);

/*
 * coda_fold_gamma -- W_out = bf16(gamma[k] * W[k, n]) for the commuted RMSNorm
 * (zeli.app, augment_me: gamma is folded into the projection weight so that only
 * the row scale r_i remains for the epilogue).  W and W_out have the layout
 * `b_layout` ([K,N] or [N,K]); gamma is bf16 [K].  W_out may equal W.
 */
CODA_API coda_status coda_fold_gamma(const void* W, const void* gamma, void* W_out, int64_t K, int64_t N,
                            int32_t b_layout, void* stream);

/*
 * coda_fold_layernorm -- weights for the commuted LayerNorm (LN_ROWSCALE): the
 * zeli.app comment (augment_me) names LayerNorm beside RMSNorm as a norm whose
 * row-wise factors commute past the projection:
 *     layernorm(X) @ W = r (.)_row ( X @ W' - mu (x) c ) + b,
 *     W' = gamma (.)_row W,  c_j = sum_k W'[k,j],  b_j = sum_k beta_k W[k,j].
 * Writes W_out = bf16(gamma[k] * W[k,n]) (layout `b_layout`), colsum_out =
 * column sums of the bf16 W_out in fp32 (so the identity holds exactly for the
 * folded weight) and bias_out = beta^T W in fp32 (NULL beta: zeros).  gamma and
 * beta are bf16 [K]; colsum_out and bias_out are fp32 [N].  W_out must not
 * alias W.
 */
CODA_API coda_status coda_fold_layernorm(const void* W, const void* gamma, const void* beta, void* W_out,
                                         float* colsum_out, float* bias_out, int64_t K, int64_t N,
                                         int32_t b_layout, void* stream);

/*
 * coda_rmsnorm -- the unfused normalisation pass: Xn[i,k] = bf16(r_i x_ik gamma_k),
 * r_i = 1/sqrt(mean_k x_ik^2 + eps); rstd_out (fp32 [M]) may be NULL.  This is the
 * separate memory-bound kernel that the commuted form removes; it exists so the
 * unfused chain can be run and measured with the library's own kernels.
 */
CODA_API coda_status coda_rmsnorm(const void* X, const void* gamma, int64_t M, int64_t K, float eps,
                         void* Xn_out, float* rstd_out, void* stream);

/*
 * coda_layernorm -- the unfused LayerNorm pass: Xn[i,k] = bf16(gamma_k (x_ik - mu_i)
 * r_i + beta_k), mu_i = mean_k x_ik, r_i = 1/sqrt(mean_k (x_ik - mu_i)^2 + eps);
 * beta may be NULL.  The memory-bound kernel the commuted form removes.
 */
CODA_API coda_status coda_layernorm(const void* X, const void* gamma, const void* beta, int64_t M, int64_t K,
                                    float eps, void* Xn_out, void* stream);

/*
 * coda_norm_backward -- the input gradient of RMSNorm / LayerNorm from the
 * gradient at the normalised value, g = gamma (.) dL/dy (y the norm's output),
 * and two row sums of it, all of which a dgrad GEMM's epilogue produces:
 *     x_hat = (x - mu) r,   S = r (sum_gx - mu sum_g)   (= sum_k g x_hat)
 *     dX    = r (g - sum_g / K - x_hat S / K)
 * RMSNorm: mu = NULL and sum_g = NULL (their terms are 0).  The CODA article
 * (d9bl.com, Fig. 4) decomposes the norms' gradients into a GEMM stage and an
 * epilogue stage; this correction needs the full-row sums of the GEMM output,
 * so it runs after it.  Typical chain (commuted LayerNorm forward, W unfolded):
 *   dgrad GEMM  A = dY, B = W (CODA_B_NK), ops
 *     COL_SUM(dbeta), COL_DOT_NORM(dgamma; rowvec r, mu; xhat = X),
 *     COL_SCALE(gamma), ROW_SUM(sum_g), ROW_DOT_AUX(sum_gx; xhat = X)
 *   -> D = g, then coda_norm_backward(g, X, r, mu, sum_g, sum_gx) -> dX.
 *   g, X, dX   bf16 [M, K] (16-byte aligned, K % 8 == 0); r, mu, sum_g,
 *   sum_gx fp32 [M].  dX must not overlap g or X.
 */
CODA_API coda_status coda_norm_backward(const void* g, const void* X, const float* r, const float* mu,
                                        const float* sum_g, const float* sum_gx, int64_t M, int64_t K, void* dX,
                                        void* stream);

/*
 * coda_quantize_e4m3_rows -- per-row FP8 quantisation for the E4M3 GEMM:
 *     amax_i = max_k |X[i,k]|,  scale_i = amax_i / 448,
 *     Q[i,k] = e4m3(X[i,k] * (448 / amax_i))   (round to nearest even, saturated
 *     to +-448; each product and quotient rounded to fp32; a zero row gives Q = 0,
 *     scale = 0), so X ~= e4m3 value * scale.
 *   X bf16 [M, K] (16-byte aligned, K % 16 == 0), Q uint8 [M, K], scale fp32 [M].
 */
CODA_API coda_status coda_quantize_e4m3_rows(const void* X, int64_t M, int64_t K, void* Q, float* scale,
                                             void* stream);

/*
 * MX (microscaling) FP8 operands.  The agentlenshq.com summary ("仕組み",
 * Scaling) makes scaling by a vector one of the epilogue's primitives; with
 * block-scaled FP8 the scaling moves inside the contraction: each block of 32
 * elements along K carries its own power-of-two scale, applied by the tensor
 * cores (tcgen05.mma kind::mxf8f6f4 block_scale) to every product before it is
 * accumulated.  Format: OCP Microscaling Formats (MX) v1.0, MXFP8 E4M3 -- E4M3
 * element codes, one E8M0 scale byte e per 32 elements (value 2^(e-127); 255 is
 * NaN and must not occur).
 *
 * Scale storage ("tiled"): for an operand of R rows and K columns, rows are
 * taken in groups of 128 and 32-element blocks in groups of 4, each group pair
 * forming a 512-byte tile, tiles ordered by row group then block group; the
 * scale of row r, block j (columns 32j .. 32j+31) is the byte at
 *     ((r / 128) * ceil(K / 128) + j / 4) * 512
 *       + (r % 32) * 16 + ((r % 128) / 32) * 4 + (j % 4).
 * One tile is exactly what the tensor cores read for 128 rows and 128
 * elements of K.  Positions beyond R rows or ceil(K/32) blocks are padding and
 * must hold a finite scale (the quantiser writes 127 there).
 */

/* Bytes of the tiled scale storage of an [R, K] MX operand (0 if R or K <= 0). */
CODA_API size_t coda_mx_scale_bytes(int64_t R, int64_t K);

/*
 * coda_quantize_mx_e4m3 -- MXFP8 quantisation of the rows of X (OCP MX v1.0
 * conversion): for each block of 32 elements along K, the shared exponent is
 * floor(log2(max |x|)) - 8 (E4M3's largest normal is 1.75 * 2^8), clamped to
 * [-127, 127]; codes are e4m3(x / 2^shared), rounded to nearest even and
 * saturated at +-448.  A block of zeros gets scale byte 0 and zero codes.
 *   X       bf16 [R, K], K % 32 == 0, 16-byte aligned
 *   Q       uint8 [R, K] E4M3 codes (output)
 *   scales  coda_mx_scale_bytes(R, K) bytes, tiled storage (output; padding 127)
 */
CODA_API coda_status coda_quantize_mx_e4m3(const void* X, int64_t R, int64_t K, void* Q, void* scales,
                                           void* stream);

/*
 * coda_gemm_epilogue_mx -- coda_gemm_epilogue with MXFP8 operands:
 *     C[i, j] = sum_k 2^(ea(i, k/32) - 127) A[i, k] * 2^(eb(j, k/32) - 127) B[j, k]
 * accumulated in fp32 by the tensor cores, then the op list as in
 * coda_gemm_epilogue.  A is E4M3 [M, K] and B is E4M3 [N, K] (both K-major: B in
 * the nn.Linear [out, in] layout); scale_A and scale_B are their tiled scales
 * (coda_mx_scale_bytes(M, K) and coda_mx_scale_bytes(N, K) bytes).  K must be a
 * multiple of 32; with SWIGLU, N/2 must be a multiple of 128 (the U half then
 * starts on a scale tile); RMS_ROWSCALE, RMS_SUMSQ_ROWSCALE and LN_ROWSCALE are
 * not available (they read bf16 A).  Other arguments, workspace and errors as
 * coda_gemm_epilogue; coda_workspace_size gives the workspace (the split over
 * K is not used with MX operands).
 */
CODA_API coda_status coda_gemm_epilogue_mx(const void* A, const void* scale_A, const void* B, const void* scale_B,
                                           int64_t M, int64_t N, int64_t K, const coda_epilogue* epi,
                                           const coda_aux* aux, void* D, float* row_stats,
                                           uint32_t* row_keep_count, void* workspace, size_t workspace_bytes,
                                           void* stream);

/*
 * coda_epilogue_apply -- the same op list applied by a separate memory-bound
 * kernel to a bf16 tensor C [M, N] already in global memory (the unfused form:
 * one read of C, one write of D).  RMS_ROWSCALE and LN_ROWSCALE are not
 * available here (they need the GEMM's A operand).  Reductions are finished inside this kernel, so it
 * needs no workspace.
 */
CODA_API coda_status coda_epilogue_apply(const void* C, int64_t M, int64_t N, const coda_epilogue* epi,
                                const coda_aux* aux, void* D, float* row_stats,
                                uint32_t* row_keep_count, void* stream);

/*
 * coda_check_device_error -- synchronises `stream`, then reads and clears the
 * current device's error word.  Returns CODA_ERR_TIMEOUT if a kernel gave up on
 * a pipeline wait since the last check (its outputs are then undefined),
 * CODA_ERR_CUDA if the synchronisation failed, else CODA_OK.  If `info` is
 * non-NULL it receives 4 words: code, block, role, tile of the first failure.
 */
CODA_API coda_status coda_check_device_error(void* stream, uint32_t* info);

/* Human-readable name of a status code (static string). */
CODA_API const char* coda_status_string(coda_status status);

/* Number of kernels this library has enqueued in this process (all devices). */
CODA_API uint64_t coda_launch_count(void);

/*
 * Tuning knobs, for measurement.  coda_set_pipeline_timeout_ns sets how long a
 * device-side pipeline wait may spin before the kernel records CODA_ERR_TIMEOUT
 * and exits (default 1e9 ns; 0 restores the default).  coda_set_max_ctas caps
 * the persistent grid (0 = one CTA per SM).  coda_set_cta_pair selects between
 * the single-CTA kernel and the CTA-pair kernel.
 */
CODA_API void coda_set_pipeline_timeout_ns(uint64_t ns);
CODA_API void coda_set_max_ctas(int32_t n);
/* 0 (default): CTA pairs (tcgen05 cta_group::2 on 256-row tiles, two SMs per
 * tile) when M > 128; 1: single-CTA 128-row tiles only; 2: CTA pairs whenever K > 0. */
CODA_API void coda_set_cta_pair(int32_t mode);
/* Split over K (stream-K): clusters take equal runs of (tile, 64-wide k-block)
 * units, CTAs that share a tile publish fp32 partial accumulators to the
 * workspace, and the last to finish applies the epilogue to their sum; no CTA
 * waits for another.  Two uses: a single-CTA problem with fewer tiles than SMs
 * splits all of its tiles; a problem of several waves of tiles runs whole
 * tiles up to its last two waves and splits the tiles of those, so that the
 * last, partly filled wave leaves no cluster idle.  0 (default): the first
 * when at most half of the SMs would have a tile, the second when the last
 * wave would leave more than 5% of the run's cluster time idle -- each where
 * the problem is eligible (see coda_workspace_size) and the workspace holds the
 * partials; 1: never; 2: whenever a problem has two k-blocks or more (the
 * second use needs at least two waves of tiles).  Results agree within
 * rounding: the sum over a split tile's K range is taken in another order. */
CODA_API void coda_set_split_k(int32_t mode);
/* Tile order of grids with more tiles than resident CTAs (clusters).
 * 0 (default): static -- a persistent grid walks tile0, tile0 + grid, ...;
 * 1: dynamic -- one cluster is launched per tile, and a running cluster takes
 * over the tile of a cluster that has not started yet (PTX cluster launch
 * control) whenever it is ready for more work, so clusters on faster SMs do
 * more tiles.  Split-K grids, a capped grid (coda_set_max_ctas) and the variant
 * with in-kernel row statistics always run the static order.  Results are
 * bit-identical either way. */
CODA_API void coda_set_tile_scheduler(int32_t dynamic);
/* Tile order (rasterisation) of the persistent grid, for measurement.  Tiles
 * run in groups: 1 = groups of `group` row blocks, the row block varying
 * fastest (A's rows of the group stay in L2 while B streams through once per
 * group); 2 = groups of `group` column blocks, the column block varying fastest
 * (B's columns of the group stay in L2 while A streams once per group);
 * 0 (default) = the library's choice: of the two, the one whose modelled DRAM
 * reads (A once + B once per row group, or B once + A once per column group,
 * with a group holding about 48 MB of the resident operand) are fewer.
 * group <= 0 with mode 1 or 2 takes the 48 MB group.  Results are bit-identical
 * in every order. */
CODA_API void coda_set_raster(int32_t mode, int32_t group);
/* 1 (default): once a CTA's last accumulator is complete, its producer, MMA and
 * other non-epilogue warps take half of that tile's epilogue chunks, loading
 * their own aux tiles (static tile order, no split over K, at most 16 tiles per
 * cluster, or 64 for op lists with aux tensors); 0: the epilogue warps alone.
 * Results are bit-identical either way. */
CODA_API void coda_set_tail_helpers(int32_t enable);

/* How the calling thread's last successful coda_gemm_epilogue call ran. */
typedef struct {
  int32_t pair;      /* 1: CTA-pair kernel (256-row tiles), 0: single CTA     */
  int32_t split;     /* 1: K split over CTAs (stream-K)                       */
  int32_t grid;      /* CTAs launched                                         */
  int32_t stages;    /* shared-memory pipeline stages                         */
  int64_t tiles;     /* output tiles                                          */
  int32_t prepass;   /* 1: a row-statistics pre-pass kernel ran first         */
  int32_t sequence;  /* 0: op-list interpreter; > 0: a fixed op sequence      */
  int32_t dynamic;   /* 1: dynamic tile order (cluster launch control)        */
  int32_t colvecs;   /* column-vector slices the epilogue reads per tile (bias,
                        column scales, LayerNorm's c and b): n > 0 copied to
                        shared memory per tile, -n prefetched into L1, 0 none */
} coda_plan;
CODA_API void coda_last_plan(coda_plan* out);

/* Fixed op sequences (the CODA article, d9bl.com, §3.3, compiles each
 * epilogue into a specialised kernel): for the op lists of the common blocks --
 * plain GEMM; RMS_ROWSCALE; LN_ROWSCALE; RESIDUAL; RESIDUAL, ROW_SUMSQ; BIAS;
 * BIAS, GELU_TANH; BIAS, GELU_ERF; BIAS, RESIDUAL; GELU_TANH; BIAS, GELU_TANH,
 * RESIDUAL; GELU_TANH_GRAD, ROW_DOT_AUX, ROW_SUM; SWIGLU; RMS_ROWSCALE, SWIGLU;
 * SWIGLU, DROPOUT (RMS_SUMSQ_ROWSCALE counts as RMS_ROWSCALE here); and, with
 * FP8 operands, ROW_SCALE, COL_SCALE_F32 (, SWIGLU) --
 * the library launches a kernel built with those opcodes fixed
 * (straight-line epilogue code); every other list runs the op interpreter.
 * Results are the same either way.  1 (default): use them; 0: interpret all. */
CODA_API void coda_set_fixed_sequences(int32_t enable);

#ifdef __cplusplus
}
#endif

#endif /* CODA_H */
