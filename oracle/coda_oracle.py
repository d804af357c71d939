"""Plain, slow, fp64 CPU oracle for the CODA GEMM+epilogue path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or run
this module: only the tests, the package smoke check and the benchmark's CPU
baseline leg use it.  It shares no code with the CUDA library.

What it computes.  The CODA article (d9bl.com, "CODA：将 Transformer 模块重新
表达为 GEMM+Epilogue 程序", §3.1 "GEMM+Epilogue 分解") defines the fused op as a
GEMM  C = alpha*A*B + beta*C_prev  followed by an epilogue  D = f(C)  applied
elementwise or row by row before the global write.  The agentlenshq.com summary
("CODA: GEMM-Epilogue FusionによるTransformerトレーニングの最適化", section
"仕組み") lists the primitive classes f is built from: scaling by a constant or
a vector, reductions (sum or mean along a dimension), pairwise/elementwise
transforms (activations), and accumulation into a residual.  The zeli.app page
("CODA: Wie Transformer-Blöcke als GEMM-Epilogue-Programme neu geschrieben
werden", comment by augment_me) adds the commuted RMSNorm: the row-wise scale
of the norm can be pulled past the following projection.

How it computes it.  Every step is a separate pass over a full fp64 tensor, in
the op-list order, with no intermediate rounding.  In particular the commuted
RMSNorm is evaluated the *unfused* way: normalise X first, then project (the
commuted form is only checked against this as a pin).  Inputs are the exact
bf16 values widened to fp64.  The GEMM uses numpy's fp64 matmul as a library
step; everything else is written out.

Readings where the pages are silent (each is also listed in the design notes):
  * GELU is the tanh form; its derivative is the tanh form's exact derivative.
    The exact form x * Phi(x) (GELU_ERF) and its derivative are separate ops.
  * dropout: keep element (row, col) of the [M, N_out] output iff
    splitmix64(seed, i) < T with i = row*N_out + col, where splitmix64(seed, i)
    is the i-th output (0-based) of the splitmix64 generator seeded with seed
    (Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
    OOPSLA 2014), and T = (uint64) floor(ldexp(1-p, 64)) evaluated in fp64.
    Kept values are scaled by 1/(1-p) (inverted dropout); p = 0 keeps all.
  * RMSNorm: r_i = 1/sqrt(mean_k x_ik^2 + eps); gamma scales the K index, so
    rmsnorm(X) @ W = r (.)_row (X @ (gamma (.)_row W)).
  * LayerNorm: mu_i = mean_k x_ik, r_i = 1/sqrt(mean_k (x_ik - mu_i)^2 + eps)
    (the biased variance); layernorm(X) = gamma (.) (x - mu) r + beta.
  * SwiGLU: the GEMM output is [G | U] with G = columns [0, N/2) and
    U = columns [N/2, N); out = silu(G) * U; ops before SWIGLU act on both
    halves (column vectors then have N entries), ops after it on N/2 columns.
  * row reductions run over the columns of the value at the op's position.
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# op names (the same names the C header uses, without the CODA_OP_ prefix)
# ---------------------------------------------------------------------------
OP_NAMES = (
    "SCALE", "COL_SCALE", "BIAS", "ROW_SCALE", "RMS_ROWSCALE", "GELU_TANH", "SILU",
    "SWIGLU", "GELU_TANH_GRAD", "DROPOUT", "RESIDUAL", "STORE_PREACT",
    "ROW_SUM", "ROW_MEAN", "ROW_SUMSQ", "ROW_DOT_AUX", "GELU_ERF", "GELU_ERF_GRAD", "LN_ROWSCALE",
    "COL_SUM", "COL_SUMSQ", "COL_DOT_AUX", "COL_DOT_NORM", "COL_SCALE_F32", "RMS_SUMSQ_ROWSCALE",
)

_U64 = np.uint64
_MASK64 = (1 << 64) - 1


# ---------------------------------------------------------------------------
# GEMM  (CODA article §3.1: C = alpha * A * B)
# ---------------------------------------------------------------------------
def gemm(A: np.ndarray, B: np.ndarray, b_layout: str = "kn") -> np.ndarray:
    """C[m, n] = sum_k A[m, k] * B(k, n) in fp64.

    b_layout "kn": B is stored [K, N] (row k, column n).
    b_layout "nk": B is stored [N, K] and the product is A @ B^T (the dgrad
                   form dY @ W^T with W stored [N, K]).
    """
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    if b_layout == "kn":
        return A @ B
    if b_layout == "nk":
        return A @ B.T
    raise ValueError(b_layout)


# ---------------------------------------------------------------------------
# RMSNorm, unfused (zeli.app page, augment_me's TLDR on RMSNorm/LayerNorm)
# ---------------------------------------------------------------------------
def rms_rstd(X: np.ndarray, eps: float) -> np.ndarray:
    """r_i = 1 / sqrt(mean_k x_ik^2 + eps), one value per row."""
    X = np.asarray(X, dtype=np.float64)
    ms = np.mean(X * X, axis=1)
    return 1.0 / np.sqrt(ms + eps)


def rmsnorm(X: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """Xn[i, k] = r_i * x_ik * gamma_k (the normalised activations, materialised)."""
    X = np.asarray(X, dtype=np.float64)
    r = rms_rstd(X, eps)
    return (r[:, None] * X) * np.asarray(gamma, dtype=np.float64)[None, :]


def rmsnorm_project(X, gamma, W, eps, b_layout="kn"):
    """Normalise-then-project: rmsnorm(X) @ W (the unfused reading)."""
    return gemm(rmsnorm(X, gamma, eps), W, b_layout)


def rms_rstd_from_sumsq(sumsq, K: int, eps: float) -> np.ndarray:
    """r_i = 1 / sqrt(s_i / K + eps) from given row sums of squares s_i = sum_k x_ik^2
    (the same r as rms_rstd when s is X's own): the commuted norm whose row
    statistics were gathered by an earlier pass over X (for X produced by a
    residual epilogue, that epilogue's row sum of squares)."""
    s = np.asarray(sumsq, dtype=np.float64)
    return 1.0 / np.sqrt(s / float(K) + eps)


def ln_stats(X: np.ndarray, eps: float):
    """mu_i = mean_k x_ik and r_i = 1 / sqrt(mean_k (x_ik - mu_i)^2 + eps)."""
    X = np.asarray(X, dtype=np.float64)
    mu = np.mean(X, axis=1)
    var = np.mean((X - mu[:, None]) ** 2, axis=1)
    return mu, 1.0 / np.sqrt(var + eps)


def layernorm(X, gamma, beta, eps):
    """Xn[i, k] = gamma_k (x_ik - mu_i) r_i + beta_k (beta None: 0)."""
    X = np.asarray(X, dtype=np.float64)
    mu, r = ln_stats(X, eps)
    out = (X - mu[:, None]) * r[:, None] * np.asarray(gamma, dtype=np.float64)[None, :]
    if beta is not None:
        out = out + np.asarray(beta, dtype=np.float64)[None, :]
    return out


def layernorm_project(X, gamma, beta, W, eps, b_layout="kn"):
    """Normalise-then-project: layernorm(X) @ W (the unfused reading)."""
    return gemm(layernorm(X, gamma, beta, eps), W, b_layout)


def rmsnorm_backward(X, gamma, dY, eps):
    """Gradients of sum(rmsnorm(X; gamma) * dY): y = gamma x_hat, x_hat = x r,
    r = 1/sqrt(mean_k x^2 + eps).  With g = gamma dY (the gradient at x_hat):
      dX = r (g - x_hat mean_k(g x_hat)),  dgamma = sum_i dY x_hat.
    Returns (dX, dgamma)."""
    X = np.asarray(X, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    gamma = np.asarray(gamma, dtype=np.float64)
    r = rms_rstd(X, eps)
    xh = X * r[:, None]
    g = dY * gamma[None, :]
    dX = r[:, None] * (g - xh * np.mean(g * xh, axis=1)[:, None])
    return dX, np.sum(dY * xh, axis=0)


def layernorm_backward(X, gamma, dY, eps):
    """Gradients of sum(layernorm(X; gamma, beta) * dY): y = gamma x_hat + beta,
    x_hat = (x - mu) r.  With g = gamma dY:
      dX = r (g - mean_k g - x_hat mean_k(g x_hat)),
      dgamma = sum_i dY x_hat,  dbeta = sum_i dY.
    Returns (dX, dgamma, dbeta)."""
    X = np.asarray(X, dtype=np.float64)
    dY = np.asarray(dY, dtype=np.float64)
    gamma = np.asarray(gamma, dtype=np.float64)
    mu, r = ln_stats(X, eps)
    xh = (X - mu[:, None]) * r[:, None]
    g = dY * gamma[None, :]
    dX = r[:, None] * (g - np.mean(g, axis=1)[:, None] - xh * np.mean(g * xh, axis=1)[:, None])
    return dX, np.sum(dY * xh, axis=0), np.sum(dY, axis=0)


# ---------------------------------------------------------------------------
# scaling primitives (agentlenshq.com, "仕組み": Scaling by a constant or vector)
# ---------------------------------------------------------------------------
def scale(x, alpha):
    return x * float(alpha)


def col_scale(x, v):
    return x * np.asarray(v, dtype=np.float64)[None, :]


def bias(x, v):
    return x + np.asarray(v, dtype=np.float64)[None, :]


def row_scale(x, v):
    return x * np.asarray(v, dtype=np.float64)[:, None]


# ---------------------------------------------------------------------------
# elementwise transforms (agentlenshq.com, "Pairwise Transformations";
# CODA article §3.2 DSL example uses gelu)
# ---------------------------------------------------------------------------
_SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
_GELU_C = 0.044715


def gelu_tanh(x):
    """0.5 x (1 + tanh( sqrt(2/pi) (x + 0.044715 x^3) ))."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(_SQRT_2_OVER_PI * (x + _GELU_C * x ** 3)))


def gelu_tanh_grad(z):
    """d/dz of gelu_tanh(z), by the product and chain rules:
    0.5 (1 + t) + 0.5 z (1 - t^2) sqrt(2/pi) (1 + 3 * 0.044715 z^2),
    t = tanh(sqrt(2/pi)(z + 0.044715 z^3))."""
    z = np.asarray(z, dtype=np.float64)
    t = np.tanh(_SQRT_2_OVER_PI * (z + _GELU_C * z ** 3))
    dinner = _SQRT_2_OVER_PI * (1.0 + 3.0 * _GELU_C * z * z)
    return 0.5 * (1.0 + t) + 0.5 * z * (1.0 - t * t) * dinner


_erf = np.vectorize(math.erf, otypes=[np.float64])


def gelu_erf(x):
    """The exact GELU: x * Phi(x) = 0.5 x (1 + erf(x / sqrt(2)))."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + _erf(x / math.sqrt(2.0)))


def gelu_erf_grad(z):
    """d/dz [z Phi(z)] = Phi(z) + z phi(z), phi(z) = exp(-z^2/2) / sqrt(2 pi)."""
    z = np.asarray(z, dtype=np.float64)
    return 0.5 * (1.0 + _erf(z / math.sqrt(2.0))) + z * np.exp(-0.5 * z * z) / math.sqrt(2.0 * math.pi)


def silu(x):
    """x * sigmoid(x) = x / (1 + exp(-x))."""
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def swiglu(c):
    """[G | U] -> silu(G) * U, G = columns [0, N/2), U = columns [N/2, N)."""
    n = c.shape[1]
    if n % 2:
        raise ValueError("SWIGLU needs an even width")
    h = n // 2
    return silu(c[:, :h]) * c[:, h:]


# ---------------------------------------------------------------------------
# dropout (CODA article §3.2 DSL example: dropout(output, 0.1))
# ---------------------------------------------------------------------------
SPLITMIX_GAMMA = 0x9E3779B97F4A7C15
SPLITMIX_M1 = 0xBF58476D1CE4E5B9
SPLITMIX_M2 = 0x94D049BB133111EB


def splitmix64(seed: int, idx) -> np.ndarray:
    """The idx-th (0-based) output of splitmix64 seeded with `seed`.

    splitmix64 advances its state by the odd constant 0x9E3779B97F4A7C15 before
    each output and returns mix64(state):
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
        z = (z ^ (z >> 27)) * 0x94D049BB133111EB
        z =  z ^ (z >> 31)
    all modulo 2^64, so output idx is mix64(seed + (idx + 1) * gamma).
    """
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = _U64(seed & _MASK64) + (idx + _U64(1)) * _U64(SPLITMIX_GAMMA)
        z = (z ^ (z >> _U64(30))) * _U64(SPLITMIX_M1)
        z = (z ^ (z >> _U64(27))) * _U64(SPLITMIX_M2)
        z = z ^ (z >> _U64(31))
    return z


def dropout_threshold(p: float) -> int:
    """T = floor((1-p) * 2^64) evaluated in fp64; None means keep everything
    (p = 0, or p so small that (1-p) * 2^64 is not below 2^64)."""
    if not (0.0 <= p < 1.0):
        raise ValueError("dropout p must be in [0, 1)")
    if p == 0.0:
        return None
    t = math.ldexp(1.0 - p, 64)
    if t >= 2.0 ** 64:
        return None
    return int(t)


def dropout_mask(seed: int, M: int, N: int, p: float, row0: int = 0, rows=None) -> np.ndarray:
    """keep[m, n] for the rows given (default row0 .. row0+M-1) of an [*, N] output."""
    T = dropout_threshold(p)
    if rows is None:
        rows = np.arange(row0, row0 + M, dtype=np.uint64)
    rows = np.asarray(rows, dtype=np.uint64)
    if T is None:
        return np.ones((rows.size, N), dtype=bool)
    idx = rows[:, None] * _U64(N) + np.arange(N, dtype=np.uint64)[None, :]
    return splitmix64(seed, idx) < _U64(T)


def dropout(x, p, seed, rows=None):
    """keep ? x / (1-p) : 0, plus the keep mask."""
    keep = dropout_mask(seed, x.shape[0], x.shape[1], p, rows=rows)
    if p == 0.0:
        return x.copy(), keep
    return np.where(keep, x / (1.0 - p), 0.0), keep


# ---------------------------------------------------------------------------
# accumulation (CODA article §3.1 beta*C_prev; agentlenshq.com "Accumulation")
# ---------------------------------------------------------------------------
def residual(x, R, beta=1.0):
    return x + float(beta) * np.asarray(R, dtype=np.float64)


# ---------------------------------------------------------------------------
# row reductions (agentlenshq.com, "Reductions": sum or mean along a dimension)
# ---------------------------------------------------------------------------
def col_sum(X) -> np.ndarray:
    """sum_i X[i, j]: the reduction over the rows (the M dimension)."""
    return np.sum(np.asarray(X, dtype=np.float64), axis=0)


def row_sum(x):
    return np.sum(x, axis=1)


def row_mean(x):
    return np.mean(x, axis=1)


def row_sumsq(x):
    return np.sum(x * x, axis=1)


def row_dot(x, aux):
    return np.sum(x * np.asarray(aux, dtype=np.float64), axis=1)


# ---------------------------------------------------------------------------
# the whole epilogue program, as separate passes in op-list order
# ---------------------------------------------------------------------------
def run_chain(A, B, ops, *, b_layout="kn", seed=0, col_vecs=None, row_vecs=None,
              residual_t=None, z=None, xhat=None, norm_gamma=None, norm_beta=None, ln_colsum=None,
              ln_bias=None, col_scale_f32=None, rows=None):
    """Evaluate D = f(A @ B) for an op list, one unfused pass per op.

    ops: sequence of (name, slot, f0) tuples, names from OP_NAMES; f0 is taken
        as the float32 the op list carries (widened exactly to fp64).
    col_vecs / row_vecs: dict slot -> vector (bf16 values widened).
    residual_t, z, xhat: [M, N_out] aux tensors (or only the sampled rows).
    norm_gamma: if given, the op list must begin with RMS_ROWSCALE,
        RMS_SUMSQ_ROWSCALE or LN_ROWSCALE; the GEMM is then evaluated as
        rmsnorm(A; gamma) @ B or layernorm(A; gamma, norm_beta) @ B (normalise,
        then project), with B the *unscaled* weight (RMS_SUMSQ_ROWSCALE takes
        its row sums of squares from row_vecs[slot] instead of from A).
        Without norm_gamma these ops scale the product by the row factor r_i
        (B then already holds gamma (.)_row W).
    ln_colsum / ln_bias: the c and b vectors of an LN_ROWSCALE evaluated as
        written (x = r (x - mu c) + b) when the norm is not given unfused.
    rows: absolute row indices of the rows of A given (used by dropout's
        counter and nothing else); default 0..M-1.

    Returns dict with D (fp64), stats {slot: fp64[M]}, stat_scale {slot: fp64[M]}
    (the error scale of each row reduction: the L2 norm over its summands of
    d(summand)/d(log x), i.e. how far the sum moves when every chain value x
    carries an independent relative error of 1 -- the summand itself for the
    linear reductions, twice it for the sums of squares), col_stats
    {slot: fp64[N_out]} and col_stat_scale (the same for the column reductions,
    which need all M rows: not with `rows`), keep_count (int64[M] or None),
    keep (bool mask or None), preact (fp64 or None).
    """
    A = np.asarray(A, dtype=np.float64)
    col_vecs = col_vecs or {}
    row_vecs = row_vecs or {}
    M = A.shape[0]
    if rows is None:
        rows = np.arange(M)
    # op parameters are float32 in the op list; use exactly those values
    ops = [(o[0], o[1] if len(o) > 1 else 0, float(np.float32(o[2])) if len(o) > 2 else 0.0) for o in ops]

    start = 0
    stats = {}
    if norm_gamma is not None:
        name, slot, eps = ops[0]
        if name == "RMS_ROWSCALE":
            x = rmsnorm_project(A, norm_gamma, B, eps, b_layout)
            if slot is not None and slot >= 0:
                stats[slot] = rms_rstd(A, eps)
        elif name == "LN_ROWSCALE":
            x = layernorm_project(A, norm_gamma, norm_beta, B, eps, b_layout)
            if slot is not None and slot >= 0:
                mu, r = ln_stats(A, eps)
                stats[slot] = r
                stats[slot + 1] = mu
        elif name == "RMS_SUMSQ_ROWSCALE":
            # normalise with r from the given row sums of squares, then project
            r = rms_rstd_from_sumsq(row_vecs[slot], A.shape[1], eps)
            xn = (r[:, None] * A) * np.asarray(norm_gamma, dtype=np.float64)[None, :]
            x = gemm(xn, B, b_layout)
        else:
            raise ValueError("norm_gamma needs RMS_ROWSCALE, RMS_SUMSQ_ROWSCALE or LN_ROWSCALE as the first op")
        start = 1
    else:
        x = gemm(A, B, b_layout)

    keep_count = None
    keep = None
    preact = None
    stat_scale = {}
    col_stats = {}
    col_stat_scale = {}
    for name, slot, f0 in ops[start:]:
        if name == "SCALE":
            x = scale(x, f0)
        elif name == "COL_SCALE":
            x = col_scale(x, col_vecs[slot])
        elif name == "BIAS":
            x = bias(x, col_vecs[slot])
        elif name == "COL_SCALE_F32":
            x = col_scale(x, col_scale_f32)
        elif name == "ROW_SCALE":
            x = row_scale(x, row_vecs[slot])
        elif name == "RMS_ROWSCALE":
            r = rms_rstd(A, f0)
            x = row_scale(x, r)
            if slot is not None and slot >= 0:
                stats[slot] = r
        elif name == "RMS_SUMSQ_ROWSCALE":
            x = row_scale(x, rms_rstd_from_sumsq(row_vecs[slot], A.shape[1], f0))
        elif name == "LN_ROWSCALE":
            mu, r = ln_stats(A, f0)
            c = np.asarray(ln_colsum, dtype=np.float64)
            b = np.zeros_like(c) if ln_bias is None else np.asarray(ln_bias, dtype=np.float64)
            if x.shape[1] != c.shape[0]:
                raise ValueError("LN_ROWSCALE vectors must match the width")
            x = r[:, None] * (x - mu[:, None] * c[None, :]) + b[None, :]
            if slot is not None and slot >= 0:
                stats[slot] = r
                stats[slot + 1] = mu
        elif name == "GELU_TANH":
            x = gelu_tanh(x)
        elif name == "SILU":
            x = silu(x)
        elif name == "GELU_ERF":
            x = gelu_erf(x)
        elif name == "GELU_ERF_GRAD":
            x = x * gelu_erf_grad(z)
        elif name == "SWIGLU":
            x = swiglu(x)
        elif name == "GELU_TANH_GRAD":
            x = x * gelu_tanh_grad(z)
        elif name == "DROPOUT":
            x, keep = dropout(x, f0, seed, rows=rows)
            keep_count = keep.sum(axis=1).astype(np.int64)
        elif name == "RESIDUAL":
            x = residual(x, residual_t, f0)
        elif name == "STORE_PREACT":
            preact = x.copy()
        elif name == "ROW_SUM":
            stats[slot] = row_sum(x)
            stat_scale[slot] = np.sqrt(row_sumsq(x))
        elif name == "ROW_MEAN":
            stats[slot] = row_mean(x)
            stat_scale[slot] = np.sqrt(row_sumsq(x)) / x.shape[1]
        elif name == "ROW_SUMSQ":
            stats[slot] = row_sumsq(x)
            stat_scale[slot] = 2.0 * np.sqrt(row_sumsq(x * x))
        elif name == "ROW_DOT_AUX":
            stats[slot] = row_dot(x, xhat)
            stat_scale[slot] = np.sqrt(row_sumsq(x * np.asarray(xhat, dtype=np.float64)))
        elif name in ("COL_SUM", "COL_SUMSQ", "COL_DOT_AUX", "COL_DOT_NORM"):
            if name == "COL_SUM":
                t = x
            elif name == "COL_SUMSQ":
                t = x * x
            elif name == "COL_DOT_AUX":
                t = x * np.asarray(xhat, dtype=np.float64)
            else:
                # x_hat = r (aux - mu), r = row vector 0, mu = row vector 1 (or 0)
                rr = np.asarray(row_vecs[0], dtype=np.float64)
                mm = np.asarray(row_vecs[1], dtype=np.float64) if 1 in row_vecs else np.zeros_like(rr)
                t = x * (rr[:, None] * (np.asarray(xhat, dtype=np.float64) - mm[:, None]))
            col_stats[slot] = col_sum(t)
            col_stat_scale[slot] = (2.0 if name == "COL_SUMSQ" else 1.0) * np.sqrt(col_sum(t * t))
        else:
            raise ValueError(f"unknown op {name}")
    return dict(D=x, stats=stats, stat_scale=stat_scale, col_stats=col_stats, col_stat_scale=col_stat_scale,
                keep_count=keep_count, keep=keep, preact=preact)


def round_bf16(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (8 significant bits), ties to
    even: the rounding every library call applies to its bf16 outputs.  Used
    where a workload chains calls, so the oracle rounds the outputs of its calls
    the same way.  (Normal range only; no overflow or subnormal handling.)"""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                    # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.round(m * 256.0) / 256.0, e)   # np.round: half to even


# ---------------------------------------------------------------------------
# FP8 E4M3 (the OCP 8-bit floating-point format with 4 exponent bits, bias 7,
# 3 mantissa bits, no infinities; S.1111.111 is NaN, so the largest finite
# magnitude is 1.75 * 2^8 = 448; exponent field 0 holds the subnormals m/8 * 2^-6)
# ---------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_decode(code) -> np.ndarray:
    """Value of each E4M3 byte (fp64); NaN for the two NaN codes."""
    c = np.asarray(code, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & ((c & 0x7) == 7), np.nan, mag)
    return sign * mag


_E4M3_POS = e4m3_decode(np.arange(0, 0x7F))     # the 127 non-negative finite values, codes 0x00..0x7E


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 code to each value, ties to the even code (mantissa LSB 0),
    magnitudes beyond 448 saturated to 448 (the 'satfinite' convention), NaN to
    0x7F, and the sign kept (a negative value that rounds to zero gives 0x80).
    For each magnitude the two neighbouring entries of the table of finite
    values are compared (searchsorted over the sorted table)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, len(_E4M3_POS) - 1)
    lo = np.clip(hi - 1, 0, len(_E4M3_POS) - 1)
    d_lo = np.abs(a - _E4M3_POS[lo])
    d_hi = np.abs(_E4M3_POS[hi] - a)
    code = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = code.astype(np.uint8) | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def quantize_rows_e4m3(X):
    """Per-row FP8 quantisation, in float32 arithmetic (as the GPU kernel):
    amax_i = max_k |x_ik|, scale_i = amax_i / 448, q_ik = e4m3(x_ik * (448 / amax_i))
    (each product and quotient rounded to float32), q = 0 and scale = 0 for a zero row.
    Returns (codes uint8 [M, K], scale float32 [M]); x ~= decode(q) * scale."""
    X = np.asarray(X, dtype=np.float32)
    amax = np.max(np.abs(X), axis=1)
    with np.errstate(divide="ignore"):
        inv = np.where(amax > 0, np.float32(E4M3_MAX) / amax, np.float32(0)).astype(np.float32)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    y = (X * inv[:, None]).astype(np.float32)
    return e4m3_encode(y.astype(np.float64)), scale


# ---------------------------------------------------------------------------
# MX (microscaling) E4M3 -- block-scaled FP8: the agentlenshq.com summary's
# scaling primitive (section "仕組み": scaling by a vector) applied per block
# of 32 elements along K.  The format is the OCP Microscaling Formats (MX)
# specification v1.0 (2023): a block of 32 E4M3 elements P_i shares one E8M0
# scale X (a bare exponent byte e, X = 2^(e-127), e = 255 is NaN); the block's
# values are X * P_i.  Conversion (the specification's algorithm): the shared
# exponent is floor(log2(max_i |V_i|)) - emax_elem, with emax_elem = 8 for E4M3
# (448 = 1.75 * 2^8), clamped to the scale's range [-127, 127]; then
# P_i = e4m3(V_i / X), rounded to nearest even and saturated at +-448.
# ---------------------------------------------------------------------------
MX_BLOCK = 32
E4M3_EMAX = 8


def e8m0_decode(e) -> np.ndarray:
    """X = 2^(e - 127) for each scale byte, NaN for 255."""
    e = np.asarray(e, dtype=np.int64) & 0xFF
    return np.where(e == 255, np.nan, np.exp2(e.astype(np.float64) - 127.0))


def quantize_mx_e4m3(X):
    """MX E4M3 quantisation of each row of X [R, K] in blocks of 32 along K (the
    last block of a row may be shorter).  Returns (codes uint8 [R, K], scale
    bytes uint8 [R, ceil(K/32)]).  A block of zeros gets scale byte 0 and zero
    codes.  Per block, from the definition: the shared exponent from the exact
    binary exponent of the block maximum (frexp: amax = m 2^e with 0.5 <= m < 1,
    so floor(log2 amax) = e - 1), clamped; the division by that power of two,
    exact in fp64; then round-to-nearest-even onto the E4M3 grid with saturation
    (e4m3_encode).  The blocks are processed as one array."""
    X = np.asarray(X, dtype=np.float64)
    R, K = X.shape
    nb = (K + MX_BLOCK - 1) // MX_BLOCK
    padded = np.zeros((R, nb * MX_BLOCK))
    padded[:, :K] = X
    blocks = padded.reshape(R, nb, MX_BLOCK)
    amax = np.max(np.abs(blocks), axis=2)
    _, e = np.frexp(amax)
    shared = np.clip((e - 1) - E4M3_EMAX, -127, 127)
    shared = np.where(amax == 0.0, -127, shared)
    codes = e4m3_encode(blocks / np.ldexp(1.0, shared)[:, :, None]).reshape(R, nb * MX_BLOCK)[:, :K]
    return np.ascontiguousarray(codes), (shared + 127).astype(np.uint8)


def dequantize_mx(codes, sexp) -> np.ndarray:
    """fp64 values X_block * P_i of MX E4M3 data (codes [R, K], scale bytes [R, ceil(K/32)])."""
    codes = np.asarray(codes)
    R, K = codes.shape
    scale = np.repeat(e8m0_decode(sexp), MX_BLOCK, axis=1)[:, :K]
    return e4m3_decode(codes) * scale


def mx_scale_offset(r: int, j: int, K: int) -> int:
    """Byte offset of the scale of row r, 32-element block j in the library's
    tiled scale storage (the layout coda.h defines for MX operands): rows in
    groups of 128 and blocks in groups of 4 form 512-byte tiles, tiles ordered
    by row group then block group, and inside a tile the scale of (row r,
    block j) at (r % 32) * 16 + ((r % 128) // 32) * 4 + (j % 4)."""
    kb = (K + 127) // 128
    return ((r // 128) * kb + j // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (j % 4)


def mx_scale_bytes(R: int, K: int) -> int:
    """Size of the tiled scale storage of an [R, K] MX operand (rows padded to
    128, blocks to 4 per row)."""
    return ((R + 127) // 128) * ((K + 127) // 128) * 512


def mx_scales_from_tiled(buf, R: int, K: int) -> np.ndarray:
    """Scale bytes [R, ceil(K/32)] read out of the tiled storage, element by element."""
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    nb = (K + MX_BLOCK - 1) // MX_BLOCK
    out = np.zeros((R, nb), dtype=np.uint8)
    for r in range(R):
        for j in range(nb):
            out[r, j] = buf[mx_scale_offset(r, j, K)]
    return out


def to_f64(t) -> np.ndarray:
    """Widen a tensor (torch bf16/fp32 or numpy) to an fp64 numpy array exactly."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)
