"""Pins for the fp64 oracle: checks against closed forms, brute force, textbook
identities and published known answers -- never against the oracle itself.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong constant) fails it.
"""
import math
import os

import numpy as np
import pytest

from oracle import coda_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


# ---------------------------------------------------------------- GEMM ------
def _brute_gemm(A, B, layout):
    M, K = len(A), len(A[0])
    N = len(B[0]) if layout == "kn" else len(B)
    C = [[0.0] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            s = 0.0
            for k in range(K):
                b = B[k][j] if layout == "kn" else B[j][k]
                s += A[i][k] * b
            C[i][j] = s
    return np.array(C)


@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_gemm_brute_force_8x8x8(layout):
    A = rng.standard_normal((8, 8))
    B = rng.standard_normal((8, 8))
    ref = _brute_gemm(A.tolist(), B.tolist(), layout)
    np.testing.assert_allclose(O.gemm(A, B, layout), ref, rtol=1e-13, atol=1e-13)


def test_gemm_brute_force_rectangular():
    A = rng.standard_normal((5, 7))
    B = rng.standard_normal((7, 3))
    np.testing.assert_allclose(O.gemm(A, B, "kn"), _brute_gemm(A.tolist(), B.tolist(), "kn"), rtol=1e-13)
    np.testing.assert_allclose(O.gemm(A, B.T.copy(), "nk"), _brute_gemm(A.tolist(), B.tolist(), "kn"),
                               rtol=1e-13)


def test_gemm_identity_and_one_hot():
    B = rng.standard_normal((6, 9))
    np.testing.assert_array_equal(O.gemm(np.eye(6), B, "kn"), B)
    A = np.zeros((4, 6))
    A[2, 5] = 1.0                      # e_2 e_5^T picks row 5 of B into row 2
    C = O.gemm(A, B, "kn")
    np.testing.assert_array_equal(C[2], B[5])
    assert np.count_nonzero(C[[0, 1, 3]]) == 0
    # [N,K] layout: C[i, n] = B[n, k]
    Bnk = rng.standard_normal((9, 6))
    C = O.gemm(A, Bnk, "nk")
    np.testing.assert_array_equal(C[2], Bnk[:, 5])


def test_gemm_small_integers_exact():
    A = rng.integers(-8, 9, (33, 64)).astype(np.float64)
    B = rng.integers(-8, 9, (64, 17)).astype(np.float64)
    ref = np.zeros((33, 17))
    for k in range(64):                 # exact integer accumulation
        ref += np.outer(A[:, k], B[k])
    np.testing.assert_array_equal(O.gemm(A, B), ref)


# ---------------------------------------------------------------- GELU ------
def _gelu_erf(x):
    return 0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0)))


def test_gelu_closed_forms():
    assert O.gelu_tanh(0.0) == 0.0
    x = np.linspace(-6, 6, 1201)
    # odd part: gelu(x) - gelu(-x) = x exactly, because tanh is odd
    np.testing.assert_allclose(O.gelu_tanh(x) - O.gelu_tanh(-x), x, atol=1e-14)
    assert abs(O.gelu_tanh(30.0) - 30.0) < 1e-12
    assert abs(O.gelu_tanh(-30.0)) < 1e-12


def test_gelu_tanh_close_to_exact_erf_gelu():
    # The tanh form approximates x*Phi(x) to within 4.8e-4 everywhere; a wrong
    # coefficient (0.04 or 0.05 instead of 0.044715, sqrt(2)/pi, x^2 for x^3)
    # moves it to >= 2.8e-3.
    x = np.linspace(-10, 10, 40001)
    exact = np.array([_gelu_erf(v) for v in x])
    err = np.abs(O.gelu_tanh(x) - exact).max()
    assert err < 5e-4, err


def test_gelu_grad_matches_finite_difference():
    z = np.linspace(-7, 7, 1401)
    h = 1e-5
    fd = (O.gelu_tanh(z + h) - O.gelu_tanh(z - h)) / (2 * h)
    np.testing.assert_allclose(O.gelu_tanh_grad(z), fd, atol=1e-9)
    assert O.gelu_tanh_grad(0.0) == 0.5
    assert abs(O.gelu_tanh_grad(40.0) - 1.0) < 1e-12


# ---------------------------------------------------------------- SiLU ------
def test_silu_closed_forms():
    assert O.silu(0.0) == 0.0
    x = np.linspace(-20, 20, 801)
    np.testing.assert_allclose(O.silu(x) - O.silu(-x), x, atol=1e-13)
    # sigmoid(x) = (1 + tanh(x/2)) / 2, an independent closed form
    np.testing.assert_allclose(O.silu(x), 0.5 * x * (1.0 + np.tanh(0.5 * x)), rtol=1e-13, atol=1e-15)
    assert abs(O.silu(50.0) - 50.0) < 1e-12


def test_swiglu_pairs_halves_not_interleaved():
    n = 6
    G = np.arange(1, n + 1, dtype=np.float64)[None, :]
    U = 10.0 + np.arange(n, dtype=np.float64)[None, :]
    out = O.swiglu(np.concatenate([G, U], axis=1))
    expect = np.array([[(j + 1) / (1 + math.exp(-(j + 1))) * (10 + j) for j in range(n)]])
    np.testing.assert_allclose(out, expect, rtol=1e-14)
    assert np.count_nonzero(O.swiglu(np.concatenate([G, 0 * U], axis=1))) == 0


# ------------------------------------------------------------- RMSNorm ------
def test_rmsnorm_constant_row():
    K, c, eps = 64, 3.0, 1e-6
    X = np.full((2, K), c)
    X[1] = -c
    gamma = rng.uniform(0.5, 1.5, K)
    Xn = O.rmsnorm(X, gamma, eps)
    f = c / math.sqrt(c * c + eps)
    np.testing.assert_allclose(Xn[0], gamma * f, rtol=1e-15)
    np.testing.assert_allclose(Xn[1], -gamma * f, rtol=1e-15)


def test_rms_rstd_hand_value():
    X = np.array([[3.0, 4.0]])          # mean square 12.5
    assert abs(O.rms_rstd(X, 0.5)[0] - 1.0 / math.sqrt(13.0)) < 1e-16
    X = np.zeros((1, 10))
    X[0, 3] = 2.0                        # mean square 0.4
    assert abs(O.rms_rstd(X, 1e-6)[0] - 1.0 / math.sqrt(0.4 + 1e-6)) < 1e-15


def test_commuted_rmsnorm_identity():
    # zeli.app (augment_me): the row-wise scale of the norm commutes past the
    # projection: rmsnorm(X) @ W == r (.)_row (X @ (gamma (.)_row W)).
    X = rng.standard_normal((40, 32))
    gamma = rng.uniform(0.5, 1.5, 32)
    W = rng.standard_normal((32, 24))
    lhs = O.rmsnorm_project(X, gamma, W, 1e-6)
    r = O.rms_rstd(X, 1e-6)
    rhs = r[:, None] * (X @ (gamma[:, None] * W))
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- dropout ------
def _golden_splitmix():
    vals = []
    with open(os.path.join(GOLDEN, "splitmix64_seed0.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                vals.append(int(line, 16))
    return vals


def test_splitmix64_known_answers():
    expect = _golden_splitmix()
    got = [int(v) for v in O.splitmix64(0, np.arange(len(expect)))]
    assert got == expect


def test_dropout_threshold_value():
    # (1 - 0.1) in fp64 times 2^64, truncated: 0.9 is 0x3FECCCCCCCCCCCCD
    assert O.dropout_threshold(0.1) == 0xE666666666666800
    assert O.dropout_threshold(0.1) == 16602069666338596864
    assert O.dropout_threshold(0.5) == 1 << 63
    assert O.dropout_threshold(0.0) is None


def test_dropout_mask_known_answers_and_flat_index():
    kat = _golden_splitmix()
    T = O.dropout_threshold(0.1)
    # the [1,5] output's element i uses stream position i
    keep = O.dropout_mask(0, 1, 5, 0.1)
    assert keep[0].tolist() == [v < T for v in kat]
    # the counter is the row-major flat index of the [M, N] output
    m, n = 7, 13
    a = O.dropout_mask(5, m, n, 0.1)
    b = O.dropout_mask(5, 1, m * n, 0.1).reshape(m, n)
    np.testing.assert_array_equal(a, b)
    c = O.dropout_mask(5, 1, n, 0.1, rows=[3])
    np.testing.assert_array_equal(a[3], c[0])


def test_dropout_keep_rate_three_sigma():
    p = 0.1
    keep = O.dropout_mask(0, 512, 8192, p)
    n = keep.size
    rate = keep.mean()
    sigma = math.sqrt(p * (1 - p) / n)
    assert abs(rate - (1 - p)) < 3 * sigma, (rate, sigma)
    # rows and columns are not correlated with position: per-row rates spread like binomials
    per_row = keep.mean(axis=1)
    assert abs(per_row.std() - math.sqrt(p * (1 - p) / 8192)) < 0.25 * math.sqrt(p * (1 - p) / 8192)


def test_dropout_scaling_and_identity():
    x = rng.standard_normal((16, 40))
    y, keep = O.dropout(x, 0.25, 3)
    np.testing.assert_array_equal(y[~keep], 0.0)
    np.testing.assert_allclose(y[keep], x[keep] / 0.75, rtol=1e-15)
    y0, k0 = O.dropout(x, 0.0, 3)
    np.testing.assert_array_equal(y0, x)
    assert k0.all()


# ---------------------------------------------------------- reductions ------
def test_row_reductions_closed_forms():
    N = 100
    x = np.tile(np.arange(N, dtype=np.float64), (3, 1))
    x[1] = 1.0
    assert O.row_sum(x)[0] == N * (N - 1) / 2
    assert O.row_sumsq(x)[0] == (N - 1) * N * (2 * N - 1) / 6
    assert O.row_mean(x)[0] == (N - 1) / 2
    assert O.row_sum(x)[1] == N and O.row_sumsq(x)[1] == N and O.row_mean(x)[1] == 1.0
    np.testing.assert_array_equal(O.row_dot(x, np.ones_like(x)), O.row_sum(x))


def test_residual_cancels():
    A = rng.standard_normal((9, 11))
    B = rng.standard_normal((11, 13))
    C = A @ B
    out = O.run_chain(A, B, [("RESIDUAL", 0, 1.0)], residual_t=-C)["D"]
    assert np.abs(out).max() < 1e-12


# --------------------------------------------------------------- chain ------
def test_chain_zero_gemm_closed_form():
    # A = 0 makes C = 0, so D = gelu(bias) + residual elementwise
    M, K, N = 5, 4, 6
    b = rng.standard_normal(N)
    R = rng.standard_normal((M, N))
    out = O.run_chain(np.zeros((M, K)), rng.standard_normal((K, N)),
                      [("BIAS", 0), ("GELU_TANH",), ("RESIDUAL", 0, 1.0)],
                      col_vecs={0: b}, residual_t=R)["D"]
    expect = np.array([[0.5 * v * (1 + math.tanh(math.sqrt(2 / math.pi) * (v + 0.044715 * v ** 3)))
                        for v in b] for _ in range(M)]) + R
    np.testing.assert_allclose(out, expect, rtol=1e-14)


def test_chain_order_matters_and_alpha_zero():
    A = rng.standard_normal((3, 4))
    B = rng.standard_normal((4, 5))
    b = rng.standard_normal(5)
    d1 = O.run_chain(A, B, [("SCALE", 0, 2.0), ("BIAS", 0)], col_vecs={0: b})["D"]
    d2 = O.run_chain(A, B, [("BIAS", 0), ("SCALE", 0, 2.0)], col_vecs={0: b})["D"]
    np.testing.assert_allclose(d2 - d1, np.tile(b, (3, 1)), rtol=1e-12)
    d0 = O.run_chain(A, B, [("SCALE", 0, 0.0), ("GELU_TANH",)])["D"]
    np.testing.assert_array_equal(d0, 0.0)


def test_chain_swiglu_then_column_ops_use_half_width():
    A = rng.standard_normal((4, 8))
    B = rng.standard_normal((8, 10))
    b = rng.standard_normal(5)
    out = O.run_chain(A, B, [("SWIGLU",), ("BIAS", 0), ("ROW_SUM", 1)], col_vecs={0: b})
    C = A @ B
    h = C[:, :5] / (1 + np.exp(-C[:, :5])) * C[:, 5:] + b
    np.testing.assert_allclose(out["D"], h, rtol=1e-13)
    np.testing.assert_allclose(out["stats"][1], h.sum(axis=1), rtol=1e-13)


def test_chain_commuted_norm_reads_unscaled_weight():
    X = rng.standard_normal((6, 16))
    gamma = rng.uniform(0.5, 1.5, 16)
    W = rng.standard_normal((16, 8))
    out = O.run_chain(X, W, [("RMS_ROWSCALE", 2, 1e-6)], norm_gamma=gamma)
    r = 1.0 / np.sqrt((X * X).mean(axis=1) + 1e-6)
    np.testing.assert_allclose(out["stats"][2], r, rtol=1e-14)
    # against the commuted evaluation with gamma folded into W
    np.testing.assert_allclose(out["D"], r[:, None] * (X @ (gamma[:, None] * W)), rtol=1e-12)


def _brute_rmsnorm_project(X, gamma, W, eps, sumsq=None):
    """Normalise, then project, written out element by element: the textbook
    definition rmsnorm(X; gamma) @ W, with the mean of squares taken over the
    K entries of each row (or from the given row sums of squares)."""
    M, K = len(X), len(X[0])
    N = len(W[0])
    out = [[0.0] * N for _ in range(M)]
    for i in range(M):
        ss = sum(X[i][k] * X[i][k] for k in range(K)) if sumsq is None else sumsq[i]
        r = 1.0 / math.sqrt(ss / K + eps)
        xn = [X[i][k] * r * gamma[k] for k in range(K)]
        for j in range(N):
            out[i][j] = sum(xn[k] * W[k][j] for k in range(K))
    return np.array(out)


def test_chain_rms_rowscale_on_folded_weight_hand_values():
    # RMS_ROWSCALE without norm_gamma: the product is scaled by r_i taken from
    # A's own rows.  Row [3, 4] has mean square 12.5 and row [0, -2] mean square
    # 2, so with eps = 0 and B = I the outputs are x / sqrt(12.5) = x sqrt(2)/5
    # and x / sqrt(2).
    X = np.array([[3.0, 4.0], [0.0, -2.0]])
    out = O.run_chain(X, np.eye(2), [("RMS_ROWSCALE", 0, 0.0)])
    s2 = math.sqrt(2.0)
    np.testing.assert_allclose(out["D"], [[3 * s2 / 5, 4 * s2 / 5], [0.0, -s2]], rtol=1e-15, atol=0)
    np.testing.assert_allclose(out["stats"][0], [s2 / 5, 1 / s2], rtol=1e-15)


def test_chain_rms_rowscale_on_folded_weight_brute_force():
    # the folded weight gamma (.)_row W with RMS_ROWSCALE gives the textbook
    # normalise-then-project result, element by element
    X = rng.standard_normal((5, 12))
    gamma = rng.uniform(0.5, 1.5, 12)
    W = rng.standard_normal((12, 7))
    out = O.run_chain(X, gamma[:, None] * W, [("RMS_ROWSCALE", None, 1e-6)])
    ref = _brute_rmsnorm_project(X.tolist(), gamma.tolist(), W.tolist(), 1e-6)
    np.testing.assert_allclose(out["D"], ref, rtol=1e-12, atol=1e-12)


def test_chain_rms_from_sumsq_hand_values_and_brute_force():
    # RMS_SUMSQ_ROWSCALE: the same row factor from given sums of squares.  With
    # the rows' own sums (25 and 4 for the hand rows above) it reproduces the
    # hand values; with norm_gamma it is normalise-then-project; with other sums
    # it follows them (s = 2 K: r = 1/sqrt(2 + eps))
    X = np.array([[3.0, 4.0], [0.0, -2.0]])
    out = O.run_chain(X, np.eye(2), [("RMS_SUMSQ_ROWSCALE", 0, 0.0)], row_vecs={0: np.array([25.0, 4.0])})
    s2 = math.sqrt(2.0)
    np.testing.assert_allclose(out["D"], [[3 * s2 / 5, 4 * s2 / 5], [0.0, -s2]], rtol=1e-15, atol=0)
    out = O.run_chain(X, np.eye(2), [("RMS_SUMSQ_ROWSCALE", 0, 0.0)], row_vecs={0: np.array([4.0, 4.0])})
    np.testing.assert_allclose(out["D"], X / s2, rtol=1e-15, atol=0)
    Xr = rng.standard_normal((4, 10))
    gamma = rng.uniform(0.5, 1.5, 10)
    W = rng.standard_normal((10, 6))
    ss = [sum(v * v for v in row) for row in Xr.tolist()]
    ref = _brute_rmsnorm_project(Xr.tolist(), gamma.tolist(), W.tolist(), 1e-6, sumsq=ss)
    folded = O.run_chain(Xr, gamma[:, None] * W, [("RMS_SUMSQ_ROWSCALE", 1, 1e-6)], row_vecs={1: np.array(ss)})
    np.testing.assert_allclose(folded["D"], ref, rtol=1e-12, atol=1e-12)
    unfused = O.run_chain(Xr, W, [("RMS_SUMSQ_ROWSCALE", 1, 1e-6)], row_vecs={1: np.array(ss)}, norm_gamma=gamma)
    np.testing.assert_allclose(unfused["D"], ref, rtol=1e-12, atol=1e-12)


def test_chain_dgrad_form():
    dY = rng.standard_normal((5, 7))
    W = rng.standard_normal((9, 7))     # [N, K]
    Z = rng.standard_normal((5, 9))
    Xh = rng.standard_normal((5, 9))
    out = O.run_chain(dY, W, [("GELU_TANH_GRAD",), ("ROW_DOT_AUX", 0), ("ROW_SUM", 1)],
                      b_layout="nk", z=Z, xhat=Xh)
    h = 1e-6
    gp = (O.gelu_tanh(Z + h) - O.gelu_tanh(Z - h)) / (2 * h)
    dX = _brute_gemm(dY.tolist(), W.T.tolist(), "kn") * gp
    np.testing.assert_allclose(out["D"], dX, rtol=1e-7, atol=1e-8)
    np.testing.assert_allclose(out["stats"][0], (dX * Xh).sum(axis=1), rtol=1e-7, atol=1e-7)
    np.testing.assert_allclose(out["stats"][1], dX.sum(axis=1), rtol=1e-7, atol=1e-7)


def test_chain_col_row_scale_and_preact_closed_form():
    # A = I, B = ones makes C = ones, so COL_SCALE then ROW_SCALE gives u_i * v_j,
    # and the stored pre-activation is that product before the GELU
    n = 6
    v = rng.standard_normal(n)
    u = rng.standard_normal(n)
    out = O.run_chain(np.eye(n), np.ones((n, n)),
                      [("COL_SCALE", 1), ("ROW_SCALE", 0), ("STORE_PREACT",), ("SILU",)],
                      col_vecs={1: v}, row_vecs={0: u})
    np.testing.assert_allclose(out["preact"], np.outer(u, v), rtol=1e-15)
    np.testing.assert_allclose(out["D"], O.silu(np.outer(u, v)), rtol=1e-15)


def test_round_bf16_against_bit_patterns():
    import torch
    # bf16 keeps the top 16 bits of an fp32 word; values already on the bf16
    # grid are unchanged, midpoints go to the even neighbour
    assert O.round_bf16(1.0) == 1.0
    assert O.round_bf16(1.0 + 2 ** -8) == 1.0                  # midpoint, even below
    assert O.round_bf16(1.0 + 3 * 2 ** -8) == 1.0 + 2 ** -6    # midpoint, even above
    assert O.round_bf16(1.0 + 2 ** -8 + 2 ** -20) == 1.0 + 2 ** -7
    assert O.round_bf16(-3.0) == -3.0
    # fp32 inputs: a single rounding, so torch's fp32 -> bf16 conversion agrees exactly
    x = np.random.default_rng(7).standard_normal(20000).astype(np.float32)
    expect = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_bf16(x.astype(np.float64)), expect)


def test_dropout_threshold_float32_parameter():
    # op-list parameters are float32: p = float32(0.1) widens exactly to fp64,
    # 1 - p is exact in fp64, and the threshold is floor((1 - p) * 2^64)
    from fractions import Fraction
    p32 = float(np.float32(0.1))
    assert O.dropout_threshold(p32) == int((1 - Fraction(p32)) * 2 ** 64)
    assert O.dropout_threshold(p32) != O.dropout_threshold(0.1)
    assert O.dropout_threshold(1e-30) is None          # (1-p) * 2^64 rounds to 2^64: keep all
    out = O.run_chain(np.eye(3), np.ones((3, 3)), [("DROPOUT", 0, 0.1)], seed=1)
    keep = O.dropout_mask(1, 3, 3, p32)
    np.testing.assert_array_equal(out["keep"], keep)


def test_gelu_erf_textbook_values():
    # x * Phi(x) at points where the standard normal distribution function has
    # well-known values: Phi(1) = 0.8413447460685429, Phi(2) = 0.9772498680518208
    assert O.gelu_erf(0.0) == 0.0
    assert abs(O.gelu_erf(1.0) - 0.8413447460685429) < 1e-15
    assert abs(O.gelu_erf(-1.0) + (1 - 0.8413447460685429)) < 1e-15
    assert abs(O.gelu_erf(2.0) - 2 * 0.9772498680518208) < 1e-15
    x = np.linspace(-6, 6, 601)
    np.testing.assert_allclose(O.gelu_erf(x) - O.gelu_erf(-x), x, atol=1e-14)   # erf is odd
    # and the tanh approximation stays within its known 5e-4 of it
    assert np.abs(O.gelu_erf(x) - O.gelu_tanh(x)).max() < 5e-4


def test_gelu_erf_grad():
    z = np.linspace(-7, 7, 1401)
    h = 1e-5
    fd = (O.gelu_erf(z + h) - O.gelu_erf(z - h)) / (2 * h)
    np.testing.assert_allclose(O.gelu_erf_grad(z), fd, atol=1e-9)
    assert O.gelu_erf_grad(0.0) == 0.5
    # phi(1) = 0.24197072451914337: Phi(1) + phi(1)
    assert abs(O.gelu_erf_grad(1.0) - (0.8413447460685429 + 0.24197072451914337)) < 1e-15


def test_layernorm_hand_values_and_constant_row():
    X = np.array([[1.0, 2.0, 3.0, 4.0]])          # mean 2.5, biased variance 1.25
    mu, r = O.ln_stats(X, 0.0)
    assert mu[0] == 2.5 and abs(r[0] - 1.0 / math.sqrt(1.25)) < 1e-15
    np.testing.assert_allclose(O.layernorm(X, np.ones(4), None, 0.0)[0],
                               (np.array([1, 2, 3, 4]) - 2.5) / math.sqrt(1.25), rtol=1e-14)
    # a constant row normalises to beta
    K = 32
    g = rng.uniform(0.5, 1.5, K)
    b = rng.standard_normal(K)
    np.testing.assert_allclose(O.layernorm(np.full((1, K), 7.0), g, b, 1e-5)[0], b, rtol=1e-14, atol=1e-14)


def test_commuted_layernorm_identity():
    # layernorm(X) @ W == r (.)_row (X @ W' - mu (x) colsum(W')) + beta^T W, W' = gamma (.)_row W
    X = rng.standard_normal((30, 48)) + 0.7
    g = rng.uniform(0.5, 1.5, 48)
    b = rng.standard_normal(48)
    W = rng.standard_normal((48, 20))
    eps = float(np.float32(1e-5))           # the op list carries eps as float32
    lhs = O.layernorm_project(X, g, b, W, eps)
    Wf = g[:, None] * W
    mu, r = O.ln_stats(X, eps)
    rhs = r[:, None] * (X @ Wf - mu[:, None] * Wf.sum(axis=0)[None, :]) + (b @ W)[None, :]
    np.testing.assert_allclose(lhs, rhs, rtol=1e-11, atol=1e-11)
    # and the chain's written-out form of LN_ROWSCALE gives the same
    out = O.run_chain(X, Wf, [("LN_ROWSCALE", 0, 1e-5)], ln_colsum=Wf.sum(axis=0), ln_bias=b @ W)
    np.testing.assert_allclose(out["D"], lhs, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(out["stats"][0], r, rtol=1e-14)
    np.testing.assert_allclose(out["stats"][1], mu, rtol=1e-14)


def test_column_reductions_transpose_identity():
    # column sums of A @ B are the row sums of (A @ B)^T = B^T @ A^T, which the
    # oracle computes through its row-reduction path
    A = rng.standard_normal((37, 20))
    B = rng.standard_normal((20, 11))
    Xh = rng.standard_normal((37, 11))
    cols = O.run_chain(A, B, [("COL_SUM", 0), ("COL_SUMSQ", 1), ("COL_DOT_AUX", 2)], xhat=Xh)
    rows = O.run_chain(B.T, A.T, [("ROW_SUM", 0), ("ROW_SUMSQ", 1), ("ROW_DOT_AUX", 2)], xhat=Xh.T)
    for s in range(3):
        np.testing.assert_allclose(cols["col_stats"][s], rows["stats"][s], rtol=1e-12, atol=1e-12)
    # both orders total the same
    rs = O.run_chain(A, B, [("ROW_SUM", 0)])["stats"][0]
    assert abs(rs.sum() - cols["col_stats"][0].sum()) < 1e-9


def test_column_reductions_closed_forms():
    M, N = 13, 6
    # D = 1 everywhere (A one-hot column of ones, B a row of ones): sum = M, sumsq = M
    A = np.ones((M, 1))
    B = np.ones((1, N))
    out = O.run_chain(A, B, [("COL_SUM", 0), ("COL_SUMSQ", 1), ("COL_DOT_AUX", 2)], xhat=np.full((M, N), 2.0))
    np.testing.assert_array_equal(out["col_stats"][0], np.full(N, M))
    np.testing.assert_array_equal(out["col_stats"][1], np.full(N, M))
    np.testing.assert_array_equal(out["col_stats"][2], np.full(N, 2 * M))
    # reductions see the chain value at their position: after SCALE 3 the sum triples
    out = O.run_chain(A, B, [("COL_SUM", 0), ("SCALE", 0, 3.0), ("COL_SUM", 1)])
    np.testing.assert_array_equal(out["col_stats"][1], 3 * out["col_stats"][0])


def _fd_grad(f, X, h=1e-6):
    """Central differences of a scalar function of X, element by element."""
    G = np.zeros_like(X)
    for idx in np.ndindex(X.shape):
        Xp = X.copy()
        Xm = X.copy()
        Xp[idx] += h
        Xm[idx] -= h
        G[idx] = (f(Xp) - f(Xm)) / (2 * h)
    return G


def test_rmsnorm_backward_matches_finite_differences():
    X = rng.standard_normal((4, 9))
    g = rng.uniform(0.5, 1.5, 9)
    dY = rng.standard_normal((4, 9))
    dX, dg = O.rmsnorm_backward(X, g, dY, 1e-6)
    np.testing.assert_allclose(dX, _fd_grad(lambda Z: np.sum(O.rmsnorm(Z, g, 1e-6) * dY), X), atol=1e-7)
    np.testing.assert_allclose(dg, _fd_grad(lambda gg: np.sum(O.rmsnorm(X, gg, 1e-6) * dY), g), atol=1e-7)


def test_layernorm_backward_matches_finite_differences():
    X = rng.standard_normal((4, 9)) + 1.5
    g = rng.uniform(0.5, 1.5, 9)
    b = rng.standard_normal(9)
    dY = rng.standard_normal((4, 9))
    dX, dg, db = O.layernorm_backward(X, g, dY, 1e-5)
    np.testing.assert_allclose(dX, _fd_grad(lambda Z: np.sum(O.layernorm(Z, g, b, 1e-5) * dY), X), atol=1e-7)
    np.testing.assert_allclose(dg, _fd_grad(lambda gg: np.sum(O.layernorm(X, gg, b, 1e-5) * dY), g), atol=1e-7)
    np.testing.assert_allclose(db, _fd_grad(lambda bb: np.sum(O.layernorm(X, g, bb, 1e-5) * dY), b), atol=1e-7)
    # a row's dX sums to zero (the mean is removed); with eps = 0 it is also
    # orthogonal to x_hat (layernorm is then invariant to scaling a row)
    np.testing.assert_allclose(dX.sum(axis=1), 0, atol=1e-12)
    dX0, _, _ = O.layernorm_backward(X, g, dY, 0.0)
    mu, r = O.ln_stats(X, 0.0)
    xh = (X - mu[:, None]) * r[:, None]
    np.testing.assert_allclose((dX0 * xh).sum(axis=1), 0, atol=1e-10)


def test_norm_backward_chain_through_the_op_list():
    # the dgrad epilogue's reductions, evaluated by run_chain on G = dY @ W^T,
    # give layernorm_backward's dbeta and dgamma, and the correction formula
    # applied to its row sums gives dX
    M, K, N = 6, 10, 7
    X = rng.standard_normal((M, K)) + 0.5
    g = rng.uniform(0.5, 1.5, K)
    W = rng.standard_normal((K, N))
    dY = rng.standard_normal((M, N))
    mu, r = O.ln_stats(X, 1e-5)
    ops = [("COL_SUM", 1), ("COL_DOT_NORM", 0), ("COL_SCALE", 0), ("ROW_SUM", 0), ("ROW_DOT_AUX", 1)]
    out = O.run_chain(dY, W, ops, b_layout="nk", col_vecs={0: g}, row_vecs={0: r, 1: mu}, xhat=X)
    dX_ref, dg_ref, db_ref = O.layernorm_backward(X, g, dY @ W.T, 1e-5)
    np.testing.assert_allclose(out["col_stats"][1], db_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["col_stats"][0], dg_ref, rtol=1e-12, atol=1e-12)
    G = out["D"]
    s1, sgx = out["stats"][0], out["stats"][1]
    xh = (X - mu[:, None]) * r[:, None]
    S = r * (sgx - mu * s1)
    dX = r[:, None] * (G - s1[:, None] / K - xh * S[:, None] / K)
    np.testing.assert_allclose(dX, dX_ref, rtol=1e-10, atol=1e-12)


def test_e4m3_decode_known_values():
    # format facts: 1.0 = 0.0111.000, 448 = 0.1111.110 (largest finite), 2^-6 =
    # 0.0001.000 (smallest normal), 2^-9 = 0.0000.001 (smallest subnormal)
    assert O.e4m3_decode(0x38) == 1.0
    assert O.e4m3_decode(0x7E) == 448.0
    assert O.e4m3_decode(0x08) == 2.0 ** -6
    assert O.e4m3_decode(0x01) == 2.0 ** -9
    assert O.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert O.e4m3_decode(0xB8) == -1.0
    assert O.e4m3_decode(0x40) == 2.0 and O.e4m3_decode(0x3C) == 1.5
    assert np.isnan(O.e4m3_decode(0x7F)) and np.isnan(O.e4m3_decode(0xFF))
    assert O.e4m3_decode(0x80) == 0.0 and np.signbit(O.e4m3_decode(0x80))
    # consecutive positive codes increase
    v = O.e4m3_decode(np.arange(0x7F))
    assert (np.diff(v) > 0).all()


def test_e4m3_encode_roundtrip_ties_and_saturation():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    np.testing.assert_array_equal(O.e4m3_encode(O.e4m3_decode(codes)), codes)
    # midpoints between neighbours go to the even code
    for c in range(0x00, 0x7E):
        mid = (O.e4m3_decode(c) + O.e4m3_decode(c + 1)) / 2
        want = c if c % 2 == 0 else c + 1
        assert O.e4m3_encode(mid) == want, hex(c)
        assert O.e4m3_encode(-mid) == want | 0x80
    # just off a midpoint goes to the nearer value
    assert O.e4m3_encode(1.0625 + 1e-9) == 0x39 and O.e4m3_encode(1.0625 - 1e-9) == 0x38
    # saturation and the special values
    assert O.e4m3_encode(448.0) == 0x7E and O.e4m3_encode(464.0) == 0x7E and O.e4m3_encode(1e30) == 0x7E
    assert O.e4m3_encode(-1e30) == 0xFE
    assert O.e4m3_encode(float("nan")) == 0x7F
    assert O.e4m3_encode(2.0 ** -11) == 0x00 and O.e4m3_encode(-(2.0 ** -11)) == 0x80


def test_quantize_rows_e4m3():
    X = np.array([[0.0, 1.0, -2.0, 4.0], [0.0, 0.0, 0.0, 0.0], [3.0, -3.0, 1.5, 0.75]], dtype=np.float32)
    q, s = O.quantize_rows_e4m3(X)
    # row 0: amax 4 -> scale 4/448, x*112 = 0, 112, -224, 448
    assert s[0] == np.float32(4.0) / np.float32(448.0)
    np.testing.assert_array_equal(q[0], O.e4m3_encode([0.0, 112.0, -224.0, 448.0]))
    np.testing.assert_array_equal(q[1], [0, 0, 0, 0]) and s[1] == 0
    # the row's largest magnitude maps to 448 exactly, and decode * scale recovers x within 2^-4 relative
    rng_ = np.random.default_rng(3)
    Y = rng_.standard_normal((8, 64)).astype(np.float32)
    q, s = O.quantize_rows_e4m3(Y)
    assert (np.abs(O.e4m3_decode(q)).max(axis=1) == 448.0).all()
    back = O.e4m3_decode(q) * s[:, None]
    assert (np.abs(back - Y) <= 2.0 ** -4 * np.abs(Y) + 2.0 ** -9 * s[:, None] * 8).all()


# ------------------------------------------------------------ MX E4M3 -------
# OCP Microscaling Formats (MX) v1.0: E8M0 scale X = 2^(e-127) shared by 32
# E4M3 elements; conversion takes the shared exponent floor(log2 amax) - 8.
def test_e8m0_decode_known_values():
    assert O.e8m0_decode(127) == 1.0
    assert O.e8m0_decode(130) == 8.0
    assert O.e8m0_decode(0) == 2.0 ** -127
    assert O.e8m0_decode(254) == 2.0 ** 127
    assert np.isnan(O.e8m0_decode(255))


def test_mx_quantize_hand_values():
    V = np.zeros((6, 32))
    V[0, :4] = [1.0, 0.5, -0.25, 0.125]          # amax 1: X = 2^-8, P = 256 V
    V[1, :3] = [448.0, 1.0, -2.0]                 # amax 448: X = 1
    V[2, :2] = [500.0, 3.0]                       # amax 500: X = 1, 500 saturates to 448
    V[3, :] = 0.0                                 # zero block: byte 0, zero codes
    V[4, 0] = 1.5 * 2.0 ** 127                    # X = 2^119, P = 384
    V[5, 0] = 3.0 * 2.0 ** -140                   # scale clamped to 2^-127; P = 3 2^-13 rounds to 0
    codes, sexp = O.quantize_mx_e4m3(V)
    assert list(sexp[:, 0]) == [119, 127, 127, 0, 246, 0]
    assert list(codes[0, :5]) == [0x78, 0x70, 0xE8, 0x60, 0x00]   # 256, 128, -64, 32, 0
    assert list(codes[1, :3]) == [0x7E, 0x38, 0xC0]              # 448, 1, -2
    assert list(codes[2, :2]) == [0x7E, 0x44]                    # 448 (saturated), 3 = 1.5 * 2^1
    assert not codes[3].any()
    assert codes[4, 0] == 0x7C                                   # 384 = 1.5 * 2^8
    assert codes[5, 0] == 0x00


def test_mx_roundtrip_error_bound_and_ragged_block():
    # elements whose scaled value lies in E4M3's normal range and below 448 are
    # within half an E4M3 ulp (2^-4 relative); the last block of a row may be short
    rng2 = np.random.default_rng(7)
    V = rng2.standard_normal((8, 70)) * np.exp2(rng2.integers(-20, 20, (8, 1)))
    codes, sexp = O.quantize_mx_e4m3(V)
    assert sexp.shape == (8, 3)
    back = O.dequantize_mx(codes, sexp)
    X = np.repeat(O.e8m0_decode(sexp), 32, axis=1)[:, :70]
    P = np.abs(V) / X
    ok = (P >= 2.0 ** -6) & (P <= 448.0)
    assert ok.mean() > 0.9
    assert (np.abs(back - V)[ok] <= 2.0 ** -4 * np.abs(V)[ok] * (1 + 1e-12)).all()
    # the block maximum's exponent sets X: amax / X in [256, 512)
    amax = np.maximum.reduceat(np.abs(V), [0, 32, 64], axis=1)
    assert ((amax / O.e8m0_decode(sexp) >= 256) & (amax / O.e8m0_decode(sexp) < 512)).all()


def test_mx_dequantized_gemm_closed_form():
    # A's row: 32 ones at scale 1, then 32 ones at scale 2 (byte 128); B all ones at
    # scale 1: every output is 32 * 1 + 32 * 2 = 96; an off-by-one block index
    # would give 64 or 128
    codes_a = np.full((2, 64), 0x38, dtype=np.uint8)
    sexp_a = np.array([[127, 128], [128, 127]], dtype=np.uint8)
    codes_b = np.full((3, 64), 0x38, dtype=np.uint8)
    sexp_b = np.full((3, 2), 127, dtype=np.uint8)
    A = O.dequantize_mx(codes_a, sexp_a)
    B = O.dequantize_mx(codes_b, sexp_b)
    np.testing.assert_array_equal(O.gemm(A, B, "nk"), np.full((2, 3), 96.0))


def test_mx_scale_tiled_offsets():
    # K = 160: 5 blocks of 32 per row, 2 groups of 4 blocks
    assert O.mx_scale_offset(0, 0, 160) == 0
    assert O.mx_scale_offset(0, 1, 160) == 1
    assert O.mx_scale_offset(1, 0, 160) == 16
    assert O.mx_scale_offset(32, 0, 160) == 4
    assert O.mx_scale_offset(127, 3, 160) == 31 * 16 + 3 * 4 + 3
    assert O.mx_scale_offset(0, 4, 160) == 512
    assert O.mx_scale_offset(128, 0, 160) == 2 * 512
    assert O.mx_scale_bytes(130, 160) == 2 * 2 * 512
    # every (row, block) of a 200 x 5 matrix has its own byte
    offs = {O.mx_scale_offset(r, j, 160) for r in range(200) for j in range(5)}
    assert len(offs) == 1000 and max(offs) < O.mx_scale_bytes(200, 160)
