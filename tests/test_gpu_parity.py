"""GPU parity: the CUDA library (through the C ABI) against the fp64 oracle.

Tolerance (bf16 inputs, fp32 accumulation, bf16 output):
    |gpu - ref| <= 1e-2 + 1e-2 |ref| elementwise, and
    ||gpu - ref||_F / ||ref||_F <= 5e-3.
Integer results (dropout mask, keep counts) and exact-arithmetic cases
(small-integer GEMMs whose sums are exact in fp32 and bf16) are bit-exact.
Full-size workloads are compared on sampled rows (first, last, tile edges and
random rows), which the oracle evaluates row by row.
"""
import math

import numpy as np
import pytest
import torch

import __graft_entry__ as entry
from gemm_epilogue_transformer_tmem_gb300 import coda, inputs
from oracle import coda_oracle as O

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2
FRO = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    entry.build()
    coda.lib()
    yield
    st, info = coda.check_device_error()
    assert st == 0, f"device error word set: {info}"


@pytest.fixture(params=["single", "pair", "split", "persist4"])
def mode(request):
    """Run a test on the single-CTA kernel (128-row tiles), on the CTA-pair
    kernel (tcgen05 cta_group::2, 256-row tiles), on the single-CTA kernel with
    K split over CTAs (stream-K; every problem with two k-blocks or more), and
    on a single-CTA grid capped at 4 CTAs: each CTA then loops over several
    tiles, and the commuted norms take their row statistics from the A stages
    in shared memory (the side path used when tiles fill the grid)."""
    m = request.param
    coda.set_cta_pair("pair" if m == "pair" else "single")
    coda.set_split_k({"single": "off", "pair": "auto", "split": "force", "persist4": "off"}[m])
    coda.set_max_ctas(4 if m == "persist4" else 0)
    yield m
    coda.set_cta_pair("auto")
    coda.set_split_k("auto")
    coda.set_max_ctas(0)


def cu(t):
    return t.to("cuda")


def f64(t):
    return O.to_f64(t)


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance, worst at {i}: "
                             f"gpu {got[i]!r} ref {ref[i]!r}")
    nref = np.linalg.norm(ref)
    if nref > 0:
        fro = np.linalg.norm(got - ref) / nref
        assert fro <= FRO, f"{what}: relative Frobenius error {fro:.3e}"


# Row and column statistics are fp32 sums of fp32 chain values (never of the
# bf16 outputs), so their error is not the output tolerance above.  Each
# summand carries the relative error tau of the chain value it is taken from:
#   TAU_LIN   GEMM and linear ops in fp32: accumulation over K (about
#             sqrt(K) 2^-24 relative) and a few ulps per op; 2^-16 covers K up to 2^14
#   TAU_ACT   an activation on the way: SiLU and the tanh-form GELU use the
#             hardware tanh (logistic absolute error <= 2^-12, i.e. <= 2^-12 |x|
#             on f(x), which stays below 2^-10 |f(x)| wherever f(x) is not near 0)
#   TAU_FOLD  the bf16 gamma fold on the way: 2^-9 relative per weight
# Independent errors add in quadrature, so the sum moves by tau * scale, scale
# being the oracle's error scale (the L2 norm of d(summand)/d(log x)); the
# fp32 rounding of the sum adds 2^-24 sqrt(n) * scale the same way.  The bound
# allows 6 standard deviations of both.  On top of that the tensor cores'
# fp32 accumulation is biased towards zero (measured: sums of squares of a
# K = 16384 GEMM output 3.2e-5 low on every row), about one ulp per MMA step
# of 16 elements of K: a relative bias b = (K/16) 2^-24 in every chain value,
# which moves a reduction by up to 2 b |ref| (sums of squares) and does not
# average out.  A summand left out of the sum moves it by |s_j|, which is far
# above all this on every full-size workload; the exact integer reductions
# (test_reductions_exact) catch a missing summand of any size.
TAU_LIN = 2.0 ** -16
TAU_ACT = 2.0 ** -10
TAU_FOLD = 2.0 ** -9
ACTIVATIONS = {"GELU_TANH", "SILU", "SWIGLU", "GELU_TANH_GRAD", "GELU_ERF", "GELU_ERF_GRAD"}


def chain_tau(ops, fold=False):
    """Relative error budget of the chain values an op list reduces."""
    tau = TAU_ACT if any(o[0] in ACTIVATIONS for o in ops) else TAU_LIN
    return max(tau, TAU_FOLD) if fold else tau


def stat_bound(ref, scale, n, tau, K):
    """Bound on |gpu - ref| of a reduction over n summands of a GEMM with reduction depth K."""
    ref = np.abs(np.asarray(ref, dtype=np.float64))
    bias = 2.0 * (max(K, 16) / 16.0) * 2.0 ** -24
    return 1e-6 + (2.0 ** -20 + bias) * ref + 6.0 * (tau + 2.0 ** -24 * math.sqrt(max(n, 1))) * np.asarray(scale)


def assert_stat_close(got, ref, scale, n, tau, K, what=""):
    """Row reductions over n columns of a GEMM with reduction depth K (see stat_bound)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bound = stat_bound(ref, scale, n, tau, K)
    err = np.abs(got - ref)
    if (err > bound).any():
        i = int(np.argmax(err - bound))
        raise AssertionError(f"{what}: {(err > bound).sum()} rows out of tolerance, worst row {i}: "
                             f"gpu {got[i]!r} ref {ref[i]!r} bound {bound[i]!r}")


def check_stats(r, ref, what, tau, K):
    n = ref["D"].shape[1] if "D" in ref else 1
    for slot, v in ref["stats"].items():
        if slot in ref["stat_scale"]:
            assert_stat_close(f64(r.row_stats[slot]), v, ref["stat_scale"][slot], n, tau, K, f"{what} stat {slot}")
        else:
            assert_close(f64(r.row_stats[slot]), v, f"{what} stat {slot}")


def sync_ok():
    torch.cuda.synchronize()
    st, info = coda.check_device_error()
    assert st == 0, f"device error {st}: {info}"


def rand(shape, seed, std=1.0):
    return inputs.randn_bf16(shape, std, seed)


# --------------------------------------------------------------- plain GEMM
@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_small_integer_gemm_bit_exact(layout, mode):
    # |values| <= 2 and K = 64: every partial sum is an integer below 2^8, so
    # fp32 accumulation and the bf16 store are exact
    M, K, N = 200, 64, 264
    A = inputs.small_int_bf16((M, K), 2, 1)
    B = inputs.small_int_bf16((K, N) if layout == "kn" else (N, K), 2, 2)
    r = coda.gemm_epilogue(cu(A), cu(B), [], b_layout=layout)
    sync_ok()
    ref = O.gemm(f64(A), f64(B), layout)
    np.testing.assert_array_equal(f64(r.D), ref)


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("M,K,N", [(128, 64, 256), (1, 8, 8), (300, 200, 264), (257, 1000, 520),
                                   (129, 4096, 264), (640, 136, 1032)])
def test_plain_gemm(layout, M, K, N, mode):
    A = rand((M, K), 10 + M)
    B = rand((K, N) if layout == "kn" else (N, K), 20 + N, 1.0 / math.sqrt(K))
    r = coda.gemm_epilogue(cu(A), cu(B), [], b_layout=layout)
    sync_ok()
    assert_close(f64(r.D), O.gemm(f64(A), f64(B), layout), f"gemm {layout} {M}x{K}x{N}")


def test_k_zero_is_empty_sum():
    M, N = 70, 40
    b = rand((N,), 5)
    ops = [("BIAS", 0), ("GELU_TANH",)]
    A = torch.empty((M, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((0, N), dtype=torch.bfloat16, device="cuda")
    r = coda.gemm_epilogue(A, B, ops, col_vecs={0: cu(b)})
    sync_ok()
    ref = O.run_chain(np.zeros((M, 0)), np.zeros((0, N)), ops, col_vecs={0: f64(b)})["D"]
    assert_close(f64(r.D), ref, "K = 0")


def test_pr1_bias_gelu_residual(mode):
    t = inputs.make_pr1(seed=0)
    ops = [("BIAS", 0), ("GELU_TANH",), ("RESIDUAL", 0, 1.0)]
    r = coda.gemm_epilogue(cu(t["X"]), cu(t["W"]), ops, col_vecs={0: cu(t["bias"])}, residual=cu(t["residual"]))
    sync_ok()
    ref = O.run_chain(f64(t["X"]), f64(t["W"]), ops, col_vecs={0: f64(t["bias"])}, residual_t=f64(t["residual"]))
    assert_close(f64(r.D), ref["D"], "pr1")


# ------------------------------------------------------------ each op alone
M_R, K_R, N_R = 300, 192, 264     # ragged in M (not /128), N (not /256, not /32) and K (not /64)

OP_CASES = {
    "scale": [("SCALE", 0, 0.5)],
    "col_scale": [("COL_SCALE", 1)],
    "bias": [("BIAS", 0)],
    "row_scale": [("ROW_SCALE", 0)],
    "gelu": [("GELU_TANH",)],
    "silu": [("SILU",)],
    "gelu_grad": [("GELU_TANH_GRAD",)],
    "gelu_erf": [("GELU_ERF",)],
    "gelu_erf_grad": [("GELU_ERF_GRAD",)],
    "bias_gelu_erf_swiglu": [("BIAS", 0), ("GELU_ERF",), ("SWIGLU",)],
    "residual": [("RESIDUAL", 0, 0.75)],
    "preact_gelu": [("STORE_PREACT",), ("GELU_TANH",)],
    "reductions": [("ROW_SUM", 0), ("ROW_MEAN", 1), ("ROW_SUMSQ", 2), ("ROW_DOT_AUX", 3)],
    "swiglu": [("SWIGLU",)],
    "bias_swiglu_bias_sum": [("BIAS", 0), ("SWIGLU",), ("BIAS", 1), ("ROW_SUM", 0)],
    "scale_preact_swiglu": [("SCALE", 0, 2.0), ("STORE_PREACT",), ("SWIGLU",), ("ROW_SUMSQ", 1)],
    "chain": [("SCALE", 0, 1.5), ("BIAS", 0), ("GELU_TANH",), ("COL_SCALE", 1), ("RESIDUAL", 0, 1.0),
              ("ROW_MEAN", 2)],
    "none": [],
    "bias_gelu_residual": [("BIAS", 0), ("GELU_TANH",), ("RESIDUAL", 0, 1.0)],
    "dgrad": [("GELU_TANH_GRAD",), ("ROW_DOT_AUX", 0), ("ROW_SUM", 1)],
    "bias_gelu": [("BIAS", 0), ("GELU_TANH",)],
    "bias_gelu_erf": [("BIAS", 0), ("GELU_ERF",)],
    "bias_residual": [("BIAS", 0), ("RESIDUAL", 0, 1.0)],
    "wgrad": [("SCALE", 0, 0.5), ("RESIDUAL", 0, 1.0), ("ROW_SUMSQ", 0)],
}

# op lists the library runs as fixed op sequences (straight-line epilogues);
# every other list runs the interpreter
FIXED_SEQUENCE_CASES = ["none", "residual", "bias_gelu_residual", "dgrad", "swiglu", "bias", "bias_gelu",
                        "bias_gelu_erf", "bias_residual", "gelu", "wgrad"]


def _op_case_tensors(ops, layout, seed):
    glu = any(o[0] == "SWIGLU" for o in ops)
    N = 2 * N_R if glu else N_R
    n_out = N // 2 if glu else N
    A = rand((M_R, K_R), seed)
    B = rand((K_R, N) if layout == "kn" else (N, K_R), seed + 1, 1.0 / math.sqrt(K_R))
    # column vectors: before SWIGLU they span N columns, after it N/2
    pos = [i for i, o in enumerate(ops) if o[0] == "SWIGLU"]
    gpos = pos[0] if pos else len(ops)
    widths = {}
    for i, o in enumerate(ops):
        if o[0] in ("COL_SCALE", "BIAS"):
            widths[o[1]] = N if i < gpos else n_out
    col = {s: rand((w,), seed + 10 + s) for s, w in widths.items()}
    row = {0: torch.rand((M_R,), generator=torch.Generator().manual_seed(seed + 20)) + 0.5}
    aux = dict(residual=rand((M_R, n_out), seed + 30), z=rand((M_R, n_out), seed + 31),
               xhat=rand((M_R, n_out), seed + 32))
    return A, B, N, n_out, col, row, aux


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("case", sorted(OP_CASES))
def test_op(case, layout, mode):
    ops = OP_CASES[case]
    A, B, N, n_out, col, row, aux = _op_case_tensors(ops, layout, 100 + len(case))
    preact = None
    if any(o[0] == "STORE_PREACT" for o in ops):
        i = [o[0] for o in ops].index("STORE_PREACT")
        g = [o[0] for o in ops].index("SWIGLU") if any(o[0] == "SWIGLU" for o in ops) else len(ops)
        preact = torch.full((M_R, N if i < g else n_out), float("nan"), dtype=torch.bfloat16, device="cuda")
    r = coda.gemm_epilogue(cu(A), cu(B), ops, b_layout=layout, col_vecs={k: cu(v) for k, v in col.items()},
                           row_vecs={0: cu(row[0])}, residual=cu(aux["residual"]), z=cu(aux["z"]),
                           xhat=cu(aux["xhat"]), preact_out=preact)
    sync_ok()
    ref = O.run_chain(f64(A), f64(B), ops, b_layout=layout, col_vecs={k: f64(v) for k, v in col.items()},
                      row_vecs={0: f64(row[0])}, residual_t=f64(aux["residual"]), z=f64(aux["z"]),
                      xhat=f64(aux["xhat"]))
    assert_close(f64(r.D), ref["D"], case)
    check_stats(r, ref, case, chain_tau(ops), K_R)
    if preact is not None:
        assert_close(f64(preact), ref["preact"], f"{case} preact")


def _random_op_list(rng, glu):
    """A valid op list drawn at random: ops before SWIGLU act on the N-wide
    accumulator, ops after it on the N/2-wide output; reductions last."""
    pre_pool = [("SCALE", 0, 1.25), ("BIAS", 0), ("COL_SCALE", 1), ("ROW_SCALE", 0), ("GELU_TANH",), ("SILU",),
                ("GELU_ERF",)]
    post_pool = [("BIAS", 2), ("RESIDUAL", 0, 0.5), ("GELU_TANH",), ("SCALE", 0, 0.75), ("GELU_TANH_GRAD",)]
    red_pool = [("ROW_SUM", 0), ("ROW_SUMSQ", 1), ("ROW_DOT_AUX", 2)]
    pick = lambda pool, n: [pool[i] for i in sorted(rng.choice(len(pool), size=n, replace=False))]  # noqa: E731
    ops = pick(pre_pool, int(rng.integers(0, 4)))
    if glu:
        ops.append(("SWIGLU",))
    ops += pick(post_pool, int(rng.integers(0, 3)))
    ops += pick(red_pool, int(rng.integers(0, 3)))
    return ops


@pytest.mark.parametrize("seed", range(96))
def test_random_op_lists(seed):
    # Random sizes (ragged in every dimension, 1 to 700 rows), layouts, kernels
    # (single CTA, CTA pair, split over K) and op lists, against the oracle.
    rng = np.random.default_rng(5000 + seed)
    M = int(rng.integers(1, 701))
    K = 8 * int(rng.integers(1, 151))
    n_out = 8 * int(rng.integers(1, 101))
    glu = bool(rng.random() < 0.3)
    N = 2 * n_out if glu else n_out
    layout = str(rng.choice(["kn", "nk"]))
    kernel = str(rng.choice(["single", "pair", "split"]))
    ops = _random_op_list(rng, glu)
    sd = 7000 + 100 * seed
    A = rand((M, K), sd)
    B = rand((K, N) if layout == "kn" else (N, K), sd + 1, 1.0 / math.sqrt(K))
    col = {0: rand((N,), sd + 2), 1: rand((N,), sd + 3), 2: rand((n_out,), sd + 4)}
    row = {0: torch.rand((M,), generator=torch.Generator().manual_seed(sd + 5)) + 0.5}
    aux = dict(residual=rand((M, n_out), sd + 6), z=rand((M, n_out), sd + 7), xhat=rand((M, n_out), sd + 8))
    coda.set_cta_pair("pair" if kernel == "pair" else "single")
    coda.set_split_k("force" if kernel == "split" else "off")
    try:
        r = coda.gemm_epilogue(cu(A), cu(B), ops, b_layout=layout, col_vecs={k: cu(v) for k, v in col.items()},
                               row_vecs={0: cu(row[0])}, residual=cu(aux["residual"]), z=cu(aux["z"]),
                               xhat=cu(aux["xhat"]))
        sync_ok()
    finally:
        coda.set_split_k("auto")
        coda.set_cta_pair("auto")
    ref = O.run_chain(f64(A), f64(B), ops, b_layout=layout, col_vecs={k: f64(v) for k, v in col.items()},
                      row_vecs={0: f64(row[0])}, residual_t=f64(aux["residual"]), z=f64(aux["z"]),
                      xhat=f64(aux["xhat"]))
    what = f"seed {seed}: {M}x{K}x{N} {layout} {kernel} {ops}"
    assert_close(f64(r.D), ref["D"], what)
    # each approximate activation on the way adds up to TAU_ACT of relative error
    n_act = sum(1 for o in ops if o[0] in ACTIVATIONS)
    check_stats(r, ref, what, TAU_ACT * n_act if n_act else TAU_LIN, K)


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("case", FIXED_SEQUENCE_CASES)
def test_fixed_sequence_matches_interpreter(case, layout, mode):
    # the same op list through its fixed-sequence kernel and through the
    # interpreter: both within the oracle's bound, reductions included
    ops = OP_CASES[case]
    A, B, N, n_out, col, row, aux = _op_case_tensors(ops, layout, 300 + len(case))
    args = dict(b_layout=layout, col_vecs={k: cu(v) for k, v in col.items()}, row_vecs={0: cu(row[0])},
                residual=cu(aux["residual"]), z=cu(aux["z"]), xhat=cu(aux["xhat"]))
    ref = O.run_chain(f64(A), f64(B), ops, b_layout=layout, col_vecs={k: f64(v) for k, v in col.items()},
                      row_vecs={0: f64(row[0])}, residual_t=f64(aux["residual"]), z=f64(aux["z"]),
                      xhat=f64(aux["xhat"]))
    try:
        for fixed in (True, False):
            coda.set_fixed_sequences(fixed)
            r = coda.gemm_epilogue(cu(A), cu(B), ops, **args)
            plan = coda.last_plan()
            sync_ok()
            assert (plan["sequence"] > 0) == fixed, plan
            assert_close(f64(r.D), ref["D"], f"{case} fixed={fixed}")
            check_stats(r, ref, f"{case} fixed={fixed}", chain_tau(ops), K_R)
    finally:
        coda.set_fixed_sequences(True)


# ------------------------------------------------------- dynamic tile order
# More tiles than resident clusters, so that running clusters take over the
# tiles of clusters that have not started (cluster launch control): single-CTA
# 128x256 tiles, 16 x 11 = 176 on 152 SMs; CTA pairs, 256x256 tiles, 8 x 11 =
# 88 on 76 clusters.  Ragged in M, N and K; K small so that the oracle is quick.
M_T, K_T, N_T = 2000, 104, 2600
TILE_ORDER_CASES = ["none", "bias_gelu_residual", "swiglu", "dgrad", "reductions", "chain", "rms",
                    "bias_swiglu_bias_sum"]


@pytest.mark.parametrize("kernel", ["single", "pair"])
@pytest.mark.parametrize("case", TILE_ORDER_CASES)
def test_dynamic_tile_order(case, kernel):
    # the same call in the dynamic and the static tile order: bit-identical
    # (each tile's arithmetic does not depend on which cluster ran it), and
    # within the oracle's bound
    ops = [("RMS_ROWSCALE", 0, 1e-6)] if case == "rms" else OP_CASES[case]
    glu = any(o[0] == "SWIGLU" for o in ops)
    N = 2 * N_T if glu else N_T
    n_out = N_T
    A = rand((M_T, K_T), 900 + len(case))
    B = rand((K_T, N), 901 + len(case), 1.0 / math.sqrt(K_T))
    pos = [i for i, o in enumerate(ops) if o[0] == "SWIGLU"]
    gpos = pos[0] if pos else len(ops)
    col = {o[1]: rand((N if i < gpos else n_out,), 910 + o[1])
           for i, o in enumerate(ops) if o[0] in ("COL_SCALE", "BIAS")}
    row = {0: torch.rand((M_T,), generator=torch.Generator().manual_seed(920)) + 0.5}
    aux = dict(residual=rand((M_T, n_out), 930), z=rand((M_T, n_out), 931), xhat=rand((M_T, n_out), 932))
    args = dict(col_vecs={k: cu(v) for k, v in col.items()}, row_vecs={0: cu(row[0])},
                residual=cu(aux["residual"]), z=cu(aux["z"]), xhat=cu(aux["xhat"]), seed=5)
    coda.set_cta_pair(kernel)
    coda.set_split_k("off")
    out = {}
    try:
        for order in ("dynamic", "static"):
            coda.set_tile_scheduler(order)
            r = coda.gemm_epilogue(cu(A), cu(B), ops, **args)
            plan = coda.last_plan()
            sync_ok()
            # the single-CTA commuted norm with tiles filling the grid computes its
            # row statistics in the kernel, a variant that keeps the static order
            dyn = order == "dynamic" and not (case == "rms" and kernel == "single")
            assert plan["dynamic"] == (1 if dyn else 0), plan
            assert plan["pair"] == (1 if kernel == "pair" else 0), plan
            if dyn:
                assert plan["grid"] == plan["tiles"] * (2 if kernel == "pair" else 1), plan
            out[order] = r
    finally:
        coda.set_tile_scheduler("static")
        coda.set_cta_pair("auto")
        coda.set_split_k("auto")
    d, s_ = out["dynamic"], out["static"]
    ref = O.run_chain(f64(A), f64(B), ops, col_vecs={k: f64(v) for k, v in col.items()}, row_vecs={0: f64(row[0])},
                      residual_t=f64(aux["residual"]), z=f64(aux["z"]), xhat=f64(aux["xhat"]), seed=5)
    assert torch.equal(d.D, s_.D), f"{case}: dynamic and static tile orders differ"
    for slot in ref["stats"]:      # the slots the op list writes
        assert torch.equal(d.row_stats[slot], s_.row_stats[slot]), f"{case}: row statistic {slot} differs"
    if d.keep_count is not None:
        assert torch.equal(d.keep_count, s_.keep_count)
    assert_close(f64(d.D), ref["D"], f"{case} {kernel} dynamic order")
    check_stats(d, ref, f"{case} {kernel} dynamic order", chain_tau(ops), K_T)


@pytest.mark.parametrize("op", ["SILU", "GELU_TANH", "GELU_TANH_GRAD"])
def test_activation_error_bound(op):
    # D = I @ B leaves the accumulator equal to B (exact), so the op sees bf16
    # inputs spread over [-20, 20]; with the logistic function taken from the
    # hardware tanh (absolute error <= 2^-12), SiLU and GELU may differ from the
    # exact function by 2.5e-4 |x| on top of the bf16 rounding of the output
    # (half an ulp: at most 2^-8 relative); GELU'(z) (z from the aux tensor,
    # B = 1) by 2.5e-4 (1 + 2|z u'(z)|)
    n = 256
    A = torch.eye(n, dtype=torch.float32).bfloat16()
    x = torch.linspace(-20.0, 20.0, n * n, dtype=torch.float64).reshape(n, n)
    xb = x.to(torch.bfloat16)
    if op == "GELU_TANH_GRAD":
        B = torch.ones((n, n), dtype=torch.bfloat16)
        r = coda.gemm_epilogue(cu(A), cu(B), [(op,)], z=cu(xb))
        ref = O.run_chain(f64(A), f64(B), [(op,)], z=f64(xb))["D"]
        zz = f64(xb)
        du = math.sqrt(2.0 / math.pi) * (1.0 + 3.0 * 0.044715 * zz * zz)
        allow = 2.5e-4 * (1.0 + 2.0 * np.abs(zz * du))
    else:
        r = coda.gemm_epilogue(cu(A), cu(xb), [(op,)])
        ref = O.run_chain(f64(A), f64(xb), [(op,)])["D"]
        allow = 2.5e-4 * np.abs(f64(xb))
    sync_ok()
    got = f64(r.D)
    err = np.abs(got - ref)
    bound = 1.01 * allow + 2.0 ** -8 * np.abs(ref) + 1e-30
    assert (err <= bound).all(), f"{op}: worst excess {np.max(err - bound)!r}"


@pytest.mark.parametrize("fixed", [True, False])
def test_swiglu_dropout_sequence_mask_bit_exact(fixed, mode):
    M, K, n_out = 333, 192, 264
    X = rand((M, K), 411)
    W = rand((K, 2 * n_out), 412, 1.0 / math.sqrt(K))
    ops = [("SWIGLU",), ("DROPOUT", 0, 0.1)]
    try:
        coda.set_fixed_sequences(fixed)
        r = coda.gemm_epilogue(cu(X), cu(W), ops, seed=77)
        assert (coda.last_plan()["sequence"] > 0) == fixed
        sync_ok()
    finally:
        coda.set_fixed_sequences(True)
    ref = O.run_chain(f64(X), f64(W), ops, seed=77)
    np.testing.assert_array_equal(r.keep_count.cpu().numpy().astype(np.int64), ref["keep_count"])
    nonzero = ref["D"] != 0
    np.testing.assert_array_equal((f64(r.D) != 0)[nonzero], ref["keep"][nonzero])
    assert_close(f64(r.D), ref["D"], "swiglu+dropout")


def test_unmatched_op_list_runs_interpreter():
    A, B = cu(rand((200, 128), 401)), cu(rand((128, 264), 402, 0.1))
    coda.gemm_epilogue(A, B, [("GELU_TANH",), ("SCALE", 0, 2.0)])
    assert coda.last_plan()["sequence"] == 0
    coda.gemm_epilogue(A, B, [("SILU",)])
    assert coda.last_plan()["sequence"] == 0
    coda.gemm_epilogue(A, B, [("RESIDUAL", 0, 1.0)], residual=cu(rand((200, 264), 403)))
    assert coda.last_plan()["sequence"] > 0
    sync_ok()


# -------------------------------------------------------- column reductions
def assert_col_close(got, ref, scale, n, tau, K, what=""):
    """Column reductions over n rows: the bound of the row reductions."""
    got = np.asarray(got, dtype=np.float64)
    bound = stat_bound(ref, scale, n, tau, K)
    err = np.abs(got - ref)
    if (err > bound).any():
        j = int(np.argmax(err - bound))
        raise AssertionError(f"{what}: {(err > bound).sum()} columns out of tolerance, worst column {j}: "
                             f"gpu {got[j]!r} ref {ref[j]!r} bound {bound[j]!r}")


COL_CASES = {
    "gelu_colsum_dot_rowsum": [("GELU_TANH",), ("COL_SUM", 0), ("COL_DOT_AUX", 1), ("ROW_SUM", 0)],
    "swiglu_colsumsq": [("SWIGLU",), ("COL_SUMSQ", 1), ("SCALE", 0, 2.0), ("COL_SUM", 0)],
    "dgrad_dbias": [("GELU_TANH_GRAD",), ("ROW_DOT_AUX", 0), ("ROW_SUM", 1), ("COL_SUM", 0)],
}


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("case", sorted(COL_CASES))
def test_column_reductions(case, layout, mode):
    ops = COL_CASES[case]
    A, B, N, n_out, col, row, aux = _op_case_tensors(ops, layout, 500 + len(case))
    r = coda.gemm_epilogue(cu(A), cu(B), ops, b_layout=layout, z=cu(aux["z"]), xhat=cu(aux["xhat"]))
    sync_ok()
    ref = O.run_chain(f64(A), f64(B), ops, b_layout=layout, z=f64(aux["z"]), xhat=f64(aux["xhat"]))
    assert_close(f64(r.D), ref["D"], case)
    check_stats(r, ref, case, chain_tau(ops), K_R)
    for slot, v in ref["col_stats"].items():
        assert_col_close(f64(r.col_stats[slot]), v, ref["col_stat_scale"][slot], ref["D"].shape[0], chain_tau(ops),
                         K_R, f"{case} col {slot}")


@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_reductions_exact(layout, mode):
    # Integer operands |a|, |b| <= 1 and K = 128: every product, partial sum and
    # accumulator value is an integer of magnitude <= 128, and every row and
    # column reduction below stays under 2^24 (sum of squares <= 520 * 128^2), so
    # the fp32 results are exact whatever the order of summation.  Any summand
    # left out, counted twice or taken from the wrong row or column changes an
    # integer result: the comparison is bit for bit.
    M, K, N = 300, 128, 520
    A = inputs.small_int_bf16((M, K), 1, 161)
    B = inputs.small_int_bf16((K, N) if layout == "kn" else (N, K), 1, 162)
    Xh = inputs.small_int_bf16((M, N), 2, 163)
    ops = [("ROW_SUM", 0), ("ROW_SUMSQ", 1), ("ROW_DOT_AUX", 2), ("ROW_MEAN", 3), ("COL_SUM", 0),
           ("COL_DOT_AUX", 1)]
    r = coda.gemm_epilogue(cu(A), cu(B), ops, b_layout=layout, xhat=cu(Xh))
    sync_ok()
    ref = O.run_chain(f64(A), f64(B), ops, b_layout=layout, xhat=f64(Xh))
    np.testing.assert_array_equal(f64(r.D), ref["D"])
    for slot in (0, 1, 2):
        np.testing.assert_array_equal(f64(r.row_stats[slot]), ref["stats"][slot], err_msg=f"row stat {slot}")
    # the mean is the exact sum times float32(1/N), one fp32 rounding
    mean32 = ref["stats"][0].astype(np.float32) * np.float32(1.0 / N)
    np.testing.assert_array_equal(r.row_stats[3].cpu().numpy(), mean32)
    for slot in (0, 1):
        np.testing.assert_array_equal(f64(r.col_stats[slot]), ref["col_stats"][slot], err_msg=f"col stat {slot}")


HELPER_CASES = {
    "none": [],
    "reductions": [("ROW_SUM", 0), ("ROW_MEAN", 1), ("ROW_SUMSQ", 2), ("ROW_DOT_AUX", 3)],
    "swiglu_dropout": [("SWIGLU",), ("DROPOUT", 0, 0.1)],
    "scale_preact_swiglu": [("SCALE", 0, 2.0), ("STORE_PREACT",), ("SWIGLU",), ("ROW_SUMSQ", 1)],
    "gelu_colsum_rowsum": [("GELU_TANH",), ("COL_SUM", 0), ("ROW_SUM", 0)],
    "rms_swiglu": [("RMS_ROWSCALE", 0, 1e-6), ("SWIGLU",)],
    "residual_sumsq": [("RESIDUAL", 0, 1.0), ("ROW_SUMSQ", 0)],
    "dgrad": [("GELU_TANH_GRAD",), ("ROW_DOT_AUX", 0), ("ROW_SUM", 1)],
    "bias_gelu_residual": [("BIAS", 0), ("GELU_TANH",), ("RESIDUAL", 0, 1.0)],
}


@pytest.mark.parametrize("case", sorted(HELPER_CASES))
def test_tail_helpers_bit_identical(case, mode):
    # the non-epilogue warps taking half of each CTA's last tile change nothing:
    # outputs, row and column statistics and keep counts are bit-identical; with
    # aux tensors (residual, Z, Xhat) the helpers stage their aux tiles themselves
    ops = HELPER_CASES[case]
    A, B, N, n_out, col, row, aux = _op_case_tensors(ops, "kn", 700 + len(case))
    preact = None
    if any(o[0] == "STORE_PREACT" for o in ops):
        preact = torch.zeros((M_R, N), dtype=torch.bfloat16, device="cuda")
    args = dict(col_vecs={k: cu(v) for k, v in col.items()}, residual=cu(aux["residual"]), z=cu(aux["z"]),
                xhat=cu(aux["xhat"]))
    out = []
    try:
        for helpers in (True, False):
            coda.set_tail_helpers(helpers)
            if preact is not None:
                preact.zero_()
            r = coda.gemm_epilogue(cu(A), cu(B), ops, seed=9, preact_out=preact, **args)
            sync_ok()
            out.append((r, None if preact is None else preact.clone()))
    finally:
        coda.set_tail_helpers(True)
    (a, pa), (b, pb) = out
    assert torch.equal(a.D, b.D), case
    ref = O.run_chain(f64(A), f64(B), ops, seed=9, col_vecs={k: f64(v) for k, v in col.items()},
                      residual_t=f64(aux["residual"]), z=f64(aux["z"]), xhat=f64(aux["xhat"]))
    for slot in ref["stats"]:
        assert torch.equal(a.row_stats[slot], b.row_stats[slot]), (case, slot)
    for slot in ref.get("col_stats", {}):
        assert torch.equal(a.col_stats[slot], b.col_stats[slot]), (case, slot)
    if a.keep_count is not None:
        assert torch.equal(a.keep_count, b.keep_count)
    if pa is not None:
        assert torch.equal(pa, pb)
    assert_close(f64(a.D), ref["D"], f"{case} with helpers")


def test_column_sums_exact_small_integers(mode):
    # integer-valued D (small-integer GEMM, exact in fp32): column sums are exact
    M, K, N = 300, 128, 264
    A = inputs.small_int_bf16((M, K), 3, 521)
    B = inputs.small_int_bf16((K, N), 3, 522)
    r = coda.gemm_epilogue(cu(A), cu(B), [("COL_SUM", 0), ("COL_SUMSQ", 1)])
    sync_ok()
    D = f64(A) @ f64(B)
    np.testing.assert_array_equal(f64(r.col_stats[0]), D.sum(axis=0))
    np.testing.assert_array_equal(f64(r.col_stats[1]), (D * D).sum(axis=0))


# ------------------------------------------------------ A given as [K, M]
@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_a_km_small_integer_bit_exact(layout, mode):
    if mode == "persist4":
        pytest.skip("same kernel as single")
    M, K, N = 264, 192, 264
    At = inputs.small_int_bf16((K, M), 4, 531)           # A^T stored [K, M]
    B = inputs.small_int_bf16((K, N) if layout == "kn" else (N, K), 4, 532)
    r = coda.gemm_epilogue(cu(At), cu(B), [], b_layout=layout, a_layout="km")
    sync_ok()
    # the integer sums are exact in fp32; D is their bf16 rounding (RNE)
    ref = O.round_bf16(O.gemm(f64(At).T, f64(B), layout))
    np.testing.assert_array_equal(f64(r.D), ref)


@pytest.mark.parametrize("cols", [True, False])
@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_wgrad_scale_accumulate_in_place(layout, cols, mode):
    # dW = s * X^T dH + dW_old, written over dW_old (output and residual alias),
    # with the per-row sums of squares (gradient-norm partials), and column
    # sums (the interpreter) or not (the fixed sequence of the weight gradient)
    T, K_in, N = 384, 264, 520          # tokens (the reduction), features, outputs
    X = rand((T, K_in), 541)
    dH = rand((T, N) if layout == "kn" else (N, T), 542, 1.0 / math.sqrt(T))
    dW_old = rand((K_in, N), 543)
    ops = [("SCALE", 0, 0.5), ("RESIDUAL", 0, 1.0), ("ROW_SUMSQ", 0)] + ([("COL_SUM", 0)] if cols else [])
    dW = cu(dW_old.clone())
    r = coda.gemm_epilogue(cu(X), cu(dH), ops, b_layout=layout, a_layout="km", residual=dW, out=dW)
    assert (coda.last_plan()["sequence"] == 0) == cols
    sync_ok()
    ref = O.run_chain(f64(X).T, f64(dH), ops, b_layout=layout, residual_t=f64(dW_old))
    assert_close(f64(dW), ref["D"], "wgrad")
    check_stats(r, ref, "wgrad", TAU_LIN, T)
    if cols:
        assert_col_close(f64(r.col_stats[0]), ref["col_stats"][0], ref["col_stat_scale"][0], K_in, TAU_LIN, T,
                         "wgrad colsum")


@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_wgrad_sequence_bit_identical_to_interpreter(layout, mode):
    # A as [K, M], in place: the weight gradient's fixed sequence and the
    # interpreter apply the same operations in the same order, so D and the
    # row sums of squares agree bit for bit
    T, K_in, N = 640, 392, 776
    X, dH = rand((T, K_in), 551), rand((T, N) if layout == "kn" else (N, T), 552, 1.0 / math.sqrt(T))
    dW_old = cu(rand((K_in, N), 553))
    ops = [("SCALE", 0, 0.125), ("RESIDUAL", 0, 1.0), ("ROW_SUMSQ", 0)]
    out = {}
    try:
        for fixed in (True, False):
            coda.set_fixed_sequences(fixed)
            dW = dW_old.clone()
            r = coda.gemm_epilogue(cu(X), cu(dH), ops, b_layout=layout, a_layout="km", residual=dW, out=dW)
            assert (coda.last_plan()["sequence"] > 0) == fixed
            sync_ok()
            out[fixed] = (dW.clone(), r.row_stats[0].clone())
    finally:
        coda.set_fixed_sequences(True)
    assert torch.equal(out[True][0], out[False][0])
    assert torch.equal(out[True][1], out[False][1])


# ------------------------------------------------------------ norm backward
@pytest.mark.parametrize("kind", ["layernorm", "rmsnorm"])
def test_norm_backward_chain(kind, mode):
    # forward: commuted norm projection (row statistics from the GPU forward);
    # backward: dgrad GEMM with dbeta, dgamma, g = gamma * dXn and its row sums
    # in the epilogue, then the correction kernel -> dX
    M, K_in, N = 300, 264, 520
    eps = 1e-5 if kind == "layernorm" else 1e-6
    X = rand((M, K_in), 601)
    if kind == "layernorm":
        X = (X.float() + 0.7).to(torch.bfloat16)
    g = inputs.uniform_bf16((K_in,), 0.5, 1.5, 602)
    W = rand((K_in, N), 603, 1.0 / math.sqrt(K_in))
    dY = rand((M, N), 604)
    if kind == "layernorm":
        Wf, c, b = coda.fold_layernorm(cu(W), cu(g), None, "kn")
        fwd = coda.gemm_epilogue(cu(X), Wf, [("LN_ROWSCALE", 0, eps)], ln_colsum=c)
        r, mu = fwd.row_stats[0].contiguous(), fwd.row_stats[1].contiguous()
        ops = [("COL_SUM", 1), ("COL_DOT_NORM", 0), ("COL_SCALE", 0), ("ROW_SUM", 0), ("ROW_DOT_AUX", 1)]
        row_vecs = {0: r, 1: mu}
    else:
        Wf = coda.fold_gamma(cu(W), cu(g), "kn")
        fwd = coda.gemm_epilogue(cu(X), Wf, [("RMS_ROWSCALE", 0, eps)])
        r, mu = fwd.row_stats[0].contiguous(), None
        ops = [("COL_DOT_NORM", 0), ("COL_SCALE", 0), ("ROW_DOT_AUX", 1)]
        row_vecs = {0: r}
    bwd = coda.gemm_epilogue(cu(dY), cu(W), ops, b_layout="nk", col_vecs={0: cu(g)}, row_vecs=row_vecs,
                             xhat=cu(X))
    sum_g = bwd.row_stats[0].contiguous() if kind == "layernorm" else None
    dX = coda.norm_backward(bwd.D, cu(X), r, bwd.row_stats[1].contiguous(), mu=mu, sum_g=sum_g)
    sync_ok()
    dXn = f64(dY) @ f64(W).T
    if kind == "layernorm":
        dX_ref, dg_ref, db_ref = O.layernorm_backward(f64(X), f64(g), dXn, eps)
        assert_col_close(f64(bwd.col_stats[1]), db_ref, np.sqrt((dXn ** 2).sum(axis=0)), M, TAU_LIN, N, "dbeta")
    else:
        dX_ref, dg_ref = O.rmsnorm_backward(f64(X), f64(g), dXn, eps)
    # dgamma's summands are dXn * x_hat with x_hat of unit RMS: 3 ||dXn|| bounds their L2 norm generously
    assert_col_close(f64(bwd.col_stats[0]), dg_ref, np.sqrt((dXn ** 2).sum(axis=0)) * 3.0, M, TAU_LIN, N, "dgamma")
    assert_close(f64(dX), dX_ref, f"{kind} dX")


# ------------------------------------------------------------------- FP8
def test_quantize_e4m3_rows_bit_exact():
    # rows of very different magnitudes, a zero row and a constant row: codes and
    # scales equal the oracle's float32 arithmetic bit for bit
    M, K = 300, 528
    X = rand((M, K), 701).float()
    X[1] = 0.0
    X[2] = 3.0
    X[3] *= 1e-30
    X[4] *= 1e30
    X = X.to(torch.bfloat16)
    q, sc = coda.quantize_e4m3_rows(cu(X))
    sync_ok()
    q_ref, sc_ref = O.quantize_rows_e4m3(X.float().numpy())
    np.testing.assert_array_equal(sc.cpu().numpy(), sc_ref)
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)


@pytest.mark.parametrize("M,K,N", [(300, 256, 264), (128, 512, 512), (520, 128, 136)])
def test_e4m3_gemm_exact(M, K, N, mode):
    # values are multiples of 1/8 below 16, so every fp32 partial sum is exact
    # and D is the bf16 rounding of the exact product
    A8 = inputs.random_e4m3_codes((M, K), 711)
    B8 = inputs.random_e4m3_codes((N, K), 712)
    r = coda.gemm_epilogue(cu(A8), cu(B8), [], b_layout="nk", e4m3=True)
    sync_ok()
    ref = O.round_bf16(O.gemm(O.e4m3_decode(A8.numpy()), O.e4m3_decode(B8.numpy()), "nk"))
    np.testing.assert_array_equal(f64(r.D), ref)


@pytest.mark.parametrize("glu", [False, True])
def test_e4m3_gemm_dequant_epilogue(glu, mode):
    # D = f(s_a (.)_row (A8 B8^T) (.)_col s_b): the dequantisation as epilogue ops
    M, K, n_out = 300, 384, 264
    N = 2 * n_out if glu else n_out
    A8 = inputs.random_e4m3_codes((M, K), 721, 0, 15)
    A8 = torch.where((A8 & 0x7F) == 0x7F, A8 & 0xF0, A8)     # no NaN codes
    B8 = inputs.random_e4m3_codes((N, K), 722, 0, 15)
    B8 = torch.where((B8 & 0x7F) == 0x7F, B8 & 0xF0, B8)
    sa = torch.rand((M,), generator=torch.Generator().manual_seed(723)) * 1e-3 + 1e-4
    sb = torch.rand((N,), generator=torch.Generator().manual_seed(724)) * 1e-2 + 1e-3
    ops = [("ROW_SCALE", 0), ("COL_SCALE_F32",)] + ([("SWIGLU",)] if glu else [("ROW_SUM", 0)])
    r = coda.gemm_epilogue(cu(A8), cu(B8), ops, b_layout="nk", e4m3=True, row_vecs={0: cu(sa)},
                           col_scale_f32=cu(sb))
    plan = coda.last_plan()
    sync_ok()
    assert plan["sequence"] > 0 if glu else True
    ref = O.run_chain(O.e4m3_decode(A8.numpy()), O.e4m3_decode(B8.numpy()), ops, b_layout="nk",
                      row_vecs={0: sa.double().numpy()}, col_scale_f32=sb.double().numpy())
    assert_close(f64(r.D), ref["D"], "e4m3 dequant")
    check_stats(r, ref, "e4m3 dequant", TAU_LIN, K)


@pytest.mark.parametrize("M,K,N", [(1, 16, 8), (129, 16, 264), (7, 4096, 40)])
def test_e4m3_gemm_edge_shapes(M, K, N):
    # one row; K below one 128-element k-block (zero-filled tail); a long K with a
    # narrow output
    A8 = inputs.random_e4m3_codes((M, K), 741)
    B8 = inputs.random_e4m3_codes((N, K), 742)
    r = coda.gemm_epilogue(cu(A8), cu(B8), [("ROW_SUM", 0)], b_layout="nk", e4m3=True)
    sync_ok()
    ref = O.run_chain(O.e4m3_decode(A8.numpy()), O.e4m3_decode(B8.numpy()), [("ROW_SUM", 0)], b_layout="nk")
    assert_close(f64(r.D), ref["D"], "e4m3 edge")
    check_stats(r, ref, "e4m3 edge", TAU_LIN, K)


@pytest.mark.parametrize("M,N", [(1, 8), (33, 40), (31, 264)])
def test_column_reductions_edge_shapes(M, N):
    # a single row, a partial last 32-row block, a partial last 32-column chunk
    K = 64
    A = rand((M, K), 751)
    B = rand((K, N), 752, 0.2)
    Xh = rand((M, N), 753)
    ops = [("COL_SUM", 0), ("COL_DOT_AUX", 1)]
    r = coda.gemm_epilogue(cu(A), cu(B), ops, xhat=cu(Xh))
    sync_ok()
    ref = O.run_chain(f64(A), f64(B), ops, xhat=f64(Xh))
    for slot in (0, 1):
        assert_col_close(f64(r.col_stats[slot]), ref["col_stats"][slot], ref["col_stat_scale"][slot], M, TAU_LIN, K,
                         f"col {slot}")


def test_e4m3_pipeline_approximates_bf16_gemm():
    # quantise X per row and W per output channel on the GPU, multiply in FP8 and
    # dequantise in the epilogue: the result stays within FP8's rounding
    # (2^-4 relative per operand) of the exact product of the bf16 operands
    M, K, N = 512, 1024, 768
    X = rand((M, K), 731)
    W = rand((N, K), 732, 1.0 / math.sqrt(K))
    xq, xs = coda.quantize_e4m3_rows(cu(X))
    wq, ws_ = coda.quantize_e4m3_rows(cu(W))
    r = coda.gemm_epilogue(xq, wq, [("ROW_SCALE", 0), ("COL_SCALE_F32",)], b_layout="nk", e4m3=True,
                           row_vecs={0: xs}, col_scale_f32=ws_)
    sync_ok()
    ref = f64(X) @ f64(W).T
    err = np.linalg.norm(f64(r.D) - ref) / np.linalg.norm(ref)
    assert err < 0.05, err


# --------------------------------------------------------------- MX FP8
def mx_tiled(sexp, R, K):
    """Scale bytes [R, ceil(K/32)] placed in the library's tiled storage (the
    layout coda.h defines), padding 127."""
    buf = np.full((O.mx_scale_bytes(R, K),), 127, dtype=np.uint8)
    for r in range(R):
        for j in range(sexp.shape[1]):
            buf[O.mx_scale_offset(r, j, K)] = sexp[r, j]
    return torch.from_numpy(buf)


def test_quantize_mx_e4m3_bit_exact():
    # rows of very different magnitudes, zero rows and blocks, a constant row,
    # and a K that is not a multiple of 128 (the scale storage has padding)
    R, K = 300, 160
    X = rand((R, K), 771).float()
    X[1] = 0.0
    X[2] = 3.0
    X[3] *= 1e-30
    X[4] *= 1e30
    X[5, :32] = 0.0
    X[6, 40] = 500.0                      # saturates to 448 after scaling
    X = X.to(torch.bfloat16)
    q, sc = coda.quantize_mx_e4m3(cu(X))
    sync_ok()
    q_ref, s_ref = O.quantize_mx_e4m3(f64(X))
    np.testing.assert_array_equal(q.cpu().numpy(), q_ref)
    buf = sc.cpu().numpy()
    np.testing.assert_array_equal(O.mx_scales_from_tiled(buf, R, K), s_ref)
    used = np.zeros(len(buf), dtype=bool)
    for r in range(R):
        for j in range(s_ref.shape[1]):
            used[O.mx_scale_offset(r, j, K)] = True
    assert (buf[~used] == 127).all(), "padding of the scale storage"


MX_EXACT_CASES = [(300, 256, 264), (200, 160, 512), (129, 384, 256), (1, 32, 16)]


@pytest.mark.parametrize("M,K,N", MX_EXACT_CASES)
def test_mx_gemm_exact(M, K, N, mode):
    # codes 1 .. 3.75 (multiples of 1/8) and block scales 1 or 2: every product
    # is a multiple of 1/64 below 56.25, so every partial sum (below 384 * 56.25
    # < 2^15) is exact in fp32 and D is the bf16 rounding of the exact product;
    # a scale applied to the wrong block, row or column changes D
    A8 = inputs.random_e4m3_codes((M, K), 781, 7, 8)
    B8 = inputs.random_e4m3_codes((N, K), 782, 7, 8)
    g = torch.Generator().manual_seed(783)
    nb = (K + 31) // 32
    sa = (127 + torch.randint(0, 2, (M, nb), generator=g)).to(torch.uint8).numpy()
    sb = (127 + torch.randint(0, 2, (N, nb), generator=g)).to(torch.uint8).numpy()
    r = coda.gemm_epilogue_mx(cu(A8), cu(mx_tiled(sa, M, K)), cu(B8), cu(mx_tiled(sb, N, K)), [])
    sync_ok()
    ref = O.round_bf16(O.gemm(O.dequantize_mx(A8.numpy(), sa), O.dequantize_mx(B8.numpy(), sb), "nk"))
    np.testing.assert_array_equal(f64(r.D), ref)


MX_OPS = {"swiglu": [("SWIGLU",)], "bias_gelu_rowsum": [("BIAS", 0), ("GELU_TANH",), ("ROW_SUM", 0)],
          "plain": []}


@pytest.mark.parametrize("case", sorted(MX_OPS))
def test_mx_gemm_epilogue(case, mode):
    # bf16 X and W quantised by the library (MXFP8), multiplied with the block
    # scales applied by the tensor cores, the op list in the epilogue; against
    # the oracle run on the dequantised codes the GPU produced
    ops = MX_OPS[case]
    M, K, n_out = 300, 384, 256
    N = 2 * n_out if case == "swiglu" else n_out
    X = rand((M, K), 791)
    W = rand((N, K), 792, 1.0 / math.sqrt(K))
    b = rand((n_out,), 793)
    xq, xs = coda.quantize_mx_e4m3(cu(X))
    wq, ws_ = coda.quantize_mx_e4m3(cu(W))
    r = coda.gemm_epilogue_mx(xq, xs, wq, ws_, ops, col_vecs={0: cu(b)})
    plan = coda.last_plan()
    sync_ok()
    assert plan["split"] == 0, plan
    A = O.dequantize_mx(xq.cpu().numpy(), O.mx_scales_from_tiled(xs.cpu().numpy(), M, K))
    B = O.dequantize_mx(wq.cpu().numpy(), O.mx_scales_from_tiled(ws_.cpu().numpy(), N, K))
    ref = O.run_chain(A, B, ops, b_layout="nk", col_vecs={0: f64(b)})
    assert_close(f64(r.D), ref["D"], f"mx {case}")
    check_stats(r, ref, f"mx {case}", chain_tau(ops), K)
    # and the whole pipeline stays within MXFP8's rounding of the bf16 product:
    # E4M3 rounds each operand element by up to 2^-4 relative (rms 2^-4/sqrt 3,
    # 3.6%), so a dot product of two quantised operands carries about 5% rms
    # relative error; the SwiGLU gate multiplies two such products (about 7%)
    exact = O.run_chain(f64(X), f64(W), ops, b_layout="nk", col_vecs={0: f64(b)})["D"]
    lim = 0.09 if case == "swiglu" else 0.065
    assert np.linalg.norm(f64(r.D) - exact) / np.linalg.norm(exact) < lim


def test_mx_rejections():
    A = cu(torch.zeros((64, 96), dtype=torch.uint8))
    B = cu(torch.zeros((288, 96), dtype=torch.uint8))
    s_a = cu(torch.full((coda.mx_scale_bytes(64, 96),), 127, dtype=torch.uint8))
    s_b = cu(torch.full((coda.mx_scale_bytes(288, 96),), 127, dtype=torch.uint8))
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):     # U half (144 rows in) not on a 128-row scale tile
        coda.gemm_epilogue_mx(A, s_a, B, s_b, [("SWIGLU",)])
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):     # the norms read bf16 A
        coda.gemm_epilogue_mx(A, s_a, B, s_b, [("RMS_ROWSCALE", None, 1e-6)])
    with pytest.raises(RuntimeError, match="INVALID_ARG"):     # K not a multiple of 32
        coda.gemm_epilogue_mx(A[:, :80].contiguous(), s_a, B[:, :80].contiguous(), s_b, [])


def test_full_mxfp8swiglu_sampled():
    # the SwiGLU up-projection with MXFP8 operands: X [8192, 4096] and W
    # [22016, 4096] quantised by the library, SiLU(G) * U in the epilogue
    t = inputs.make_swiglu()
    X = cu(t["X"])
    W = cu(t["W"].t().contiguous())          # [N, K]
    M, K = X.shape
    N = W.shape[0]
    xq, xs = coda.quantize_mx_e4m3(X)
    wq, ws_ = coda.quantize_mx_e4m3(W)
    r = coda.gemm_epilogue_mx(xq, xs, wq, ws_, [("SWIGLU",)])
    plan = coda.last_plan()
    sync_ok()
    assert plan["pair"] == 1 and plan["sequence"] > 0, plan
    rows = _sampled(M, 6)
    xq_ref, xs_ref = O.quantize_mx_e4m3(f64(t["X"][rows]))
    np.testing.assert_array_equal(xq.cpu().numpy()[rows], xq_ref)
    np.testing.assert_array_equal(O.mx_scales_from_tiled(xs.cpu().numpy(), M, K)[rows], xs_ref)
    A = O.dequantize_mx(xq_ref, xs_ref)
    B = O.dequantize_mx(wq.cpu().numpy(), O.mx_scales_from_tiled(ws_.cpu().numpy(), N, K))
    ref = O.run_chain(A, B, [("SWIGLU",)], b_layout="nk")
    assert_close(f64(r.D[rows]), ref["D"], "mxfp8 swiglu")


# ------------------------------------------------------------------ dropout
@pytest.mark.parametrize("seed", [0, 12345])
@pytest.mark.parametrize("glu", [False, True])
def test_dropout_mask_bit_exact(glu, seed, mode):
    # pre-dropout value = bias[j] != 0 exactly (SCALE 0 kills the GEMM), so the
    # mask is read off D without ambiguity
    M, K = 333, 64
    n_out = 264
    N = 2 * n_out if glu else n_out
    A = rand((M, K), 7)
    B = rand((K, N), 8)
    b = rand((N,), 9)
    b = torch.where(b == 0, torch.ones_like(b), b)
    ops = [("SCALE", 0, 0.0), ("BIAS", 0)]
    if glu:
        # silu(bias_G) * bias_U: pick bias so that both halves are nonzero
        ops += [("SWIGLU",)]
    ops += [("DROPOUT", 0, 0.1)]
    r = coda.gemm_epilogue(cu(A), cu(B), ops, seed=seed, col_vecs={0: cu(b)})
    sync_ok()
    ref = O.run_chain(f64(A), f64(B), ops, seed=seed, col_vecs={0: f64(b)})
    nonzero = ref["D"] != 0
    keep_gpu = f64(r.D) != 0
    np.testing.assert_array_equal(keep_gpu[nonzero | ~ref["keep"]], ref["keep"][nonzero | ~ref["keep"]])
    np.testing.assert_array_equal(r.keep_count.cpu().numpy().astype(np.int64), ref["keep_count"])
    assert_close(f64(r.D), ref["D"], "dropout values")


def test_dropout_p_zero_keeps_all(mode):
    M, K, N = 130, 64, 256
    A = rand((M, K), 1)
    B = rand((K, N), 2, 0.125)
    r = coda.gemm_epilogue(cu(A), cu(B), [("DROPOUT", 0, 0.0)], seed=99)
    r0 = coda.gemm_epilogue(cu(A), cu(B), [])
    sync_ok()
    assert torch.equal(r.D, r0.D)
    assert (r.keep_count.cpu() == N).all()


# ----------------------------------------------------------- commuted norm
@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_fold_gamma_bit_exact(layout):
    K, N = 200, 264
    W = rand((K, N) if layout == "kn" else (N, K), 3)
    g = inputs.uniform_bf16((K,), 0.5, 1.5, 4)
    got = coda.fold_gamma(cu(W), cu(g), layout)
    sync_ok()
    gw = f64(g)[:, None] * f64(W) if layout == "kn" else f64(W) * f64(g)[None, :]
    # the product of two bf16 values is exact in fp64; one RNE rounding to bf16
    expect = torch.from_numpy(gw).to(torch.bfloat16)
    assert torch.equal(got.cpu(), expect)


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("M,K,N", [(300, 192, 264), (128, 2048, 512)])
def test_commuted_rmsnorm(layout, M, K, N, mode):
    X = rand((M, K), 41)
    g = inputs.uniform_bf16((K,), 0.5, 1.5, 42)
    W = rand((K, N) if layout == "kn" else (N, K), 43, 1.0 / math.sqrt(K))
    Wf = coda.fold_gamma(cu(W), cu(g), layout)
    ops = [("RMS_ROWSCALE", 1, 1e-6)]
    r = coda.gemm_epilogue(cu(X), Wf, ops, b_layout=layout)
    plan = coda.last_plan()
    sync_ok()
    # the row statistics come from the in-kernel side path only when the tiles
    # fill the (capped) grid; otherwise from the pre-pass kernel
    assert plan["prepass"] == (0 if mode == "persist4" and plan["tiles"] >= 4 else 1), plan
    ref = O.run_chain(f64(X), f64(W), ops, b_layout=layout, norm_gamma=f64(g))
    assert_close(f64(r.D), ref["D"], "commuted rmsnorm")
    assert_close(f64(r.row_stats[1]), ref["stats"][1], "rms row scale")


@pytest.mark.parametrize("exact_gamma", [False, True])
def test_commuted_rmsnorm_then_swiglu(exact_gamma, mode):
    # r_i applies to both halves before the nonlinearity: silu(r G) * (r U).
    # With gamma in {1/2, 1, 2} the fold gamma*W is exact in bf16, so the GPU
    # and the oracle see the same weights and the row sum gets the strict bound.
    M, K, n_out = 200, 256, 136
    X = rand((M, K), 51)
    if exact_gamma:
        g = torch.tensor([0.5, 1.0, 2.0])[torch.randint(0, 3, (K,), generator=torch.Generator().manual_seed(5))]
        g = g.to(torch.bfloat16)
    else:
        g = inputs.uniform_bf16((K,), 0.5, 1.5, 52)
    W = rand((K, 2 * n_out), 53, 1.0 / math.sqrt(K))
    Wf = coda.fold_gamma(cu(W), cu(g), "kn")
    ops = [("RMS_ROWSCALE", 0, 1e-6), ("SWIGLU",), ("ROW_SUM", 1)]
    r = coda.gemm_epilogue(cu(X), Wf, ops)
    sync_ok()
    ref = O.run_chain(f64(X), f64(W), ops, norm_gamma=f64(g))
    assert_close(f64(r.D), ref["D"], "rms -> swiglu")
    assert_close(f64(r.row_stats[0]), ref["stats"][0], "rms r")
    if exact_gamma:
        assert_close(f64(r.row_stats[1]), ref["stats"][1], "row sum (exact fold)")
    else:
        check_stats(r, ref, "rms -> swiglu", chain_tau(ops, fold=True), K)


@pytest.mark.parametrize("glu", [False, True])
@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_commuted_rmsnorm_from_row_sumsq(layout, glu, mode):
    # RMS_SUMSQ_ROWSCALE: r_i from the row sums of squares of A supplied by the
    # caller (here by the library's own unfused ROW_SUMSQ pass over A), no
    # pre-pass; the result is rmsnorm(A; gamma) @ W, the oracle's
    # normalise-then-project, within the bound of the fold (the weights are the
    # bf16 fold gamma (.)_row W)
    M, K, n_out = 300, 192, 264
    N = 2 * n_out if glu else n_out
    X = rand((M, K), 171)
    g = inputs.uniform_bf16((K,), 0.5, 1.5, 172)
    W = rand((K, N) if layout == "kn" else (N, K), 173, 1.0 / math.sqrt(K))
    Wf = coda.fold_gamma(cu(W), cu(g), layout)
    ss = coda.epilogue_apply(cu(X), [("ROW_SUMSQ", 0)]).row_stats[0].contiguous()
    ops = [("RMS_SUMSQ_ROWSCALE", 1, 1e-6)] + ([("SWIGLU",)] if glu else []) + [("ROW_SUM", 0)]
    before = coda.launch_count()
    r = coda.gemm_epilogue(cu(X), Wf, ops, b_layout=layout, row_vecs={1: ss})
    plan = coda.last_plan()
    launched = coda.launch_count() - before
    sync_ok()
    assert plan["prepass"] == 0, plan
    # the GEMM and the row sum's finishing kernel, nothing else (no pass over A)
    assert launched == 2, launched
    # elementwise against the oracle given the prepared weights (the fold
    # bf16(gamma (.)_row W), rounded by the oracle itself: its 2^-9 rounding
    # reaches the bound in silu(G) * U where U is near zero), and within the
    # Frobenius bound of the pages' normalise-then-project with exact gamma
    ss64 = O.row_sumsq(f64(X))
    Wp = O.round_bf16(f64(g)[:, None] * f64(W) if layout == "kn" else f64(W) * f64(g)[None, :])
    ref = O.run_chain(f64(X), Wp, ops, b_layout=layout, row_vecs={1: ss64})
    assert_close(f64(r.D), ref["D"], "rms from sums of squares")
    check_stats(r, ref, "rms from sums of squares", chain_tau(ops), K)
    ref0 = O.run_chain(f64(X), f64(W), ops, b_layout=layout, norm_gamma=f64(g), row_vecs={1: ss64})
    assert np.linalg.norm(f64(r.D) - ref0["D"]) / np.linalg.norm(ref0["D"]) <= FRO
    # the supplied sums themselves: fp32 sums of exact bf16 squares
    assert_stat_close(f64(ss), ss64, 2.0 * np.sqrt(O.row_sumsq(f64(X) ** 2)), K, TAU_LIN, 0, "sumsq")


def test_rms_from_row_sumsq_rejections():
    X = cu(rand((64, 64), 181))
    ss = torch.ones((64,), dtype=torch.float32, device="cuda")
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):
        coda.epilogue_apply(X, [("RMS_SUMSQ_ROWSCALE", 0, 1e-6)], row_vecs={0: ss})
    with pytest.raises(RuntimeError, match="INVALID_ARG"):     # no row vector in the slot
        coda.gemm_epilogue(X, X, [("RMS_SUMSQ_ROWSCALE", 1, 1e-6)], row_vecs={0: ss})
    with pytest.raises(RuntimeError, match="INVALID_ARG"):     # two norms
        coda.gemm_epilogue(X, X, [("RMS_SUMSQ_ROWSCALE", 0, 1e-6), ("RMS_ROWSCALE", None, 1e-6)],
                           row_vecs={0: ss})


@pytest.mark.parametrize("kernel", ["single", "pair"])
def test_raster_orders_bit_identical(kernel):
    # the same call in row-group and column-group tile orders of several group
    # sizes: every tile's arithmetic is the same wherever it runs, so D and the
    # row and column statistics are bit-identical; more tiles than resident
    # CTAs (pairs) in both dimensions, ragged M, N and K
    M, K, N = 2000, 104, 2600
    A = rand((M, K), 191)
    B = rand((K, N), 192, 1.0 / math.sqrt(K))
    b = rand((N,), 193)
    ops = [("BIAS", 0), ("GELU_TANH",), ("ROW_SUM", 0), ("ROW_SUMSQ", 1), ("COL_SUM", 0)]
    coda.set_cta_pair(kernel)
    coda.set_split_k("off")
    outs = []
    try:
        for mode, grp in (("rows", 1), ("rows", 3), ("cols", 1), ("cols", 4), ("cols", 0), ("auto", 0)):
            coda.set_raster(mode, grp)
            outs.append(coda.gemm_epilogue(cu(A), cu(B), ops, col_vecs={0: cu(b)}))
            sync_ok()
    finally:
        coda.set_raster("auto", 0)
        coda.set_cta_pair("auto")
        coda.set_split_k("auto")
    r0 = outs[0]
    for r in outs[1:]:
        assert torch.equal(r.D, r0.D)
        assert torch.equal(r.row_stats, r0.row_stats)
        assert torch.equal(r.col_stats, r0.col_stats)
    ref = O.run_chain(f64(A), f64(B), ops, col_vecs={0: f64(b)})
    assert_close(f64(r0.D), ref["D"], "raster orders")
    check_stats(r0, ref, "raster orders", chain_tau(ops), K)


# ------------------------------------------------------ commuted LayerNorm
@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("with_beta", [True, False])
def test_fold_layernorm(layout, with_beta):
    K, N = 200, 264
    W = rand((K, N) if layout == "kn" else (N, K), 81, 1.0 / math.sqrt(K))
    g = inputs.uniform_bf16((K,), 0.5, 1.5, 82)
    beta = rand((K,), 83, 0.3) if with_beta else None
    Wf, c, b = coda.fold_layernorm(cu(W), cu(g), cu(beta) if with_beta else None, layout)
    sync_ok()
    # the folded weights are the RMS fold's (one RNE rounding of an exact product)
    assert torch.equal(Wf.cpu(), coda.fold_gamma(cu(W), cu(g), layout).cpu())
    Wkn = f64(W) if layout == "kn" else f64(W).T
    Wf_kn = f64(Wf) if layout == "kn" else f64(Wf).T
    # c = the column sums of the weights the GEMM actually multiplies (the bf16
    # fold), so X@Wf - mu c is (X - mu)@Wf up to fp32 summation error
    c_ref = Wf_kn.sum(axis=0)
    c_tol = 1e-5 * np.abs(Wf_kn).sum(axis=0) + 1e-6
    assert (np.abs(f64(c) - c_ref) <= c_tol).all()
    b_ref = f64(beta) @ Wkn if with_beta else np.zeros(N)
    b_tol = 1e-5 * (np.abs(f64(beta)) @ np.abs(Wkn) if with_beta else np.zeros(N)) + 1e-6
    assert (np.abs(f64(b) - b_ref) <= b_tol).all()


def _ln_problem(M, K, N, layout, seed, mean=0.5):
    # nonzero row means (a common offset plus a per-row shift), so the mu c term matters
    X = inputs.randn_bf16((M, K), 1.0, seed)
    shift = inputs.randn_bf16((M, 1), 0.5, seed + 1)
    X = (X.float() + mean + shift.float()).to(torch.bfloat16)
    g = inputs.uniform_bf16((K,), 0.5, 1.5, seed + 2)
    beta = rand((K,), seed + 3, 0.3)
    W = rand((K, N) if layout == "kn" else (N, K), seed + 4, 1.0 / math.sqrt(K))
    return X, g, beta, W


@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("M,K,N", [(300, 192, 264), (128, 2048, 512), (520, 512, 136), (300, 264, 264)])
def test_commuted_layernorm(layout, M, K, N, mode):
    X, g, beta, W = _ln_problem(M, K, N, layout, 91)
    Wf, c, b = coda.fold_layernorm(cu(W), cu(g), cu(beta), layout)
    ops = [("LN_ROWSCALE", 1, 1e-5)]
    r = coda.gemm_epilogue(cu(X), Wf, ops, b_layout=layout, ln_colsum=c, ln_bias=b)
    sync_ok()
    ref = O.run_chain(f64(X), f64(W), ops, b_layout=layout, norm_gamma=f64(g), norm_beta=f64(beta))
    assert_close(f64(r.D), ref["D"], "commuted layernorm")
    assert_close(f64(r.row_stats[1]), ref["stats"][1], "ln r")
    # mu is a mean of bf16 values: fp32 summation error only
    mu = f64(r.row_stats[2])
    assert (np.abs(mu - ref["stats"][2]) <= 1e-5 * (1 + np.abs(ref["stats"][2]))).all()


def test_commuted_layernorm_large_mean(mode):
    # rows with mean 30 and spread 1: the variance must come from the spread,
    # not from the difference of two large second moments
    M, K, N = 260, 1024, 264
    X, g, beta, W = _ln_problem(M, K, N, "kn", 141, mean=30.0)
    Wf, c, b = coda.fold_layernorm(cu(W), cu(g), cu(beta), "kn")
    ops = [("LN_ROWSCALE", 0, 1e-5)]
    r = coda.gemm_epilogue(cu(X), Wf, ops, ln_colsum=c, ln_bias=b)
    sync_ok()
    ref = O.run_chain(f64(X), f64(W), ops, norm_gamma=f64(g), norm_beta=f64(beta))
    assert_close(f64(r.D), ref["D"], "layernorm, mean 30")
    assert_close(f64(r.row_stats[0]), ref["stats"][0], "ln r, mean 30")
    mu = f64(r.row_stats[1])
    assert (np.abs(mu - ref["stats"][1]) <= 1e-5 * (1 + np.abs(ref["stats"][1]))).all()


def test_commuted_layernorm_no_beta_no_slot(mode):
    M, K, N = 260, 320, 200
    X, g, _, W = _ln_problem(M, K, N, "kn", 101, mean=-1.0)
    Wf, c, b = coda.fold_layernorm(cu(W), cu(g), None, "kn")
    ops = [("LN_ROWSCALE", -1, 1e-5), ("GELU_ERF",)]
    r = coda.gemm_epilogue(cu(X), Wf, ops, ln_colsum=c)
    sync_ok()
    ref = O.run_chain(f64(X), f64(W), ops, norm_gamma=f64(g))
    assert_close(f64(r.D), ref["D"], "ln (no beta) -> erf gelu")


@pytest.mark.parametrize("with_beta", [True, False])
def test_commuted_layernorm_then_swiglu(with_beta, mode):
    # r and mu apply to both halves before the nonlinearity, each half with its
    # own column sums and bias (none without beta).  Elementwise against the
    # oracle given the prepared weights (the fold bf16(gamma (.)_row W), rounded
    # by the oracle itself, its column sums and beta^T W: the 2^-9 rounding of
    # the fold reaches the elementwise bound in silu(G) * U where U is near
    # zero), and within the Frobenius bound of normalise-then-project
    M, K, n_out = 200, 256, 136
    X, g, beta, W = _ln_problem(M, K, 2 * n_out, "kn", 111)
    Wf, c, b = coda.fold_layernorm(cu(W), cu(g), cu(beta) if with_beta else None, "kn")
    ops = [("LN_ROWSCALE", 0, 1e-5), ("SWIGLU",), ("ROW_SUM", 2)]
    r = coda.gemm_epilogue(cu(X), Wf, ops, ln_colsum=c, ln_bias=b if with_beta else None)
    assert abs(coda.last_plan()["colvecs"]) == (4 if with_beta else 2)   # c (and b), each with its up half
    sync_ok()
    Wp = O.round_bf16(f64(g)[:, None] * f64(W))
    ref = O.run_chain(f64(X), Wp, ops, ln_colsum=Wp.sum(axis=0),
                      ln_bias=f64(beta) @ f64(W) if with_beta else None)
    assert_close(f64(r.D), ref["D"], "ln -> swiglu")
    assert_close(f64(r.row_stats[0]), ref["stats"][0], "ln r")
    check_stats(r, {"D": ref["D"], "stats": {2: ref["stats"][2]}, "stat_scale": ref["stat_scale"]}, "ln -> swiglu",
                chain_tau(ops), K)
    ref0 = O.run_chain(f64(X), f64(W), ops, norm_gamma=f64(g), norm_beta=f64(beta) if with_beta else None)
    assert np.linalg.norm(f64(r.D) - ref0["D"]) / np.linalg.norm(ref0["D"]) <= FRO


def test_column_vector_slices_staged_or_prefetched(mode):
    # Column vectors reach the epilogue as per-tile slices copied to shared
    # memory (up to 8: here 5, the SwiGLU up halves included) or, past 8, as
    # global loads prefetched into L1 (here 10 slices): both against the oracle,
    # ragged in every dimension, several tiles per CTA in persist4
    cases = {5: [("BIAS", 0), ("COL_SCALE", 1), ("SWIGLU",), ("BIAS", 2)],
             -8: [("BIAS", 0), ("COL_SCALE", 1), ("BIAS", 2), ("COL_SCALE", 3), ("BIAS", 0), ("SWIGLU",)]}
    for want, ops in cases.items():
        A, B, N, n_out, col, row, aux = _op_case_tensors(ops, "kn", 700 + want)
        r = coda.gemm_epilogue(cu(A), cu(B), ops, col_vecs={k: cu(v) for k, v in col.items()})
        assert coda.last_plan()["colvecs"] == want, coda.last_plan()
        sync_ok()
        ref = O.run_chain(f64(A), f64(B), ops, col_vecs={k: f64(v) for k, v in col.items()})
        assert_close(f64(r.D), ref["D"], f"{len(ops)} ops, colvecs {want}")


def test_layernorm_rowscale_rejected_unfused_and_without_colsum():
    C = cu(rand((64, 64), 121))
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):
        coda.epilogue_apply(C, [("LN_ROWSCALE", -1, 1e-5)])
    with pytest.raises(RuntimeError, match="INVALID_ARG"):
        coda.gemm_epilogue(C, C, [("LN_ROWSCALE", -1, 1e-5)])


# --------------------------------------------------------------------- dgrad
def test_dgrad_small(mode):
    M, K, N = 300, 128, 520
    dY = rand((M, K), 61)
    W = rand((N, K), 62, 1.0 / math.sqrt(K))
    Z = rand((M, N), 63)
    Xh = rand((M, N), 64)
    ops = [("GELU_TANH_GRAD",), ("ROW_DOT_AUX", 0), ("ROW_SUM", 1)]
    r = coda.gemm_epilogue(cu(dY), cu(W), ops, b_layout="nk", z=cu(Z), xhat=cu(Xh))
    sync_ok()
    ref = O.run_chain(f64(dY), f64(W), ops, b_layout="nk", z=f64(Z), xhat=f64(Xh))
    assert_close(f64(r.D), ref["D"], "dgrad dX")
    check_stats(r, ref, "dgrad", chain_tau(ops), K)


# --------------------------------------------------------- unfused kernels
def test_unfused_rmsnorm():
    M, K = 300, 520
    X = rand((M, K), 71)
    g = inputs.uniform_bf16((K,), 0.5, 1.5, 72)
    xn, rstd = coda.rmsnorm(cu(X), cu(g), 1e-6)
    sync_ok()
    assert_close(f64(xn), O.rmsnorm(f64(X), f64(g), 1e-6), "rmsnorm")
    assert_close(f64(rstd), O.rms_rstd(f64(X), 1e-6), "rstd")


@pytest.mark.parametrize("with_beta", [True, False])
def test_unfused_layernorm(with_beta):
    M, K = 300, 520
    X, g, beta, _ = _ln_problem(M, K, 8, "kn", 131)
    xn = coda.layernorm(cu(X), cu(g), cu(beta) if with_beta else None, 1e-5)
    sync_ok()
    assert_close(f64(xn), O.layernorm(f64(X), f64(g), f64(beta) if with_beta else None, 1e-5), "layernorm")


@pytest.mark.parametrize("case", ["chain", "swiglu", "reductions", "gelu_grad", "bias_swiglu_bias_sum"])
def test_unfused_epilogue_apply(case):
    ops = OP_CASES[case]
    A, B, N, n_out, col, row, aux = _op_case_tensors(ops, "kn", 300)
    C = rand((M_R, N), 301)
    r = coda.epilogue_apply(cu(C), ops, col_vecs={k: cu(v) for k, v in col.items()}, row_vecs={0: cu(row[0])},
                            residual=cu(aux["residual"]), z=cu(aux["z"]), xhat=cu(aux["xhat"]))
    sync_ok()
    # C = C @ I exactly, so the oracle chain on (C, I) is the epilogue alone
    ref = O.run_chain(f64(C), np.eye(N), ops, col_vecs={k: f64(v) for k, v in col.items()},
                      row_vecs={0: f64(row[0])}, residual_t=f64(aux["residual"]), z=f64(aux["z"]),
                      xhat=f64(aux["xhat"]))
    assert_close(f64(r.D), ref["D"], f"apply {case}")
    check_stats(r, ref, f"apply {case}", chain_tau(ops), 0)


def test_unfused_dropout_matches_fused_mask():
    M, N = 257, 264
    C = rand((M, N), 81)
    r = coda.epilogue_apply(cu(C), [("DROPOUT", 0, 0.1)], seed=7)
    sync_ok()
    ref = O.run_chain(f64(C), np.eye(N), [("DROPOUT", 0, 0.1)], seed=7)
    np.testing.assert_array_equal(r.keep_count.cpu().numpy().astype(np.int64), ref["keep_count"])
    assert_close(f64(r.D), ref["D"], "unfused dropout")


# ------------------------------------------------- full-size, sampled rows
def _sampled(M, seed):
    """512 random rows, the first and last row, and both rows at every 128-row
    boundary (so at every 256-row CTA-pair tile boundary too)."""
    return inputs.sample_rows(M, 512, seed)


def test_full_rmsproj_sampled():
    w = inputs.WORKLOADS["rmsproj"]
    t = inputs.make_rmsproj()
    Wf = coda.fold_gamma(cu(t["W"]), cu(t["gamma"]), "kn")
    ops = [("RMS_ROWSCALE", 0, inputs.EPS_RMS)]
    r = coda.gemm_epilogue(cu(t["X"]), Wf, ops)
    sync_ok()
    rows = _sampled(w.M, 1)
    ref = O.run_chain(f64(t["X"][rows]), f64(t["W"]), ops, norm_gamma=f64(t["gamma"]))
    assert_close(f64(r.D[rows]), ref["D"], "rmsproj")
    assert_close(f64(r.row_stats[0][rows]), ref["stats"][0], "rmsproj r")


def test_full_lnproj_sampled():
    w = inputs.WORKLOADS["lnproj"]
    t = inputs.make_lnproj()
    Wf, c, b = coda.fold_layernorm(cu(t["W"]), cu(t["gamma"]), cu(t["beta"]), "kn")
    ops = [("LN_ROWSCALE", 0, inputs.EPS_LN)]
    r = coda.gemm_epilogue(cu(t["X"]), Wf, ops, ln_colsum=c, ln_bias=b)
    sync_ok()
    rows = _sampled(w.M, 2)
    ref = O.run_chain(f64(t["X"][rows]), f64(t["W"]), ops, norm_gamma=f64(t["gamma"]), norm_beta=f64(t["beta"]))
    assert_close(f64(r.D[rows]), ref["D"], "lnproj")
    assert_close(f64(r.row_stats[0][rows]), ref["stats"][0], "lnproj r")
    assert_close(f64(r.row_stats[1][rows]), ref["stats"][1], "lnproj mu")


def test_split_k_plan_and_segments():
    # 3 x 2 tiles over 3 k-blocks: 18 units on 9 CTAs, two per tile's k range
    coda.set_cta_pair("single")
    coda.set_split_k("force")
    try:
        M, K, N = 300, 192, 264
        X = rand((M, K), 151)
        W = rand((K, N), 152, 1.0 / math.sqrt(K))
        ops = [("GELU_TANH",), ("ROW_SUM", 0)]
        r = coda.gemm_epilogue(cu(X), cu(W), ops)
        plan = coda.last_plan()
        sync_ok()
        assert plan["split"] == 1 and plan["pair"] == 0 and plan["tiles"] == 6 and plan["grid"] == 9, plan
        ref = O.run_chain(f64(X), f64(W), ops)
        assert_close(f64(r.D), ref["D"], "split GEMM")
        check_stats(r, ref, "split GEMM", chain_tau(ops), K)
        # too small a workspace for the partials: same result without the split
        need = coda.workspace_size(M, N, K, ops)
        small = torch.empty((2 * M * 4,), dtype=torch.uint8, device="cuda")
        assert need > small.numel()
        r2 = coda.gemm_epilogue(cu(X), cu(W), ops, workspace=small)
        assert coda.last_plan()["split"] == 0
        sync_ok()
        assert_close(f64(r2.D), ref["D"], "unsplit GEMM")
    finally:
        coda.set_split_k("auto")
        coda.set_cta_pair("auto")


WAVE_SPLIT_CASES = {
    "plain": [],
    "gelu_rowsum": [("GELU_TANH",), ("ROW_SUM", 0)],
    "residual_sumsq": [("RESIDUAL", 0, 1.0), ("ROW_SUMSQ", 0)],
    "swiglu": [("SWIGLU",)],
    "dgrad_dbias": [("GELU_TANH_GRAD",), ("ROW_DOT_AUX", 0), ("ROW_SUM", 1), ("COL_SUM", 0)],
}


@pytest.mark.parametrize("kernel", ["pair", "single"])
@pytest.mark.parametrize("case", sorted(WAVE_SPLIT_CASES))
def test_last_waves_split(kernel, case):
    # Enough tiles for three waves on the device's clusters (160 CTA-pair tiles,
    # 320 single-CTA tiles; ragged in M, N and K): forced, the tiles of the last
    # two waves are shared out as (tile, k-block) runs over every cluster, the
    # earlier ones run whole.  Split and unsplit runs both match the oracle.
    ops = WAVE_SPLIT_CASES[case]
    glu = any(o[0] == "SWIGLU" for o in ops)
    M, K = 4000, 456
    N = 2528 if glu else 2520
    n_out = N // 2 if glu else N
    A = rand((M, K), 1301)
    B = rand((K, N), 1302, 1.0 / math.sqrt(K))
    aux = dict(residual=rand((M, n_out), 1303), z=rand((M, n_out), 1304), xhat=rand((M, n_out), 1305))
    ref = O.run_chain(f64(A), f64(B), ops, residual_t=f64(aux["residual"]), z=f64(aux["z"]), xhat=f64(aux["xhat"]))
    coda.set_cta_pair(kernel)
    try:
        for mode in ("force", "off"):
            coda.set_split_k(mode)
            r = coda.gemm_epilogue(cu(A), cu(B), ops, residual=cu(aux["residual"]), z=cu(aux["z"]),
                                   xhat=cu(aux["xhat"]))
            plan = coda.last_plan()
            sync_ok()
            assert plan["pair"] == (1 if kernel == "pair" else 0), plan
            clusters = plan["grid"] // (2 if kernel == "pair" else 1)
            assert plan["tiles"] >= 2 * clusters, plan
            assert plan["split"] == (1 if mode == "force" else 0), plan
            what = f"{case} {kernel} split={mode}"
            assert_close(f64(r.D), ref["D"], what)
            check_stats(r, ref, what, chain_tau(ops), K)
            for slot, v in ref.get("col_stats", {}).items():
                assert_col_close(f64(r.col_stats[slot]), v, ref["col_stat_scale"][slot], M, chain_tau(ops), K,
                                 f"{what} col stat {slot}")
    finally:
        coda.set_split_k("auto")
        coda.set_cta_pair("auto")


@pytest.mark.parametrize("kernel", ["pair", "single"])
def test_last_waves_split_e4m3_exact(kernel):
    # FP8 codes that are multiples of 1/8 below 16 and K = 512: every partial
    # sum is exact in fp32, so the split tiles (partials published, added by
    # the last contributor) give D bit for bit
    M, K, N = 4000, 512, 2560
    A8 = inputs.random_e4m3_codes((M, K), 1321)
    B8 = inputs.random_e4m3_codes((N, K), 1322)
    ref = O.round_bf16(O.gemm(O.e4m3_decode(A8.numpy()), O.e4m3_decode(B8.numpy()), "nk"))
    coda.set_cta_pair(kernel)
    coda.set_split_k("force")
    try:
        r = coda.gemm_epilogue(cu(A8), cu(B8), [], b_layout="nk", e4m3=True)
        plan = coda.last_plan()
        sync_ok()
    finally:
        coda.set_split_k("auto")
        coda.set_cta_pair("auto")
    assert plan["split"] == 1 and plan["pair"] == (1 if kernel == "pair" else 0), plan
    np.testing.assert_array_equal(f64(r.D), ref)


def test_last_waves_split_auto_plan():
    # automatic: 160 CTA-pair tiles (4096 x 2560) on 76 clusters leave 68 of 228
    # cluster-tile slots of the third wave idle (30%), so the last waves split;
    # 152 tiles (4864 x 2048) fill two waves exactly and 1024 tiles (16384 x
    # 4096) leave 40 of 1064 slots (3.8%) idle, and neither splits
    for M, N, want in ((4096, 2560, 1), (4864, 2048, 0), (16384, 4096, 0)):
        A = rand((M, 512), 1311)
        B = rand((512, N), 1312, 1.0 / math.sqrt(512))
        coda.gemm_epilogue(cu(A), cu(B), [])
        plan = coda.last_plan()
        sync_ok()
        clusters = plan["grid"] // 2
        if clusters != 76:
            pytest.skip(f"plan for 76 clusters of CTA pairs; this device gives {clusters}")
        assert plan["split"] == want, (N, plan)


@pytest.mark.parametrize("split", ["auto", "force", "sumsq"])
def test_full_skinny_sampled(split):
    # the decode-sized up-projection: 86 tiles on one CTA each (automatic), split
    # over K across all SMs (forced), and with the input's row sums of squares
    # supplied (as the benchmark runs it: no pre-pass)
    w = inputs.WORKLOADS["skinny"]
    t = inputs.make_skinny()
    Wf = coda.fold_gamma(cu(t["W"]), cu(t["gamma"]), "kn")
    ops = [("RMS_ROWSCALE", 0, inputs.EPS_RMS), ("SWIGLU",)]
    coda.set_split_k("auto" if split == "sumsq" else split)
    try:
        if split == "sumsq":
            from gemm_epilogue_transformer_tmem_gb300 import workloads
            X = cu(t["X"])
            rs = torch.empty((1, w.M), dtype=torch.float32, device="cuda")
            r = coda.gemm_epilogue(X, Wf, [("RMS_SUMSQ_ROWSCALE", 0, inputs.EPS_RMS), ("SWIGLU",)],
                                   row_vecs={0: workloads.row_sumsq(X)}, row_stats=rs)
        else:
            r = coda.gemm_epilogue(cu(t["X"]), Wf, ops)
        plan = coda.last_plan()
        sync_ok()
    finally:
        coda.set_split_k("auto")
    assert plan["prepass"] == (0 if split == "sumsq" else 1), plan
    assert plan["split"] == (1 if split == "force" else 0), plan
    if split == "force":
        assert plan["grid"] > plan["tiles"], plan
    assert r.D.shape == (w.M, w.N // 2)
    # As in the LLaMA block (the same weights at 128 tokens): the weight fold
    # bf16(gamma (.)_row W) is the documented preparation, rounded by the
    # oracle itself.  Its rounding error (2^-9 relative per weight) grows to
    # ~1e-2 absolute in silu(G)*U where |U| is large and silu(G) small, so the
    # elementwise bound takes the prepared weights, and the unprepared oracle
    # gets the Frobenius bound.
    g, W = f64(t["gamma"]), f64(t["W"])
    ref = O.run_chain(f64(t["X"]), O.round_bf16(g[:, None] * W), ops, norm_gamma=np.ones_like(g))
    assert_close(f64(r.D), ref["D"], "skinny")
    if split != "sumsq":     # with supplied sums r is not written out
        assert_close(f64(r.row_stats[0]), ref["stats"][0], "skinny r")
    ref0 = O.run_chain(f64(t["X"]), W, ops, norm_gamma=g)
    got = f64(r.D)
    fro0 = np.linalg.norm(got - ref0["D"]) / np.linalg.norm(ref0["D"])
    over = np.abs(got - ref0["D"]) > ATOL + RTOL * np.abs(ref0["D"])
    print(f"skinny ({split}) against the unprepared oracle: {int(over.sum())} of {over.size} elements over the "
          f"elementwise bound, worst excess {float(np.max(np.abs(got - ref0['D']) - ATOL - RTOL * np.abs(ref0['D']))):.3e}, "
          f"relative Frobenius {fro0:.3e}")
    assert fro0 <= FRO


def test_full_wgrad_sampled():
    # dW = s * up^T dY + dW_old written in place, on the full-size shapes
    t = inputs.make_wgrad()
    ops = [("SCALE", 0, inputs.WGRAD_SCALE), ("RESIDUAL", 0, 1.0), ("ROW_SUMSQ", 0)]
    dW = cu(t["dW_old"].clone())
    r = coda.gemm_epilogue(cu(t["up"]), cu(t["dY"]), ops, a_layout="km", residual=dW, out=dW)
    sync_ok()
    rows = _sampled(t["dW_old"].shape[0], 5)
    ref = O.run_chain(f64(t["up"][:, rows]).T, f64(t["dY"]), ops, residual_t=f64(t["dW_old"][rows]))
    assert_close(f64(dW[rows]), ref["D"], "wgrad")
    assert_stat_close(f64(r.row_stats[0][rows]), ref["stats"][0], ref["stat_scale"][0], dW.shape[1], TAU_LIN,
                      t["up"].shape[0], "wgrad row sumsq")


def test_full_swiglu_dropout_sampled():
    w = inputs.WORKLOADS["swiglu"]
    t = inputs.make_swiglu()
    ops = [("SWIGLU",), ("DROPOUT", 0, inputs.DROPOUT_P)]
    r = coda.gemm_epilogue(cu(t["X"]), cu(t["W"]), ops, seed=inputs.DROPOUT_SEED)
    sync_ok()
    rows = _sampled(w.M, 2)
    ref = O.run_chain(f64(t["X"][rows]), f64(t["W"]), ops, seed=inputs.DROPOUT_SEED, rows=rows)
    assert_close(f64(r.D[rows]), ref["D"], "swiglu+dropout")
    kc = r.keep_count.cpu().numpy().astype(np.int64)
    np.testing.assert_array_equal(kc[rows], ref["keep_count"])
    # keep rate over the whole 8192 x 11008 output within 1-p +- 3 sigma
    n = w.M * (w.N // 2)
    p = inputs.DROPOUT_P
    rate = kc.sum() / n
    assert abs(rate - (1 - p)) < 3 * math.sqrt(p * (1 - p) / n), rate


def test_full_dgrad_sampled():
    w = inputs.WORKLOADS["dgrad"]
    t = inputs.make_dgrad()
    ops = [("GELU_TANH_GRAD",), ("ROW_DOT_AUX", 0), ("ROW_SUM", 1)]
    r = coda.gemm_epilogue(cu(t["dY"]), cu(t["W"]), ops, b_layout="nk", z=cu(t["Z"]), xhat=cu(t["Xhat"]))
    sync_ok()
    rows = _sampled(w.M, 3)
    ref = O.run_chain(f64(t["dY"][rows]), f64(t["W"]), ops, b_layout="nk", z=f64(t["Z"][rows]),
                      xhat=f64(t["Xhat"][rows]))
    assert_close(f64(r.D[rows]), ref["D"], "dgrad")
    for slot in (0, 1):
        assert_stat_close(f64(r.row_stats[slot][rows]), ref["stats"][slot], ref["stat_scale"][slot], w.N,
                          chain_tau(ops), w.K, f"dgrad stat {slot}")


def test_llama_e2e_token_blocks_match_the_step():
    # The end-to-end step copies the block's inputs in, runs its calls and
    # reads its outputs back in token blocks on three streams (events order
    # them).  Every call is row-wise, so with the split over K off the outputs
    # read back equal the device-resident step's bit for bit.
    from gemm_epilogue_transformer_tmem_gb300 import workloads
    coda.set_split_k("off")
    try:
        step = workloads.build_llama(dev="cuda", tokens=2048)
        step.fused()
        torch.cuda.synchronize()
        ref = {k: v.detach().cpu().clone() for k, v in step.host_outputs.items()}
        hin = {k: v.detach().cpu().clone().pin_memory() for k, v in step.host_inputs.items()}
        hout = {k: torch.full(v.shape, float("nan"), dtype=v.dtype).pin_memory() for k, v in step.host_outputs.items()}
        for v in step.host_outputs.values():
            v.zero_()      # the e2e step must write every output again
        step.e2e(hin, hout)
        sync_ok()
    finally:
        coda.set_split_k("auto")
    for k in ref:
        assert torch.equal(hout[k], ref[k]), k


def test_full_llama_block_chain_sampled():
    # One layer of the stack: the input arrives with its row sums of squares
    # (here from the library's unfused ROW_SUMSQ pass), the out-projection's
    # residual epilogue emits those of h for the MLP norm, the down-projection
    # those of y; no call runs a pre-pass over its A operand.
    # Each call is checked elementwise against the oracle of that call on the
    # bf16 tensors it actually read (the previous calls' GPU outputs); the
    # block as a whole against the oracle's own chain (every call's output
    # rounded to bf16 by the oracle) within the Frobenius bound.
    from gemm_epilogue_transformer_tmem_gb300 import workloads
    t = inputs.make_llama_block()
    td = {k: cu(v) for k, v in t.items()}
    td["X_sumsq"] = workloads.row_sumsq(td["X"])
    prepared = dict(W_qkv=coda.fold_gamma(td["W_qkv"], td["gamma_attn"], "kn"),
                    W_up=coda.fold_gamma(td["W_up"], td["gamma_mlp"], "kn"))
    before = coda.launch_count()
    out = workloads.llama_block_forward(td, prepared)
    launched = coda.launch_count() - before
    sync_ok()
    assert launched == 6, f"{launched} launches: four GEMMs and two row-sum finishing kernels expected"
    rows = _sampled(inputs.LLAMA_BLOCK["tokens"], 4)
    d, ffn = inputs.LLAMA_BLOCK["d"], inputs.LLAMA_BLOCK["ffn"]
    eps = inputs.EPS_RMS
    ref = workloads_oracle_llama(t, rows, prepared=True)
    X = f64(t["X"][rows])
    h_gpu, up_gpu = f64(out["h"][rows]), f64(out["up"][rows])
    # qkv and h read the block's own inputs
    assert_close(f64(out["qkv"][rows]), ref["qkv"], "llama qkv")
    assert_close(h_gpu, ref["h"], "llama h")
    # h is a bf16 output that later calls read.  It is computed from exact
    # inputs, and the GPU (fp32) and oracle (fp64) values agree to ~1e-6
    # relative, so their bf16 roundings are equal except where the two straddle
    # a rounding boundary: there they are neighbours, one bf16 ulp apart.  (Near
    # zero the bf16 spacing falls below fp32's absolute accumulation error over
    # K = 4096, about 4e-6, so the ulp is taken at no less than |h| = 2^-6.)
    r = O.round_bf16(ref["h"])
    diff = h_gpu != r
    assert diff.mean() < 1e-2, f"h: {diff.mean():.2e} of elements differ from the rounded oracle"
    ulp = bf16_ulp(np.maximum(np.abs(r), 2.0 ** -6))
    assert (np.abs(h_gpu - r)[diff] <= ulp[diff] * (1 + 1e-12)).all(), "h: a difference above 1 ulp"
    # up reads the GPU's h (norm statistics from h as stored; weights prepared as the block does)
    g_mlp, W_up = f64(t["gamma_mlp"]), f64(t["W_up"])
    up_call = O.run_chain(h_gpu, O.round_bf16(g_mlp[:, None] * W_up), [("RMS_ROWSCALE", None, eps), ("SWIGLU",)],
                          norm_gamma=np.ones_like(g_mlp))["D"]
    assert_close(up_gpu, up_call, "llama up (on the GPU's h)")
    # y reads the GPU's up and h
    yo = O.run_chain(up_gpu, f64(t["W_down"]), [("RESIDUAL", 0, 1.0), ("ROW_SUMSQ", 0)], residual_t=h_gpu)
    y = f64(out["y"][rows])
    assert_close(y, yo["D"], "llama y (on the GPU's up and h)")
    # the row sums of squares: the input's, and each residual call's on what it read
    assert_stat_close(f64(td["X_sumsq"][rows]), O.row_sumsq(X), 2.0 * np.sqrt(O.row_sumsq(X * X)), d, TAU_LIN, 0,
                      "llama X sum of squares")
    assert_stat_close(f64(out["h_sumsq"][rows]), ref["h_sumsq"], ref["h_sumsq_scale"], d, TAU_LIN, d,
                      "llama h sum of squares")
    assert_stat_close(f64(out["y_sumsq"][rows]), yo["stats"][0], yo["stat_scale"][0], d, TAU_LIN, ffn,
                      "llama y sum of squares")
    # the whole block against the oracle's own chain, prepared weights and
    # unprepared (gamma applied in fp64 to the activations, no bf16 weight
    # preparation): within the Frobenius bound; elementwise excess reported
    ref0 = workloads_oracle_llama(t, rows, prepared=False)
    for tag, rr in (("prepared", ref), ("unprepared", ref0)):
        for name in ("qkv", "up", "y"):
            got = f64(out[name][rows])
            fro = np.linalg.norm(got - rr[name]) / np.linalg.norm(rr[name])
            over = np.abs(got - rr[name]) > ATOL + RTOL * np.abs(rr[name])
            print(f"llama {name} against the {tag} oracle chain: {int(over.sum())} of {over.size} sampled elements "
                  f"over the elementwise bound, relative Frobenius {fro:.3e}")
            assert fro <= FRO, (tag, name)


def bf16_ulp(v):
    """Spacing of the bf16 grid at v (8 significant bits): 2^(e-8) for v = m 2^e, 0.5 <= |m| < 1."""
    return np.ldexp(1.0, np.frexp(np.asarray(v, dtype=np.float64))[1] - 8)


def workloads_oracle_llama(t, rows, prepared):
    """The block evaluated by the oracle on the given rows, unfused, in fp64.
    Each of the four calls returns bf16, so the oracle rounds each call's output
    to bf16 before the next call reads it.  With prepared=True the norm weights
    are the prepared ones, bf16(gamma (.)_row W) -- the block's documented weight
    preparation, rounded by the oracle itself -- and the norm is applied with
    unit gamma; with prepared=False gamma is applied in fp64 to the activations."""
    eps = inputs.EPS_RMS
    R = O.round_bf16
    X = f64(t["X"][rows])

    def norm_proj(A, W, g, extra):
        W, g = f64(W), f64(g)
        if prepared:
            return O.run_chain(A, R(g[:, None] * W), [("RMS_ROWSCALE", None, eps)] + extra,
                               norm_gamma=np.ones_like(g))["D"]
        return O.run_chain(A, W, [("RMS_ROWSCALE", None, eps)] + extra, norm_gamma=g)["D"]

    qkv = norm_proj(X, t["W_qkv"], t["gamma_attn"], [])
    ho = O.run_chain(f64(t["attn_out"][rows]), f64(t["W_o"]), [("RESIDUAL", 0, 1.0), ("ROW_SUMSQ", 0)], residual_t=X)
    h = ho["D"]
    up = norm_proj(R(h), t["W_up"], t["gamma_mlp"], [("SWIGLU",)])
    yo = O.run_chain(R(up), f64(t["W_down"]), [("RESIDUAL", 0, 1.0), ("ROW_SUMSQ", 0)], residual_t=R(h))
    return dict(qkv=qkv, h=h, up=up, y=yo["D"], h_sumsq=ho["stats"][0], h_sumsq_scale=ho["stat_scale"][0],
                y_sumsq=yo["stats"][0], y_sumsq_scale=yo["stat_scale"][0])
