"""coda_gemm_epilogue_noalloc: the entry point for callers that cannot allocate
device memory when they call the library (for example a serving loop that fixes
its memory footprint at start-up, since cudaMalloc can synchronise the device
and has no latency bound).  It keeps its row-reduction and keep-count partials
in the library's own fixed scratch buffer instead of a caller workspace.

Checked here through the C ABI: four calls in a row, on different problems that
all use the scratch buffer (row reductions and keep counts, column-reduction
partials with FP8 operands, then a long-K problem whose K range is split over
CTAs, with its fp32 partial accumulators and arrival counters in the buffer
over what the earlier calls left there), each against the regular entry point
(which gets a workspace from the caller).  Both run the same kernels with the
same plan, so their outputs must agree bit for bit; the first call is also
checked against the fp64 oracle within the parity tolerance of the other GPU
tests.  Finally, a problem that needs more scratch than the buffer holds is
refused.
This file is collected last so a stop-at-first-failure run has already run
every other test; it also passes when run alone.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import __graft_entry__ as entry
from gemm_epilogue_transformer_tmem_gb300 import coda, inputs

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2


def _close(got, ref, what):
    """Within the parity tolerance of the fp64 oracle (ref: numpy fp64)."""
    got = got.detach().to("cpu", torch.float64).numpy()
    bad = np.abs(got - ref) > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{what}: {bad.sum()} elements differ"


def _same(got, ref, what):
    """Bit for bit: the same kernels on the same inputs with the same plan."""
    assert torch.equal(got, ref), f"{what}: the no-alloc and regular entry points differ"


def test_noalloc_matches_regular_entry_point_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    entry.build()
    dev = "cuda"

    # call 1: dgrad form with two row reductions (partials in the scratch buffer)
    M, K, N = 300, 128, 520
    dY = inputs.randn_bf16((M, K), 1.0, 901).to(dev)
    W = inputs.randn_bf16((N, K), 1.0 / math.sqrt(K), 902).to(dev)
    Z = inputs.randn_bf16((M, N), 1.0, 903).to(dev)
    Xh = inputs.randn_bf16((M, N), 1.0, 904).to(dev)
    ops1 = [("GELU_TANH_GRAD",), ("ROW_DOT_AUX", 0), ("ROW_SUM", 1)]
    assert 0 < coda.workspace_size(M, N, K, ops1) <= coda.NOALLOC_SCRATCH_BYTES
    out1 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    st1 = torch.empty((2, M), dtype=torch.float32, device=dev)
    coda.gemm_epilogue_noalloc(dY, W, ops1, out=out1, row_stats=st1, b_layout="nk", z=Z, xhat=Xh)

    # call 2, right after: SwiGLU + dropout + a row sum on another shape, so the
    # buffer now holds call 1's partials where call 2 writes its own
    M2, K2, n_out = 257, 192, 264
    X2 = inputs.randn_bf16((M2, K2), 1.0, 905).to(dev)
    W2 = inputs.randn_bf16((K2, 2 * n_out), 1.0 / math.sqrt(K2), 906).to(dev)
    ops2 = [("SWIGLU",), ("DROPOUT", 0, 0.1), ("ROW_SUM", 0)]
    out2 = torch.empty((M2, n_out), dtype=torch.bfloat16, device=dev)
    st2 = torch.empty((1, M2), dtype=torch.float32, device=dev)
    kc2 = torch.empty((M2,), dtype=torch.int32, device=dev)
    coda.gemm_epilogue_noalloc(X2, W2, ops2, out=out2, row_stats=st2, keep_count=kc2, seed=77)
    torch.cuda.synchronize()
    st, info = coda.check_device_error()
    assert st == 0, info

    ref1 = coda.gemm_epilogue(dY, W, ops1, b_layout="nk", z=Z, xhat=Xh)
    ref2 = coda.gemm_epilogue(X2, W2, ops2, seed=77)
    torch.cuda.synchronize()
    _same(out1, ref1.D, "call 1 D")
    _same(st1, ref1.row_stats, "call 1 row stats")
    _same(out2, ref2.D, "call 2 D")
    _same(st2, ref2.row_stats, "call 2 row sum")
    _same(kc2, ref2.keep_count, "call 2 keep counts")
    # and call 1 against the oracle
    from oracle import coda_oracle as O
    f64 = O.to_f64
    oref = O.run_chain(f64(dY.cpu()), f64(W.cpu()), ops1, b_layout="nk", z=f64(Z.cpu()), xhat=f64(Xh.cpu()))
    _close(out1, oref["D"], "call 1 D against the oracle")

    # call 3: FP8 operands with a column reduction (partials in the scratch buffer)
    A8 = inputs.random_e4m3_codes((M, 256), 907)
    B8 = inputs.random_e4m3_codes((264, 256), 908)
    ops3 = [("COL_SUM", 0)]
    out3 = torch.empty((M, 264), dtype=torch.bfloat16, device=dev)
    cs3 = torch.empty((1, 264), dtype=torch.float32, device=dev)
    A8d, B8d = A8.to(dev), B8.to(dev)     # kept alive until the kernels have run
    e3 = coda.make_epilogue(ops3)
    a3 = coda.make_aux(col_stats=cs3)
    st = coda.lib().coda_gemm_epilogue_noalloc(A8d.data_ptr(), B8d.data_ptr(), M, 264, 256,
                                               coda.B_LAYOUTS["nk"] | coda.AB_E4M3, ctypes.byref(e3),
                                               ctypes.byref(a3), out3.data_ptr(), None, None,
                                               torch.cuda.current_stream().cuda_stream)
    assert st == 0
    ref3 = coda.gemm_epilogue(A8d, B8d, ops3, b_layout="nk", e4m3=True)
    torch.cuda.synchronize()
    _same(out3, ref3.D, "call 3 D")
    _same(cs3, ref3.col_stats, "call 3 column sums")

    # call 4: few tiles and a long K (2 tiles, 32 k-blocks), so the K range is
    # split over CTAs: the fp32 partial accumulators and the per-tile arrival
    # counters live in the scratch buffer too, over the bytes calls 1-3 left
    # there (the counters must be cleared by the call itself)
    M4, K4, N4 = 128, 2048, 512
    X4 = inputs.randn_bf16((M4, K4), 1.0, 909).to(dev)
    W4 = inputs.randn_bf16((K4, N4), 1.0 / math.sqrt(K4), 910).to(dev)
    ops4 = [("GELU_TANH",), ("ROW_SUM", 0)]
    out4 = torch.empty((M4, N4), dtype=torch.bfloat16, device=dev)
    st4 = torch.empty((1, M4), dtype=torch.float32, device=dev)
    coda.gemm_epilogue_noalloc(X4, W4, ops4, out=out4, row_stats=st4)
    plan4 = coda.last_plan()
    ref4 = coda.gemm_epilogue(X4, W4, ops4)
    plan4_ref = coda.last_plan()
    torch.cuda.synchronize()
    st, info = coda.check_device_error()
    assert st == 0, info
    assert plan4["split"] == 1 and plan4 == plan4_ref, (plan4, plan4_ref)
    _same(out4, ref4.D, "call 4 D (split over K)")
    _same(st4, ref4.row_stats, "call 4 row sum (split over K)")

    # a problem needing more scratch than the buffer holds is refused up front
    big_M = 70000
    need = coda.workspace_size(big_M, 8192, 64, [("ROW_SUM", 0), ("ROW_SUMSQ", 1)])
    assert need > coda.NOALLOC_SCRATCH_BYTES
    e = coda.make_epilogue([("ROW_SUM", 0), ("ROW_SUMSQ", 1)])
    a = coda.CodaAux()
    status = coda.lib().coda_gemm_epilogue_noalloc(0x1000, 0x2000, big_M, 8192, 64, 0, ctypes.byref(e),
                                                   ctypes.byref(a), 0x3000, 0x4000, None, None)
    assert coda.STATUS[status] == "CODA_ERR_WORKSPACE"
