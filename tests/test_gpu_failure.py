"""Failure detection on the GPU without a GPU fault.

Every pipeline wait in the fused kernel has a time limit.  With the limit set
to 1 ns, the first wait that is not already satisfied gives up: the kernel
records CODA_ERR_TIMEOUT (with the block, role and tile) in the device error
word, lets its in-flight copies land, frees tensor memory and returns.  The
test checks that the status reaches the host and that the context is still
usable afterwards: the same call with the default limit is correct again.
No trap, assert, bad address or endless loop is involved.
"""
import math

import numpy as np
import pytest
import torch

import __graft_entry__ as entry
from gemm_epilogue_transformer_tmem_gb300 import coda, inputs
from oracle import coda_oracle as O

pytestmark = pytest.mark.gpu

TIMEOUT = 5
ROLES = {1: "producer", 2: "mma", 3: "epilogue", 4: "row statistics", 5: "tile scheduler"}


@pytest.mark.parametrize("mode", ["single", "pair", "split", "dynamic_single", "dynamic_pair"])
def test_pipeline_wait_times_out_and_context_recovers(mode):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    entry.build()
    # the dynamic modes have more tiles than resident clusters (one cluster per
    # tile, later tiles taken over through cluster launch control)
    M, K, N = (2048, 256, 4096) if mode.startswith("dynamic") else (512, 1024, 512)
    A = inputs.randn_bf16((M, K), 1.0, 71).cuda()
    B = inputs.randn_bf16((K, N), 1.0 / math.sqrt(K), 72).cuda()
    ops = [("GELU_TANH",), ("ROW_SUM", 0)]
    st0, _ = coda.check_device_error()
    assert st0 == 0
    coda.set_cta_pair("pair" if mode.endswith("pair") else "single")
    coda.set_tile_scheduler("dynamic" if mode.startswith("dynamic") else "static")
    coda.set_split_k("force" if mode == "split" else "off")
    try:
        coda.set_pipeline_timeout_ns(1)
        coda.gemm_epilogue(A, B, ops)          # enqueued fine; the kernel gives up
        assert coda.last_plan()["dynamic"] == (1 if mode.startswith("dynamic") else 0)
        st, info = coda.check_device_error()
        assert coda.STATUS[st] == "CODA_ERR_TIMEOUT", (st, info)
        assert info[0] == TIMEOUT and info[2] in ROLES, info
        # the error word was cleared by the read
        st2, _ = coda.check_device_error()
        assert st2 == 0
    finally:
        coda.set_pipeline_timeout_ns(0)        # back to the default limit
    r = coda.gemm_epilogue(A, B, ops)
    st3, info3 = coda.check_device_error()
    coda.set_cta_pair("auto")
    coda.set_split_k("auto")
    coda.set_tile_scheduler("static")
    assert st3 == 0, info3
    ref = O.run_chain(O.to_f64(A), O.to_f64(B), ops)
    got = O.to_f64(r.D)
    assert (np.abs(got - ref["D"]) <= 1e-2 + 1e-2 * np.abs(ref["D"])).all()
