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
ROLES = {1: "producer", 2: "mma", 3: "epilogue", 4: "row statistics"}


@pytest.mark.parametrize("mode", ["single", "pair", "split"])
def test_pipeline_wait_times_out_and_context_recovers(mode):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    entry.build()
    M, K, N = 512, 1024, 512
    A = inputs.randn_bf16((M, K), 1.0, 71).cuda()
    B = inputs.randn_bf16((K, N), 1.0 / math.sqrt(K), 72).cuda()
    ops = [("GELU_TANH",), ("ROW_SUM", 0)]
    st0, _ = coda.check_device_error()
    assert st0 == 0
    coda.set_cta_pair("pair" if mode == "pair" else "single")
    coda.set_split_k("force" if mode == "split" else "off")
    try:
        coda.set_pipeline_timeout_ns(1)
        coda.gemm_epilogue(A, B, ops)          # enqueued fine; the kernel gives up
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
    assert st3 == 0, info3
    ref = O.run_chain(O.to_f64(A), O.to_f64(B), ops)
    got = O.to_f64(r.D)
    assert (np.abs(got - ref["D"]) <= 1e-2 + 1e-2 * np.abs(ref["D"])).all()
