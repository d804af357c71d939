"""CPU-side checks of the C ABI: the library builds, loads and exports every
symbol include/coda.h declares; struct layouts match; host validation rejects
bad arguments before anything reaches a device.  No kernel runs here."""
import ctypes
import os
import re

import pytest

import __graft_entry__ as entry
from gemm_epilogue_transformer_tmem_gb300 import coda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "coda.h")

OK, INVALID, UNSUPPORTED, ALIGN, CUDA, TIMEOUT, WORKSPACE = range(7)


@pytest.fixture(scope="module")
def L():
    entry.build()
    return coda.lib()


def _declared():
    src = open(HEADER).read()
    return re.findall(r"CODA_API\s+[\w\s\*]+?\b(coda_\w+)\s*\(", src)


def test_header_declares_entry_points():
    names = _declared()
    for n in ["coda_gemm_epilogue", "coda_workspace_size", "coda_fold_gamma", "coda_rmsnorm",
              "coda_epilogue_apply", "coda_check_device_error", "coda_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in _declared():
        assert hasattr(L, n), n


def test_struct_layouts():
    assert ctypes.sizeof(coda.CodaOp) == 16
    assert ctypes.sizeof(coda.CodaEpilogue) == 16 + 16 * 16
    assert ctypes.sizeof(coda.CodaAux) == 8 * (4 + 2 + 4 + 2 + 1 + 1)


def test_opcode_values_match_header():
    src = open(HEADER).read()
    for name, val in coda.OPCODES.items():
        m = re.search(r"CODA_OP_%s\s*=\s*(\d+)" % name, src)
        assert m and int(m.group(1)) == val, name


def test_status_strings(L):
    for code, name in coda.STATUS.items():
        assert L.coda_status_string(code).decode() == name


def _ws(L, M, N, K, ops):
    e = coda.make_epilogue(ops)
    n = ctypes.c_size_t(123)
    st = L.coda_workspace_size(M, N, K, ctypes.byref(e), ctypes.byref(n))
    return st, n.value


def test_workspace_size_closed_form(L):
    # one fp32 partial per (reduction, 256-column tile, row); 128-column tiles with SWIGLU;
    # one fp32 row scale per row with RMS_ROWSCALE
    assert _ws(L, 1000, 1024, 64, []) == (OK, 0)
    assert _ws(L, 1000, 1024, 64, [("ROW_SUM", 0)]) == (OK, 4 * 4 * 1000)
    assert _ws(L, 1000, 1032, 64, [("ROW_SUM", 0), ("ROW_SUMSQ", 1)]) == (OK, 2 * 5 * 4 * 1000)
    assert _ws(L, 8, 2 * 264, 64, [("SWIGLU",), ("DROPOUT", 0, 0.1)]) == (OK, 3 * 8 * 4)
    assert _ws(L, 8, 64, 64, [("RMS_ROWSCALE", 0, 1e-6)]) == (OK, 8 * 4)       # row scales [M]
    assert _ws(L, 8, 64, 64, [("RMS_ROWSCALE", 0, 1e-6), ("ROW_SUM", 1)]) == (OK, 8 * 4 + 8 * 4)


@pytest.mark.parametrize("ops,why", [
    ([("ROW_SUM", 9)], "stat slot out of range"),
    ([("SWIGLU",), ("SWIGLU",)], "two SWIGLU"),
    ([("DROPOUT", 0, 1.0)], "p = 1"),
    ([("DROPOUT", 0, -0.1)], "p < 0"),
    ([("DROPOUT", 0, 0.1), ("DROPOUT", 0, 0.1)], "two dropouts"),
    ([("ROW_SUM", 0)] * 5, "five reductions"),
    ([("RESIDUAL", 0, 1.0), ("SWIGLU",)], "residual before SWIGLU"),
    ([("SCALE", 0, float("nan"))], "nan parameter"),
    ([("RMS_ROWSCALE", 0, 1e-6), ("RMS_SUMSQ_ROWSCALE", 0, 1e-6)], "two norms"),
    ([("RMS_SUMSQ_ROWSCALE", 2, 1e-6)], "row-vector slot out of range"),
    ([("RMS_SUMSQ_ROWSCALE", 0, -1.0)], "negative eps"),
])
def test_invalid_op_lists(L, ops, why):
    st, _ = _ws(L, 64, 64, 64, ops)
    assert st == INVALID, why


def test_unknown_opcode(L):
    e = coda.make_epilogue([("SCALE", 0, 1.0)])
    e.ops[0].opcode = 77
    n = ctypes.c_size_t(0)
    assert L.coda_workspace_size(8, 8, 8, ctypes.byref(e), ctypes.byref(n)) == INVALID
    e.ops[0].opcode = 0
    e.reserved = 1
    assert L.coda_workspace_size(8, 8, 8, ctypes.byref(e), ctypes.byref(n)) == INVALID


def test_dims_validation(L):
    assert _ws(L, 64, 60, 64, [])[0] == INVALID        # N % 8
    assert _ws(L, 64, 64, 60, [])[0] == INVALID        # K % 8
    assert _ws(L, -1, 64, 64, [])[0] == INVALID
    assert _ws(L, 64, 2 * 12, 64, [("SWIGLU",)])[0] == INVALID   # N % 16 with SWIGLU
    assert _ws(L, 64, 64, 0, [("RMS_ROWSCALE", 0, 1e-6)])[0] == INVALID


def _gemm(L, A, B, M, N, K, ops=(), aux=None, D=0x1000, stats=None, ws=None, ws_bytes=0, layout=0):
    e = coda.make_epilogue(ops)
    a = aux if aux is not None else coda.CodaAux()
    return L.coda_gemm_epilogue(A, B, M, N, K, layout, ctypes.byref(e), ctypes.byref(a), D, stats, None, ws,
                                ws_bytes, None)


def test_gemm_validation_before_device(L):
    # every one of these fails in host validation, before any CUDA call
    assert _gemm(L, 0x1000, 0x2000, 64, 64, 64, layout=8) == INVALID
    assert _gemm(L, 0x1008, 0x2000, 64, 64, 64) == ALIGN
    assert _gemm(L, 0x1000, 0x2000, 64, 64, 64, D=0x1004) == ALIGN
    assert _gemm(L, None, 0x2000, 64, 64, 64) == INVALID
    assert _gemm(L, 0x1000, 0x2000, 64, 64, 64, D=None) == INVALID
    assert _gemm(L, 0x1000, 0x2000, 64, 64, 64, ops=[("BIAS", 0)]) == INVALID          # no bias vector
    assert _gemm(L, 0x1000, 0x2000, 64, 64, 64, ops=[("ROW_SUM", 0)]) == INVALID       # no row_stats
    assert _gemm(L, 0x1000, 0x2000, 64, 64, 64, ops=[("ROW_SUM", 0)], stats=0x3000) == WORKSPACE
    aux = coda.CodaAux()
    aux.residual = 0x4004
    assert _gemm(L, 0x1000, 0x2000, 64, 64, 64, ops=[("RESIDUAL", 0, 1.0)], aux=aux) == ALIGN


def test_empty_problems_enqueue_nothing(L):
    # M == 0 or N == 0: nothing to compute, nothing touched, no device needed
    before = L.coda_launch_count()
    assert _gemm(L, 0x1000, 0x2000, 0, 64, 64) == OK
    assert _gemm(L, 0x1000, 0x2000, 64, 0, 64) == OK
    assert L.coda_launch_count() == before


def test_other_entry_points_validate(L):
    assert L.coda_fold_gamma(0x1000, 0x2000, 0x3000, 64, 64, 5, None) == INVALID
    assert L.coda_fold_gamma(0x1000, 0x2004, 0x3000, 64, 64, 0, None) == ALIGN
    assert L.coda_rmsnorm(0x1000, 0x2000, 64, 60, 1e-6, 0x3000, None, None) == INVALID
    assert L.coda_rmsnorm(0x1000, 0x2000, 64, 64, -1.0, 0x3000, None, None) == INVALID
    e = coda.make_epilogue([("RMS_ROWSCALE", 0, 1e-6)])
    a = coda.CodaAux()
    assert L.coda_epilogue_apply(0x1000, 64, 64, ctypes.byref(e), ctypes.byref(a), 0x2000, 0x3000, None,
                                 None) == UNSUPPORTED


def test_binding_helpers():
    assert coda.output_width(22016, [("SWIGLU",), ("DROPOUT", 0, 0.1)]) == 11008
    assert coda.stat_slots([("RMS_ROWSCALE", 2, 1e-6), ("ROW_SUM", 0)]) == 3
    assert coda.stat_slots([("RMS_ROWSCALE", None, 1e-6)]) == 0


def test_workspace_size_for_layernorm_op_list():
    # sizing needs no aux tensors: r_i and mu_i per row for the commuted LayerNorm
    M, N, K = 300, 264, 192
    assert coda.workspace_size(M, N, K, [("LN_ROWSCALE", 0, 1e-5)]) == 2 * M * 4
    assert coda.workspace_size(M, N, K, [("LN_ROWSCALE", -1, 1e-5), ("ROW_SUM", 2)]) >= 2 * M * 4


def test_plan_struct_layout():
    assert ctypes.sizeof(coda.CodaPlan) == 40


def test_workspace_size_split_k_closed_form(L):
    # split-K part: per slot 3 partial accumulators of 256 x 128 fp32 and a u32
    # counter, after the rest rounded up to 256 bytes; one slot per tile for
    # few-tile problems, 160 (one per CTA) for problems of at least 128 tiles
    part = lambda slots: slots * (3 * 256 * 128 * 4 + 4)   # noqa: E731
    up = lambda b: (b + 255) // 256 * 256                  # noqa: E731
    # SwiGLU up-projection, 64 tiles of 128 output columns, K = 4096
    assert coda.workspace_size(128, 16384, 4096, [("RMS_ROWSCALE", -1, 1e-6), ("SWIGLU",)]) == up(128 * 4) + part(64)
    # plain GEMM, 16 tiles, K = 1024 (16 k-blocks): eligible with no other scratch
    assert coda.workspace_size(100, 4096, 1024, []) == part(16)
    # K = 960 (15 k-blocks) or between 77 and 127 tiles (the decode-sized 86): not split automatically
    assert coda.workspace_size(100, 4096, 960, []) == 0
    assert coda.workspace_size(128, 77 * 256, 4096, []) == 0
    assert coda.workspace_size(128, 22016, 4096, [("RMS_ROWSCALE", -1, 1e-6), ("SWIGLU",)]) == 128 * 4
    # 32 CTA-pair tiles: too few for the last-wave split, too many CTAs for the other
    assert coda.workspace_size(300, 4096, 4096, [("ROW_SUM", 0)]) == 16 * 300 * 4
    # 512 CTA-pair tiles (4096 x 8192): the last waves may split
    assert coda.workspace_size(4096, 8192, 2048, []) == part(160)
    assert coda.workspace_size(4096, 8192, 2048, [("ROW_SUM", 0)]) == up(32 * 4096 * 4) + part(160)
    try:
        coda.set_split_k("off")
        assert coda.workspace_size(100, 4096, 1024, []) == 0
        assert coda.workspace_size(4096, 8192, 2048, []) == 0
        coda.set_split_k("force")
        coda.set_cta_pair("single")
        # forced: any problem with two k-blocks or more (3 x 2 tiles here; room
        # for both uses, the larger being the per-CTA slots)
        assert coda.workspace_size(300, 264, 192, [("ROW_SUM", 0)]) == up(2 * 300 * 4) + part(160)
        assert coda.workspace_size(300, 264, 64, [("ROW_SUM", 0)]) == 2 * 300 * 4
    finally:
        coda.set_split_k("auto")
        coda.set_cta_pair("auto")


def test_workspace_size_column_reductions(L):
    # one fp32 partial per (column reduction, 32-row block, output column)
    M, N, K = 300, 264, 64
    assert coda.workspace_size(M, N, K, [("COL_SUM", 0)]) == 10 * N * 4
    assert coda.workspace_size(M, N, K, [("COL_SUM", 0), ("COL_DOT_AUX", 1)]) == 2 * 10 * N * 4
    # after the row-reduction partials (SwiGLU: 128-column tiles, 3 of them for 264
    # output columns); the column partials span the output width N/2
    assert coda.workspace_size(M, 2 * N, K, [("SWIGLU",), ("ROW_SUM", 0), ("COL_SUMSQ", 0)]) == \
        3 * M * 4 + 10 * N * 4


@pytest.mark.parametrize("ops,why", [
    ([("COL_SUM", 0)] * 3, "three column reductions"),
    ([("COL_SUM", 0), ("SWIGLU",)], "column reduction before SWIGLU"),
    ([("COL_SUM", 9)], "slot out of range"),
])
def test_column_reduction_lists_rejected(L, ops, why):
    st, _ = _ws(L, 300, 528, 64, ops)
    assert st == INVALID, why


def test_a_km_layout_validation(L):
    # A as [K, M] needs M a multiple of 8, and no commuted norm (row statistics read A by rows)
    assert _gemm(L, 0x1000, 0x2000, 100, 64, 64, layout=2) == INVALID
    e = coda.make_epilogue([("RMS_ROWSCALE", -1, 1e-6)])
    st = L.coda_gemm_epilogue(0x1000, 0x2000, 128, 64, 64, 2, ctypes.byref(e), None, 0x3000, None, None, None, 0,
                              None)
    assert st == UNSUPPORTED


def test_e4m3_layout_validation(L):
    # FP8 operands: B as [N, K] only, A as [M, K] only, K a multiple of 16, no commuted norm
    assert _gemm(L, 0x1000, 0x2000, 64, 64, 64, layout=4) == INVALID          # B as [K, N]
    assert _gemm(L, 0x1000, 0x2000, 64, 64, 64, layout=4 | 1 | 2) == INVALID  # A as [K, M]
    assert _gemm(L, 0x1000, 0x2000, 64, 64, 40, layout=4 | 1) == INVALID      # K % 16
    e = coda.make_epilogue([("RMS_ROWSCALE", -1, 1e-6)])
    st = L.coda_gemm_epilogue(0x1000, 0x2000, 128, 64, 64, 4 | 1, ctypes.byref(e), None, 0x3000, None, None, None,
                              0, None)
    assert st == UNSUPPORTED


def test_workspace_size_accepts_every_opcode(L):
    # sizing validates an op list without its aux tensors: every opcode is accepted
    for name in coda.OPCODES:
        ops = [(name, 0, 0.1 if name == "DROPOUT" else 1e-5)]
        if name == "SWIGLU":
            ops = [("SWIGLU",)]
        st, _ = _ws(L, 300, 528, 64, ops)
        assert st == OK, name


def test_tuning_knobs_round_trip(L):
    # the knobs are host-side settings; setting and restoring them launches nothing
    before = L.coda_launch_count()
    coda.set_tile_scheduler("dynamic")
    coda.set_tile_scheduler("static")
    coda.set_tail_helpers(False)
    coda.set_tail_helpers(True)
    coda.set_split_k("off")
    coda.set_split_k("auto")
    coda.set_raster("cols", 4)
    coda.set_raster("rows", 0)
    coda.set_raster("auto", 0)
    assert L.coda_launch_count() == before
    with pytest.raises(KeyError):
        coda.set_raster("diagonal", 1)
    with pytest.raises(ValueError):
        coda.set_tile_scheduler("round-robin")


def test_mx_scale_bytes_and_validation(L):
    # tiled scale storage: 512 bytes per 128 rows and 128 elements of K
    assert coda.mx_scale_bytes(128, 128) == 512
    assert coda.mx_scale_bytes(129, 160) == 2 * 2 * 512
    assert coda.mx_scale_bytes(0, 128) == 0
    e = coda.make_epilogue([("SWIGLU",)])
    a = coda.CodaAux()
    # SwiGLU whose U half does not start on a 128-row scale tile (N/2 = 144)
    st = L.coda_gemm_epilogue_mx(0x1000, 0x2000, 0x3000, 0x4000, 64, 288, 128, ctypes.byref(e), ctypes.byref(a),
                                 0x5000, None, None, None, 0, None)
    assert coda.STATUS[st] == "CODA_ERR_UNSUPPORTED"
    # K not a multiple of 32
    e0 = coda.make_epilogue([])
    st = L.coda_gemm_epilogue_mx(0x1000, 0x2000, 0x3000, 0x4000, 64, 256, 80, ctypes.byref(e0), ctypes.byref(a),
                                 0x5000, None, None, None, 0, None)
    assert coda.STATUS[st] == "CODA_ERR_INVALID_ARG"
    # the commuted norms read bf16 A
    en = coda.make_epilogue([("RMS_ROWSCALE", None, 1e-6)])
    st = L.coda_gemm_epilogue_mx(0x1000, 0x2000, 0x3000, 0x4000, 64, 256, 128, ctypes.byref(en), ctypes.byref(a),
                                 0x5000, None, None, None, 0, None)
    assert coda.STATUS[st] == "CODA_ERR_UNSUPPORTED"
    # missing scales
    st = L.coda_gemm_epilogue_mx(0x1000, None, 0x3000, 0x4000, 64, 256, 128, ctypes.byref(e0), ctypes.byref(a),
                                 0x5000, None, None, None, 0, None)
    assert coda.STATUS[st] == "CODA_ERR_INVALID_ARG"
    # the quantiser wants K % 32 == 0
    assert coda.STATUS[L.coda_quantize_mx_e4m3(0x1000, 4, 48, 0x2000, 0x3000, None)] == "CODA_ERR_INVALID_ARG"
