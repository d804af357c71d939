"""ctypes binding of libcoda.so, the GB300 GEMM + on-chip epilogue library.

Argument marshalling only: every computation runs in the library's CUDA
kernels.  PyTorch provides device memory (torch tensors) and the current CUDA
stream.  If the library is not built this module raises instead of falling
back to anything else.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcoda.so")

OPCODES = {
    "SCALE": 0, "COL_SCALE": 1, "BIAS": 2, "ROW_SCALE": 3, "RMS_ROWSCALE": 4, "GELU_TANH": 5,
    "SILU": 6, "SWIGLU": 7, "GELU_TANH_GRAD": 8, "DROPOUT": 9, "RESIDUAL": 10, "STORE_PREACT": 11,
    "ROW_SUM": 12, "ROW_MEAN": 13, "ROW_SUMSQ": 14, "ROW_DOT_AUX": 15, "GELU_ERF": 16, "GELU_ERF_GRAD": 17,
    "LN_ROWSCALE": 18, "COL_SUM": 19, "COL_SUMSQ": 20, "COL_DOT_AUX": 21, "COL_DOT_NORM": 22,
    "COL_SCALE_F32": 23, "RMS_SUMSQ_ROWSCALE": 24,
}
COL_REDUCTIONS = ("COL_SUM", "COL_SUMSQ", "COL_DOT_AUX", "COL_DOT_NORM")
REDUCTIONS = ("ROW_SUM", "ROW_MEAN", "ROW_SUMSQ", "ROW_DOT_AUX")
MAX_OPS = 16
NO_SLOT = 0xFFFFFFFF
B_LAYOUTS = {"kn": 0, "nk": 1}
A_KM = 2   # flag: A is given as [K, M] (the weight gradient X^T @ dY from stored X)
AB_E4M3 = 4   # flag: A [M, K] and B [N, K] are FP8 E4M3 bytes
STATUS = {0: "CODA_OK", 1: "CODA_ERR_INVALID_ARG", 2: "CODA_ERR_UNSUPPORTED", 3: "CODA_ERR_ALIGNMENT",
          4: "CODA_ERR_CUDA", 5: "CODA_ERR_TIMEOUT", 6: "CODA_ERR_WORKSPACE"}


class CodaOp(ctypes.Structure):
    _fields_ = [("opcode", ctypes.c_uint32), ("slot", ctypes.c_uint32), ("f0", ctypes.c_float),
                ("f1", ctypes.c_float)]


class CodaEpilogue(ctypes.Structure):
    _fields_ = [("n_ops", ctypes.c_uint32), ("reserved", ctypes.c_uint32), ("seed", ctypes.c_uint64),
                ("ops", CodaOp * MAX_OPS)]


class CodaAux(ctypes.Structure):
    _fields_ = [("col_vec", ctypes.c_void_p * 4), ("row_vec", ctypes.c_void_p * 2), ("residual", ctypes.c_void_p),
                ("z", ctypes.c_void_p), ("xhat", ctypes.c_void_p), ("preact_out", ctypes.c_void_p),
                ("ln_colsum", ctypes.c_void_p), ("ln_bias", ctypes.c_void_p), ("col_stats", ctypes.c_void_p),
                ("col_scale_f32", ctypes.c_void_p)]


class CodaPlan(ctypes.Structure):
    _fields_ = [("pair", ctypes.c_int32), ("split", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("tiles", ctypes.c_int64), ("prepass", ctypes.c_int32),
                ("sequence", ctypes.c_int32), ("dynamic", ctypes.c_int32), ("colvecs", ctypes.c_int32)]


class CodaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


_lib = None

_VP = ctypes.c_void_p
_I64 = ctypes.c_int64
_SIGS = {
    "coda_gemm_epilogue": (ctypes.c_int, [_VP, _VP, _I64, _I64, _I64, ctypes.c_int32, _VP, _VP, _VP, _VP, _VP,
                                          _VP, ctypes.c_size_t, _VP]),
    "coda_gemm_epilogue_noalloc": (ctypes.c_int, [_VP, _VP, _I64, _I64, _I64, ctypes.c_int32, _VP, _VP, _VP, _VP,
                                                  _VP, _VP]),
    "coda_workspace_size": (ctypes.c_int, [_I64, _I64, _I64, _VP, ctypes.POINTER(ctypes.c_size_t)]),
    "coda_fold_gamma": (ctypes.c_int, [_VP, _VP, _VP, _I64, _I64, ctypes.c_int32, _VP]),
    "coda_rmsnorm": (ctypes.c_int, [_VP, _VP, _I64, _I64, ctypes.c_float, _VP, _VP, _VP]),
    "coda_fold_layernorm": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, ctypes.c_int32, _VP]),
    "coda_layernorm": (ctypes.c_int, [_VP, _VP, _VP, _I64, _I64, ctypes.c_float, _VP, _VP]),
    "coda_norm_backward": (ctypes.c_int, [_VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _VP, _VP]),
    "coda_quantize_e4m3_rows": (ctypes.c_int, [_VP, _I64, _I64, _VP, _VP, _VP]),
    "coda_quantize_mx_e4m3": (ctypes.c_int, [_VP, _I64, _I64, _VP, _VP, _VP]),
    "coda_mx_scale_bytes": (ctypes.c_size_t, [_I64, _I64]),
    "coda_gemm_epilogue_mx": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I64, _I64, _I64, _VP, _VP, _VP, _VP, _VP, _VP,
                                             ctypes.c_size_t, _VP]),
    "coda_epilogue_apply": (ctypes.c_int, [_VP, _I64, _I64, _VP, _VP, _VP, _VP, _VP, _VP]),
    "coda_check_device_error": (ctypes.c_int, [_VP, _VP]),
    "coda_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "coda_launch_count": (ctypes.c_uint64, []),
    "coda_set_pipeline_timeout_ns": (None, [ctypes.c_uint64]),
    "coda_set_max_ctas": (None, [ctypes.c_int32]),
    "coda_set_cta_pair": (None, [ctypes.c_int32]),
    "coda_set_split_k": (None, [ctypes.c_int32]),
    "coda_set_tile_scheduler": (None, [ctypes.c_int32]),
    "coda_set_tail_helpers": (None, [ctypes.c_int32]),
    "coda_last_plan": (None, [_VP]),
    "coda_set_fixed_sequences": (None, [ctypes.c_int32]),
    "coda_set_raster": (None, [ctypes.c_int32, ctypes.c_int32]),
}


def lib() -> ctypes.CDLL:
    """Load libcoda.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(python -m gemm_epilogue_transformer_tmem_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(status: int, what: str) -> None:
    if status != 0:
        raise CodaError(status, what)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to the CUDA library must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the CUDA library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _norm_ops(ops: Sequence) -> list[tuple[str, int, float]]:
    out = []
    for o in ops:
        if isinstance(o, str):
            o = (o,)
        name = o[0]
        slot = o[1] if len(o) > 1 else 0
        f0 = o[2] if len(o) > 2 else 0.0
        if slot is None or slot < 0:
            slot = NO_SLOT
        out.append((name, int(slot), float(f0)))
    return out


def make_epilogue(ops: Sequence, seed: int = 0) -> CodaEpilogue:
    """Op list [(name, slot, f0), ...] -> the C descriptor."""
    ops = _norm_ops(ops)
    if len(ops) > MAX_OPS:
        raise ValueError("too many ops")
    e = CodaEpilogue()
    e.n_ops = len(ops)
    e.reserved = 0
    e.seed = seed & ((1 << 64) - 1)
    for i, (name, slot, f0) in enumerate(ops):
        e.ops[i].opcode = OPCODES[name]
        e.ops[i].slot = slot
        e.ops[i].f0 = f0
        e.ops[i].f1 = 0.0
    return e


def make_aux(col_vecs=None, row_vecs=None, residual=None, z=None, xhat=None, preact_out=None, ln_colsum=None,
             ln_bias=None, col_stats=None, col_scale_f32=None) -> CodaAux:
    a = CodaAux()
    a.col_stats = _ptr(col_stats)
    a.col_scale_f32 = _ptr(col_scale_f32)
    a.ln_colsum = _ptr(ln_colsum)
    a.ln_bias = _ptr(ln_bias)
    for k, t in (col_vecs or {}).items():
        a.col_vec[k] = _ptr(t)
    for k, t in (row_vecs or {}).items():
        a.row_vec[k] = _ptr(t)
    a.residual = _ptr(residual)
    a.z = _ptr(z)
    a.xhat = _ptr(xhat)
    a.preact_out = _ptr(preact_out)
    return a


def output_width(N: int, ops: Sequence) -> int:
    return _out_width(N, _norm_ops(ops))


def stat_slots(ops: Sequence) -> int:
    return _stat_slots(_norm_ops(ops))


def col_slots(ops: Sequence) -> int:
    return _col_slots(_norm_ops(ops))


# the same on an op list already normalised by _norm_ops (each call below
# normalises its list once)
def _out_width(N: int, nops: list) -> int:
    return N // 2 if any(name == "SWIGLU" for name, _, _ in nops) else N


def _stat_slots(nops: list) -> int:
    n = 0
    for name, slot, _ in nops:
        if (name in REDUCTIONS or name == "RMS_ROWSCALE") and slot != NO_SLOT:
            n = max(n, slot + 1)
        if name == "LN_ROWSCALE" and slot != NO_SLOT:
            n = max(n, slot + 2)        # r_i and mu_i
    return n


def _col_slots(nops: list) -> int:
    n = 0
    for name, slot, _ in nops:
        if name in COL_REDUCTIONS and slot != NO_SLOT:
            n = max(n, slot + 1)
    return n


def _workspace_bytes(M: int, N: int, K: int, e: CodaEpilogue) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().coda_workspace_size(M, N, K, ctypes.byref(e), ctypes.byref(n)), "coda_workspace_size")
    return n.value


def workspace_size(M: int, N: int, K: int, ops: Sequence = ()) -> int:
    return _workspace_bytes(M, N, K, make_epilogue(ops))


@dataclass
class Result:
    D: torch.Tensor
    row_stats: Optional[torch.Tensor]
    keep_count: Optional[torch.Tensor]
    col_stats: Optional[torch.Tensor] = None


def gemm_epilogue(A: torch.Tensor, B: torch.Tensor, ops: Sequence = (), *, b_layout: str = "kn", a_layout: str = "mk",
                  seed: int = 0,
                  col_vecs=None, row_vecs=None, residual=None, z=None, xhat=None, preact_out=None,
                  ln_colsum=None, ln_bias=None, col_stats: Optional[torch.Tensor] = None, col_scale_f32=None,
                  e4m3: bool = False,
                  out: Optional[torch.Tensor] = None, row_stats: Optional[torch.Tensor] = None,
                  keep_count: Optional[torch.Tensor] = None, want_keep_count: bool = True,
                  workspace: Optional[torch.Tensor] = None, stream=None) -> Result:
    """D = f(A @ B) through coda_gemm_epilogue; allocates missing outputs with torch.
    a_layout "km": A is [K, M] and the product is A^T @ B.  e4m3: A [M, K] and
    B [N, K] (b_layout "nk") are uint8 tensors of FP8 E4M3 codes."""
    if a_layout not in ("mk", "km"):
        raise ValueError(a_layout)
    M, K = A.shape if a_layout == "mk" else (A.shape[1], A.shape[0])
    N = B.shape[1] if b_layout == "kn" else B.shape[0]
    nops = _norm_ops(ops)
    n_out = _out_width(N, nops)
    dev = A.device
    if out is None:
        out = torch.empty((M, n_out), dtype=torch.bfloat16, device=dev)
    ns = _stat_slots(nops)
    if row_stats is None and ns > 0:
        row_stats = torch.empty((ns, M), dtype=torch.float32, device=dev)
    has_dropout = any(name == "DROPOUT" for name, _, _ in nops)
    if keep_count is None and has_dropout and want_keep_count:
        keep_count = torch.empty((M,), dtype=torch.int32, device=dev)
    nc = _col_slots(nops)
    if col_stats is None and nc > 0:
        col_stats = torch.empty((nc, n_out), dtype=torch.float32, device=dev)
    e = make_epilogue(nops, seed)
    if workspace is None:
        wbytes = _workspace_bytes(M, N, K, e)
        if wbytes > 0:
            workspace = torch.empty((wbytes,), dtype=torch.uint8, device=dev)
    a = make_aux(col_vecs, row_vecs, residual, z, xhat, preact_out, ln_colsum, ln_bias, col_stats, col_scale_f32)
    layout = B_LAYOUTS[b_layout] | (A_KM if a_layout == "km" else 0) | (AB_E4M3 if e4m3 else 0)
    st = lib().coda_gemm_epilogue(_ptr(A), _ptr(B), M, N, K, layout, ctypes.byref(e), ctypes.byref(a),
                                  _ptr(out), _ptr(row_stats), _ptr(keep_count), _ptr(workspace),
                                  workspace.numel() if workspace is not None else 0, _stream(stream))
    _check(st, "coda_gemm_epilogue")
    return Result(out, row_stats, keep_count, col_stats)


def mx_scale_bytes(R: int, K: int) -> int:
    """Bytes of the tiled E8M0 scale storage of an [R, K] MX operand."""
    return int(lib().coda_mx_scale_bytes(R, K))


def quantize_mx_e4m3(X: torch.Tensor, out: Optional[torch.Tensor] = None, scales: Optional[torch.Tensor] = None,
                     stream=None):
    """MXFP8 quantisation of X bf16 [R, K] (K % 32 == 0): (codes uint8 [R, K],
    scales uint8 [mx_scale_bytes(R, K)] in the library's tiled storage)."""
    R, K = X.shape
    if out is None:
        out = torch.empty((R, K), dtype=torch.uint8, device=X.device)
    if scales is None:
        scales = torch.empty((max(mx_scale_bytes(R, K), 16),), dtype=torch.uint8, device=X.device)
    _check(lib().coda_quantize_mx_e4m3(_ptr(X), R, K, _ptr(out), _ptr(scales), _stream(stream)),
           "coda_quantize_mx_e4m3")
    return out, scales


def gemm_epilogue_mx(A: torch.Tensor, scale_A: torch.Tensor, B: torch.Tensor, scale_B: torch.Tensor,
                     ops: Sequence = (), *, seed: int = 0, col_vecs=None, row_vecs=None, residual=None, z=None,
                     xhat=None, preact_out=None, col_stats: Optional[torch.Tensor] = None, col_scale_f32=None,
                     out: Optional[torch.Tensor] = None, row_stats: Optional[torch.Tensor] = None,
                     keep_count: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                     stream=None) -> Result:
    """D = f(A @ B^T) with MXFP8 operands: A uint8 E4M3 [M, K], B uint8 E4M3 [N, K],
    scale_A / scale_B their tiled E8M0 scales (coda_gemm_epilogue_mx)."""
    M, K = A.shape
    N = B.shape[0]
    nops = _norm_ops(ops)
    n_out = _out_width(N, nops)
    dev = A.device
    if out is None:
        out = torch.empty((M, n_out), dtype=torch.bfloat16, device=dev)
    ns = _stat_slots(nops)
    if row_stats is None and ns > 0:
        row_stats = torch.empty((ns, M), dtype=torch.float32, device=dev)
    if keep_count is None and any(name == "DROPOUT" for name, _, _ in nops):
        keep_count = torch.empty((M,), dtype=torch.int32, device=dev)
    nc = _col_slots(nops)
    if col_stats is None and nc > 0:
        col_stats = torch.empty((nc, n_out), dtype=torch.float32, device=dev)
    e = make_epilogue(nops, seed)
    if workspace is None:
        wbytes = _workspace_bytes(M, N, K, e)
        if wbytes > 0:
            workspace = torch.empty((wbytes,), dtype=torch.uint8, device=dev)
    a = make_aux(col_vecs, row_vecs, residual, z, xhat, preact_out, None, None, col_stats, col_scale_f32)
    st = lib().coda_gemm_epilogue_mx(_ptr(A), _ptr(scale_A), _ptr(B), _ptr(scale_B), M, N, K, ctypes.byref(e),
                                     ctypes.byref(a), _ptr(out), _ptr(row_stats), _ptr(keep_count), _ptr(workspace),
                                     workspace.numel() if workspace is not None else 0, _stream(stream))
    _check(st, "coda_gemm_epilogue_mx")
    return Result(out, row_stats, keep_count, col_stats)


def gemm_epilogue_noalloc(A: torch.Tensor, B: torch.Tensor, ops: Sequence, *, out: torch.Tensor,
                          row_stats: Optional[torch.Tensor] = None, keep_count: Optional[torch.Tensor] = None,
                          b_layout: str = "kn", seed: int = 0, col_vecs=None, row_vecs=None, residual=None, z=None,
                          xhat=None, preact_out=None, ln_colsum=None, ln_bias=None, stream=None) -> Result:
    """coda_gemm_epilogue_noalloc: the caller passes every output; the library's
    fixed scratch buffer replaces the workspace, so nothing is allocated here."""
    M, K = A.shape
    N = B.shape[1] if b_layout == "kn" else B.shape[0]
    e = make_epilogue(ops, seed)
    a = make_aux(col_vecs, row_vecs, residual, z, xhat, preact_out, ln_colsum, ln_bias)
    _check(lib().coda_gemm_epilogue_noalloc(_ptr(A), _ptr(B), M, N, K, B_LAYOUTS[b_layout], ctypes.byref(e),
                                            ctypes.byref(a), _ptr(out), _ptr(row_stats), _ptr(keep_count),
                                            _stream(stream)), "coda_gemm_epilogue_noalloc")
    return Result(out, row_stats, keep_count)


NOALLOC_SCRATCH_BYTES = 8 << 20


def fold_gamma(W: torch.Tensor, gamma: torch.Tensor, b_layout: str = "kn", out: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    """bf16(gamma (.)_row W): gamma scales W's K index (rows for [K,N], columns for [N,K])."""
    if b_layout == "kn":
        K, N = W.shape
    else:
        N, K = W.shape
    if out is None:
        out = torch.empty_like(W)
    _check(lib().coda_fold_gamma(_ptr(W), _ptr(gamma), _ptr(out), K, N, B_LAYOUTS[b_layout], _stream(stream)),
           "coda_fold_gamma")
    return out


def fold_layernorm(W: torch.Tensor, gamma: torch.Tensor, beta: Optional[torch.Tensor] = None, b_layout: str = "kn",
                   stream=None):
    """Commuted-LayerNorm weights: (bf16(gamma (.)_row W), colsum of it (fp32), beta^T W (fp32))."""
    if b_layout == "kn":
        K, N = W.shape
    else:
        N, K = W.shape
    W_out = torch.empty_like(W)
    c = torch.empty((N,), dtype=torch.float32, device=W.device)
    b = torch.empty((N,), dtype=torch.float32, device=W.device)
    _check(lib().coda_fold_layernorm(_ptr(W), _ptr(gamma), _ptr(beta), _ptr(W_out), _ptr(c), _ptr(b), K, N,
                                     B_LAYOUTS[b_layout], _stream(stream)), "coda_fold_layernorm")
    return W_out, c, b


def layernorm(X: torch.Tensor, gamma: torch.Tensor, beta: Optional[torch.Tensor], eps: float,
              out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    M, K = X.shape
    if out is None:
        out = torch.empty_like(X)
    _check(lib().coda_layernorm(_ptr(X), _ptr(gamma), _ptr(beta), M, K, eps, _ptr(out), _stream(stream)),
           "coda_layernorm")
    return out


def norm_backward(g: torch.Tensor, X: torch.Tensor, r: torch.Tensor, sum_gx: torch.Tensor,
                  mu: Optional[torch.Tensor] = None, sum_g: Optional[torch.Tensor] = None,
                  out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """dX of RMSNorm (mu = sum_g = None) or LayerNorm from g = gamma * dL/dy and its row sums."""
    M, K = g.shape
    if out is None:
        out = torch.empty_like(g)
    _check(lib().coda_norm_backward(_ptr(g), _ptr(X), _ptr(r), _ptr(mu), _ptr(sum_g), _ptr(sum_gx), M, K, _ptr(out),
                                    _stream(stream)), "coda_norm_backward")
    return out


def quantize_e4m3_rows(X: torch.Tensor, out: Optional[torch.Tensor] = None,
                       scale: Optional[torch.Tensor] = None, stream=None):
    """Per-row FP8 E4M3 quantisation: (codes uint8 [M, K], scale fp32 [M])."""
    M, K = X.shape
    if out is None:
        out = torch.empty((M, K), dtype=torch.uint8, device=X.device)
    if scale is None:
        scale = torch.empty((M,), dtype=torch.float32, device=X.device)
    _check(lib().coda_quantize_e4m3_rows(_ptr(X), M, K, _ptr(out), _ptr(scale), _stream(stream)),
           "coda_quantize_e4m3_rows")
    return out, scale


def rmsnorm(X: torch.Tensor, gamma: torch.Tensor, eps: float, out: Optional[torch.Tensor] = None,
            rstd: Optional[torch.Tensor] = None, stream=None):
    M, K = X.shape
    if out is None:
        out = torch.empty_like(X)
    if rstd is None:
        rstd = torch.empty((M,), dtype=torch.float32, device=X.device)
    _check(lib().coda_rmsnorm(_ptr(X), _ptr(gamma), M, K, eps, _ptr(out), _ptr(rstd), _stream(stream)),
           "coda_rmsnorm")
    return out, rstd


def epilogue_apply(C: torch.Tensor, ops: Sequence, *, seed: int = 0, col_vecs=None, row_vecs=None, residual=None,
                   z=None, xhat=None, preact_out=None, col_scale_f32=None, out: Optional[torch.Tensor] = None,
                   row_stats: Optional[torch.Tensor] = None, keep_count: Optional[torch.Tensor] = None,
                   stream=None) -> Result:
    """The unfused form: the op list applied to a bf16 tensor C already in memory."""
    M, N = C.shape
    n_out = output_width(N, ops)
    if out is None:
        out = torch.empty((M, n_out), dtype=torch.bfloat16, device=C.device)
    ns = stat_slots(ops)
    if row_stats is None and ns > 0:
        row_stats = torch.empty((ns, M), dtype=torch.float32, device=C.device)
    if keep_count is None and any(o[0] == "DROPOUT" for o in _norm_ops(ops)):
        keep_count = torch.empty((M,), dtype=torch.int32, device=C.device)
    e = make_epilogue(ops, seed)
    a = make_aux(col_vecs, row_vecs, residual, z, xhat, preact_out, col_scale_f32=col_scale_f32)
    _check(lib().coda_epilogue_apply(_ptr(C), M, N, ctypes.byref(e), ctypes.byref(a), _ptr(out), _ptr(row_stats),
                                     _ptr(keep_count), _stream(stream)), "coda_epilogue_apply")
    return Result(out, row_stats, keep_count)


def check_device_error(stream=None) -> tuple[int, list[int]]:
    info = (ctypes.c_uint32 * 4)()
    st = lib().coda_check_device_error(_stream(stream), info)
    return st, list(info)


def launch_count() -> int:
    return int(lib().coda_launch_count())


def set_pipeline_timeout_ns(ns: int) -> None:
    lib().coda_set_pipeline_timeout_ns(ns)


def set_max_ctas(n: int) -> None:
    lib().coda_set_max_ctas(n)


PAIR_MODES = {"auto": 0, "single": 1, "pair": 2}


def set_cta_pair(mode: str) -> None:
    """'auto' (CTA pairs when M > 128), 'single' (one-CTA kernel) or 'pair' (CTA pairs)."""
    lib().coda_set_cta_pair(PAIR_MODES[mode])


SPLIT_MODES = {"auto": 0, "off": 1, "force": 2}


def last_plan() -> dict:
    """How this thread's last gemm_epilogue call ran (kernel, split, grid, ...)."""
    pl = CodaPlan()
    lib().coda_last_plan(ctypes.byref(pl))
    return {k: getattr(pl, k) for k, _ in CodaPlan._fields_}


def set_fixed_sequences(enable: bool) -> None:
    """Use the kernels built for fixed op sequences (default) or always interpret."""
    lib().coda_set_fixed_sequences(1 if enable else 0)


def set_split_k(mode: str) -> None:
    """'auto' (split K over idle SMs for eligible problems), 'off' or 'force'."""
    lib().coda_set_split_k(SPLIT_MODES[mode])


def set_tail_helpers(enable: bool) -> None:
    """Let the non-epilogue warps share the epilogue of each CTA's last tile (default on)."""
    lib().coda_set_tail_helpers(1 if enable else 0)


RASTER_MODES = {"auto": 0, "rows": 1, "cols": 2}


def set_raster(mode: str = "auto", group: int = 0) -> None:
    """Tile order: 'rows' (groups of `group` row blocks, row fastest), 'cols'
    (groups of `group` column blocks, column fastest) or 'auto' (the library's
    choice); group <= 0 takes the library's 48 MB group."""
    lib().coda_set_raster(RASTER_MODES[mode], int(group))


def set_tile_scheduler(mode: str) -> None:
    """'static' (default: persistent round robin) or 'dynamic' (one cluster per
    tile, running clusters take over the tiles of clusters not yet started)."""
    if mode not in ("dynamic", "static"):
        raise ValueError(f"tile scheduler {mode!r}: 'dynamic' or 'static'")
    lib().coda_set_tile_scheduler(1 if mode == "dynamic" else 0)
