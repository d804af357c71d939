"""The GEMM+epilogue workloads as library calls: the fused step, the same chain
unfused (the library's own GEMM with no epilogue, then one separate
memory-bound kernel per step), and their algorithmic DRAM bytes.

Shapes and distributions come from `inputs`; every call here goes through the
C ABI (coda.py).  The commuted-RMSNorm weights are folded once (gamma (.)_row W)
when a step is built: the fold is weight preparation, like a layout change of
a static weight, and it is timed separately, not inside the step.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, Optional

import torch

from . import coda, inputs

BF16 = 2
F32 = 4


@dataclass
class Step:
    name: str
    flops: int
    fused_bytes: int          # algorithmic DRAM bytes of the fused step
    unfused_bytes: int        # algorithmic DRAM bytes of the unfused chain
    fused: Callable[[], None]
    unfused: Callable[[], None]
    host_inputs: dict = field(default_factory=dict)    # name -> device tensor fed per step in e2e mode
    host_outputs: dict = field(default_factory=dict)   # name -> device tensor read back per step
    bound: str = "tensor"     # what bounds the fused kernel: "tensor" or "hbm"
    peak_scale: float = 1.0   # tensor peak relative to bf16 (2 for FP8 operands)
    kernels_per_fused: int = 1
    kernels_per_unfused: int = 1
    prep: Optional[Callable[[], None]] = None           # weight preparation (gamma fold)
    outputs: dict = field(default_factory=dict)
    # the step's GEMMs alone (no epilogue) through torch.matmul, i.e. the vendor
    # library (cuBLAS), on the same operands: a measured reference point for the
    # GEMM core, not part of the step
    library: Optional[Callable[[], None]] = None
    # the fused step as its separate calls, (name, call, GEMM flops), when it has
    # more than one: the bench times each call with its own events, so that the
    # roofline of the dominant call is measured on that call alone
    parts: Optional[list] = None
    parts_bytes: dict = field(default_factory=dict)    # name -> algorithmic DRAM bytes of that call
    # the unfused chain with the vendor library's GEMM (torch.matmul, cuBLAS) in
    # place of the library's own, the other steps the same separate kernels
    unfused_library: Optional[Callable[[], None]] = None
    # end to end with host buffers: (h_in, h_out) -> None runs one step copying
    # h_in[name] into host_inputs[name] first and host_outputs[name] into
    # h_out[name] last; a step may overlap those copies with its own calls
    # (side streams, ordered by events).  None: copy in, step, copy out.
    e2e: Optional[Callable[[dict, dict], None]] = None


def _ws(M, N, K, ops, dev):
    n = coda.workspace_size(M, N, K, ops)
    return torch.empty((max(n, 16),), dtype=torch.uint8, device=dev), n


def build_rmsproj(dev="cuda", seed=0, M=4096, K=2048, N=8192, t=None) -> Step:
    """D = rsqrt(mean(X^2)+eps) * (X @ (gamma (.) W)), commuted, with r_i written out."""
    t = t or inputs.make_rmsproj(seed, M, K, N)
    X, g, W = (t[k].to(dev) for k in ("X", "gamma", "W"))
    Wf = torch.empty_like(W)
    prep = lambda: coda.fold_gamma(W, g, "kn", out=Wf)   # noqa: E731
    prep()
    ops = [("RMS_ROWSCALE", 0, inputs.EPS_RMS)]
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    rs = torch.empty((1, M), dtype=torch.float32, device=dev)
    ws, _ = _ws(M, N, K, ops, dev)
    Xn = torch.empty_like(X)
    rstd = torch.empty((M,), dtype=torch.float32, device=dev)
    Du = torch.empty_like(D)

    def fused():
        coda.gemm_epilogue(X, Wf, ops, out=D, row_stats=rs, workspace=ws)

    def unfused():
        coda.rmsnorm(X, g, inputs.EPS_RMS, out=Xn, rstd=rstd)
        coda.gemm_epilogue(Xn, W, [], out=Du)

    Cl = torch.empty_like(D)
    library = lambda: torch.matmul(X, Wf, out=Cl)   # noqa: E731

    def unfused_library():
        coda.rmsnorm(X, g, inputs.EPS_RMS, out=Xn, rstd=rstd)
        torch.matmul(Xn, W, out=Du)

    fb = M * K * BF16 + K * N * BF16 + M * N * BF16 + M * F32
    ub = (M * K * BF16 + K * BF16 + M * K * BF16 + M * F32) + (M * K * BF16 + K * N * BF16 + M * N * BF16)
    return Step("rmsproj", 2 * M * N * K, fb, ub, fused, unfused, host_inputs=dict(X=X),
                host_outputs=dict(D=D, r=rs), kernels_per_fused=1, kernels_per_unfused=2, prep=prep,
                outputs=dict(D=D, r=rs, D_unfused=Du, Xn=Xn), library=library, unfused_library=unfused_library)


def build_lnproj(dev="cuda", seed=0, M=4096, K=2048, N=8192, t=None) -> Step:
    """D = r (X @ Wf - mu colsum(Wf)) + beta@W, Wf = gamma (.) W: commuted LayerNorm
    projection, with r_i and mu_i written out.  The fold (Wf, its column sums
    and beta@W) is weight preparation."""
    t = t or inputs.make_lnproj(seed, M, K, N)
    X, g, beta, W = (t[k].to(dev) for k in ("X", "gamma", "beta", "W"))
    prepared = {}

    def prep():
        prepared["Wf"], prepared["c"], prepared["b"] = coda.fold_layernorm(W, g, beta, "kn")

    prep()
    ops = [("LN_ROWSCALE", 0, inputs.EPS_LN)]
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    rs = torch.empty((2, M), dtype=torch.float32, device=dev)
    ws, _ = _ws(M, N, K, ops, dev)
    Xn = torch.empty_like(X)
    Du = torch.empty_like(D)

    def fused():
        coda.gemm_epilogue(X, prepared["Wf"], ops, ln_colsum=prepared["c"], ln_bias=prepared["b"], out=D,
                           row_stats=rs, workspace=ws)

    def unfused():
        coda.layernorm(X, g, beta, inputs.EPS_LN, out=Xn)
        coda.gemm_epilogue(Xn, W, [], out=Du)

    Cl = torch.empty_like(D)
    library = lambda: torch.matmul(X, prepared["Wf"], out=Cl)   # noqa: E731

    def unfused_library():
        coda.layernorm(X, g, beta, inputs.EPS_LN, out=Xn)
        torch.matmul(Xn, W, out=Du)

    fb = M * K * BF16 + K * N * BF16 + 2 * N * F32 + M * N * BF16 + 2 * M * F32
    ub = (M * K * BF16 + 2 * K * BF16 + M * K * BF16) + (M * K * BF16 + K * N * BF16 + M * N * BF16)
    return Step("lnproj", 2 * M * N * K, fb, ub, fused, unfused, host_inputs=dict(X=X),
                host_outputs=dict(D=D, stats=rs), kernels_per_fused=1, kernels_per_unfused=2, prep=prep,
                outputs=dict(D=D, stats=rs, D_unfused=Du, Xn=Xn), library=library,
                unfused_library=unfused_library)


def build_swiglu(dev="cuda", seed=0, M=8192, K=4096, N_out=11008, t=None) -> Step:
    """out = dropout(silu(G) * U, p), [G|U] = X @ W."""
    t = t or inputs.make_swiglu(seed, M, K, N_out)
    X, W = t["X"].to(dev), t["W"].to(dev)
    N = 2 * N_out
    ops = [("SWIGLU",), ("DROPOUT", 0, inputs.DROPOUT_P)]
    D = torch.empty((M, N_out), dtype=torch.bfloat16, device=dev)
    kc = torch.empty((M,), dtype=torch.int32, device=dev)
    ws, _ = _ws(M, N, K, ops, dev)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    H = torch.empty((M, N_out), dtype=torch.bfloat16, device=dev)
    Du = torch.empty_like(D)
    kcu = torch.empty_like(kc)

    def fused():
        coda.gemm_epilogue(X, W, ops, seed=inputs.DROPOUT_SEED, out=D, keep_count=kc, workspace=ws)

    def unfused():
        coda.gemm_epilogue(X, W, [], out=C)
        coda.epilogue_apply(C, [("SWIGLU",)], out=H)
        coda.epilogue_apply(H, [("DROPOUT", 0, inputs.DROPOUT_P)], seed=inputs.DROPOUT_SEED, out=Du, keep_count=kcu)

    library = lambda: torch.matmul(X, W, out=C)   # noqa: E731

    def unfused_library():
        torch.matmul(X, W, out=C)
        coda.epilogue_apply(C, [("SWIGLU",)], out=H)
        coda.epilogue_apply(H, [("DROPOUT", 0, inputs.DROPOUT_P)], seed=inputs.DROPOUT_SEED, out=Du, keep_count=kcu)

    fb = M * K * BF16 + K * N * BF16 + M * N_out * BF16 + M * 4
    ub = (M * K + K * N + M * N) * BF16 + (M * N + M * N_out) * BF16 + (2 * M * N_out * BF16 + M * 4)
    return Step("swiglu", 2 * M * N * K, fb, ub, fused, unfused, host_inputs=dict(X=X), host_outputs=dict(D=D),
                kernels_per_fused=2, kernels_per_unfused=3, outputs=dict(D=D, keep=kc, D_unfused=Du),
                library=library, unfused_library=unfused_library)


def build_skinny(dev="cuda", seed=0, M=128, K=4096, N_out=11008, t=None) -> Step:
    """up = silu(r G) * (r U), [G|U] = X @ (gamma (.) W): commuted RMSNorm into the
    SwiGLU up-projection at a decode-sized batch.  The 180 MB weight stream
    bounds it, so its roofline is HBM bandwidth.  As in the LLaMA block, X is
    the hidden state the out-projection's residual epilogue wrote, and it
    arrives with its row sums of squares (that epilogue's ROW_SUMSQ), so the
    norm needs no pass over X."""
    t = t or inputs.make_skinny(seed, M, K, N_out)
    X, g, W = (t[k].to(dev) for k in ("X", "gamma", "W"))
    x_ss = row_sumsq(X)
    N = 2 * N_out
    Wf = torch.empty_like(W)
    prep = lambda: coda.fold_gamma(W, g, "kn", out=Wf)   # noqa: E731
    prep()
    ops = [("RMS_SUMSQ_ROWSCALE", 0, inputs.EPS_RMS), ("SWIGLU",)]
    D = torch.empty((M, N_out), dtype=torch.bfloat16, device=dev)
    ws, _ = _ws(M, N, K, ops, dev)
    Xn = torch.empty_like(X)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    Du = torch.empty_like(D)

    def fused():
        coda.gemm_epilogue(X, Wf, ops, row_vecs={0: x_ss}, out=D, workspace=ws)

    def unfused():
        coda.rmsnorm(X, g, inputs.EPS_RMS, out=Xn)
        coda.gemm_epilogue(Xn, W, [], out=C)
        coda.epilogue_apply(C, [("SWIGLU",)], out=Du)

    library = lambda: torch.matmul(X, Wf, out=C)   # noqa: E731

    def unfused_library():
        coda.rmsnorm(X, g, inputs.EPS_RMS, out=Xn)
        torch.matmul(Xn, W, out=C)
        coda.epilogue_apply(C, [("SWIGLU",)], out=Du)

    fb = M * K * BF16 + M * F32 + K * N * BF16 + M * N_out * BF16
    ub = (2 * M * K * BF16 + K * BF16) + (M * K + K * N + M * N) * BF16 + (M * N + M * N_out) * BF16
    return Step("skinny", 2 * M * N * K, fb, ub, fused, unfused, host_inputs=dict(X=X, X_sumsq=x_ss),
                host_outputs=dict(D=D),
                bound="hbm", kernels_per_fused=1, kernels_per_unfused=3, prep=prep,
                outputs=dict(D=D, D_unfused=Du), library=library, unfused_library=unfused_library)


def build_fp8swiglu(dev="cuda", seed=0, M=8192, K=4096, N_out=11008, t=None) -> Step:
    """The swiglu up-projection with FP8 E4M3 operands: X quantised per row in
    the step, W ([N, K], output channels as rows) quantised per row once;
    out = SiLU(G) * U of s_x (.)_row (X8 W8^T) (.)_col s_w."""
    t = t or inputs.make_swiglu(seed, M, K, N_out)
    X = t["X"].to(dev)
    W = t["W"].to(dev).t().contiguous()          # [2*N_out, K]
    N = 2 * N_out
    w8 = torch.empty((N, K), dtype=torch.uint8, device=dev)
    sw = torch.empty((N,), dtype=torch.float32, device=dev)
    prep = lambda: coda.quantize_e4m3_rows(W, out=w8, scale=sw)   # noqa: E731
    prep()
    x8 = torch.empty((M, K), dtype=torch.uint8, device=dev)
    sx = torch.empty((M,), dtype=torch.float32, device=dev)
    ops = [("ROW_SCALE", 0), ("COL_SCALE_F32",), ("SWIGLU",)]
    D = torch.empty((M, N_out), dtype=torch.bfloat16, device=dev)
    ws, _ = _ws(M, N, K, ops, dev)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    Du = torch.empty_like(D)

    def fused():
        coda.quantize_e4m3_rows(X, out=x8, scale=sx)
        coda.gemm_epilogue(x8, w8, ops, b_layout="nk", e4m3=True, row_vecs={0: sx}, col_scale_f32=sw, out=D,
                           workspace=ws)

    def unfused():
        coda.quantize_e4m3_rows(X, out=x8, scale=sx)
        coda.gemm_epilogue(x8, w8, [], b_layout="nk", e4m3=True, out=C)
        coda.epilogue_apply(C, ops, row_vecs={0: sx}, col_scale_f32=sw, out=Du)

    q = M * K * BF16 + M * K + M * F32
    fb = q + (M * K + N * K) + (M + N) * F32 + M * N_out * BF16
    ub = q + (M * K + N * K) + M * N * BF16 + (M * N * BF16 + (M + N) * F32 + M * N_out * BF16)
    return Step("fp8swiglu", 2 * M * N * K, fb, ub, fused, unfused, host_inputs=dict(X=X), host_outputs=dict(D=D),
                peak_scale=2.0, kernels_per_fused=2, kernels_per_unfused=3, prep=prep, outputs=dict(D=D, D_unfused=Du))


def build_mxfp8swiglu(dev="cuda", seed=0, M=8192, K=4096, N_out=11008, t=None) -> Step:
    """The swiglu up-projection with MXFP8 operands (OCP MX: E4M3 codes, one
    E8M0 scale per 32 elements of K, applied by the tensor cores): X quantised
    in the step, W ([N, K]) once; out = SiLU(G) * U."""
    t = t or inputs.make_swiglu(seed, M, K, N_out)
    X = t["X"].to(dev)
    W = t["W"].to(dev).t().contiguous()          # [2*N_out, K]
    N = 2 * N_out
    w8 = torch.empty((N, K), dtype=torch.uint8, device=dev)
    sw = torch.empty((coda.mx_scale_bytes(N, K),), dtype=torch.uint8, device=dev)
    prep = lambda: coda.quantize_mx_e4m3(W, out=w8, scales=sw)   # noqa: E731
    prep()
    x8 = torch.empty((M, K), dtype=torch.uint8, device=dev)
    sx = torch.empty((coda.mx_scale_bytes(M, K),), dtype=torch.uint8, device=dev)
    ops = [("SWIGLU",)]
    D = torch.empty((M, N_out), dtype=torch.bfloat16, device=dev)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    Du = torch.empty_like(D)

    def fused():
        coda.quantize_mx_e4m3(X, out=x8, scales=sx)
        coda.gemm_epilogue_mx(x8, sx, w8, sw, ops, out=D)

    def unfused():
        coda.quantize_mx_e4m3(X, out=x8, scales=sx)
        coda.gemm_epilogue_mx(x8, sx, w8, sw, [], out=C)
        coda.epilogue_apply(C, ops, out=Du)

    sbytes = coda.mx_scale_bytes(M, K) + coda.mx_scale_bytes(N, K)
    q = M * K * BF16 + M * K + coda.mx_scale_bytes(M, K)
    fb = q + (M * K + N * K) + sbytes + M * N_out * BF16
    ub = q + (M * K + N * K) + sbytes + M * N * BF16 + (M * N * BF16 + M * N_out * BF16)
    return Step("mxfp8swiglu", 2 * M * N * K, fb, ub, fused, unfused, host_inputs=dict(X=X), host_outputs=dict(D=D),
                peak_scale=2.0, kernels_per_fused=2, kernels_per_unfused=3, prep=prep, outputs=dict(D=D, D_unfused=Du))


def build_wgrad(dev="cuda", seed=0, T=16384, d=4096, ffn=11008, t=None) -> Step:
    """dW = s * up^T @ dY + dW (in place), per-row sums of squares of the new dW:
    the down-projection's weight gradient, A read as [K, M] (the stored
    activations, tokens x features)."""
    t = t or inputs.make_wgrad(seed, T, d, ffn)
    up, dY, dW0 = (t[k].to(dev) for k in ("up", "dY", "dW_old"))
    ops = [("SCALE", 0, inputs.WGRAD_SCALE), ("RESIDUAL", 0, 1.0), ("ROW_SUMSQ", 0)]
    dW = dW0.clone()
    rs = torch.empty((1, ffn), dtype=torch.float32, device=dev)
    ws, _ = _ws(ffn, d, T, ops, dev)
    C = torch.empty((ffn, d), dtype=torch.bfloat16, device=dev)
    dWu = dW0.clone()
    rsu = torch.empty_like(rs)

    def fused():
        coda.gemm_epilogue(up, dY, ops, a_layout="km", residual=dW, out=dW, row_stats=rs, workspace=ws)

    def unfused():
        coda.gemm_epilogue(up, dY, [], a_layout="km", out=C)
        coda.epilogue_apply(C, ops, residual=dWu, out=dWu, row_stats=rsu)

    library = lambda: torch.matmul(up.t(), dY, out=C)   # noqa: E731

    def unfused_library():
        torch.matmul(up.t(), dY, out=C)
        coda.epilogue_apply(C, ops, residual=dWu, out=dWu, row_stats=rsu)

    fb = (T * ffn + T * d + 2 * ffn * d) * BF16 + ffn * F32
    ub = (T * ffn + T * d + ffn * d) * BF16 + (3 * ffn * d * BF16 + ffn * F32)
    return Step("wgrad", 2 * ffn * d * T, fb, ub, fused, unfused, host_inputs=dict(dY=dY),
                host_outputs=dict(norms=rs), kernels_per_fused=2, kernels_per_unfused=3,
                outputs=dict(dW=dW, norms=rs), library=library, unfused_library=unfused_library)


def build_dgrad(dev="cuda", seed=0, M=8192, K=4096, N=16384, t=None) -> Step:
    """dX = (dY @ W^T) * GELU'(Z), sum_j dX*Xhat and sum_j dX per row."""
    t = t or inputs.make_dgrad(seed, M, K, N)
    dY, W, Z, Xh = (t[k].to(dev) for k in ("dY", "W", "Z", "Xhat"))
    ops = [("GELU_TANH_GRAD",), ("ROW_DOT_AUX", 0), ("ROW_SUM", 1)]
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    rs = torch.empty((2, M), dtype=torch.float32, device=dev)
    ws, _ = _ws(M, N, K, ops, dev)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    Du = torch.empty_like(D)
    rsu = torch.empty_like(rs)
    Dz = torch.empty_like(D)

    def fused():
        coda.gemm_epilogue(dY, W, ops, b_layout="nk", z=Z, xhat=Xh, out=D, row_stats=rs, workspace=ws)

    def unfused():
        coda.gemm_epilogue(dY, W, [], b_layout="nk", out=C)
        coda.epilogue_apply(C, [("GELU_TANH_GRAD",)], z=Z, out=Du)
        coda.epilogue_apply(Du, [("ROW_DOT_AUX", 0), ("ROW_SUM", 1)], xhat=Xh, out=Dz, row_stats=rsu)

    library = lambda: torch.matmul(dY, W.t(), out=C)   # noqa: E731

    def unfused_library():
        torch.matmul(dY, W.t(), out=C)
        coda.epilogue_apply(C, [("GELU_TANH_GRAD",)], z=Z, out=Du)
        coda.epilogue_apply(Du, [("ROW_DOT_AUX", 0), ("ROW_SUM", 1)], xhat=Xh, out=Dz, row_stats=rsu)

    fb = (M * K + N * K + 3 * M * N) * BF16 + 2 * M * F32
    ub = (M * K + N * K + M * N) * BF16 + 3 * M * N * BF16 + (2 * M * N * BF16 + 2 * M * F32)
    return Step("dgrad", 2 * M * N * K, fb, ub, fused, unfused, host_inputs=dict(dY=dY),
                host_outputs=dict(D=D, stats=rs), kernels_per_fused=2, kernels_per_unfused=3,
                outputs=dict(D=D, stats=rs, D_unfused=Du, stats_unfused=rsu), library=library,
                unfused_library=unfused_library)


E2E_CHUNKS = 8   # token blocks of the LLaMA block's end-to-end step (copies overlapped with calls)


def llama_block_calls(t: dict, prepared: dict, out: dict, rows: Optional[slice] = None) -> list:
    """The LLaMA-like non-attention block's four fused calls, in order, as
    closures over `out` (preallocated outputs, filled in when missing), as one
    layer of a stack whose hidden states carry their row sums of squares:
      qkv = rmsnorm(X; g_attn) @ W_qkv          commuted RMSNorm, r from sum_k X^2
      h   = attn_out @ W_o + X,  sum_j h^2      residual; the MLP norm's statistics
      up  = silu(G) * U, [G|U] = rmsnorm(h; g_mlp) @ W_up   commuted, r from sum_j h^2
      y   = up @ W_down + h,     sum_j y^2      residual; the next layer's statistics
    t["X_sumsq"] (fp32 [tokens]) holds sum_k X^2 as the previous layer's
    down-projection emits it; without it the qkv call gathers r itself (a
    pre-pass over X).  attn_out stands in for the attention output (attention
    is not part of this path).  prepared: W_qkv and W_up with gamma folded in.
    rows: the calls on these token rows only (every step is row-wise, so a block
    of rows is a block of the same computation); `out` must then be allocated."""
    eps = inputs.EPS_RMS
    ws = out.get("ws", {})
    sl = rows if rows is not None else slice(None)

    def rs(key):      # [1, tokens] row statistics, restricted to the rows
        v = out.get(key)
        return None if v is None else v[:, sl]

    def qkv():
        x_ss = t.get("X_sumsq")
        q_out = out.get("qkv")
        q_out = None if q_out is None else q_out[sl]
        if x_ss is None:
            r = coda.gemm_epilogue(t["X"][sl], prepared["W_qkv"], [("RMS_ROWSCALE", None, eps)], out=q_out)
        else:
            r = coda.gemm_epilogue(t["X"][sl], prepared["W_qkv"], [("RMS_SUMSQ_ROWSCALE", 0, eps)],
                                   row_vecs={0: x_ss[sl]}, out=q_out)
        if rows is None:
            out["qkv"] = r.D

    def oproj():
        h = out.get("h")
        r = coda.gemm_epilogue(t["attn_out"][sl], t["W_o"], [("RESIDUAL", 0, 1.0), ("ROW_SUMSQ", 0)],
                               residual=t["X"][sl], out=None if h is None else h[sl], row_stats=rs("h_sumsq"),
                               workspace=ws.get("h"))
        if rows is None:
            out["h"], out["h_sumsq"] = r.D, r.row_stats

    def up():
        u = out.get("up")
        r = coda.gemm_epilogue(out["h"][sl], prepared["W_up"], [("RMS_SUMSQ_ROWSCALE", 0, eps), ("SWIGLU",)],
                               row_vecs={0: out["h_sumsq"][0][sl]}, out=None if u is None else u[sl])
        if rows is None:
            out["up"] = r.D

    def down():
        y = out.get("y")
        r = coda.gemm_epilogue(out["up"][sl], t["W_down"], [("RESIDUAL", 0, 1.0), ("ROW_SUMSQ", 0)],
                               residual=out["h"][sl], out=None if y is None else y[sl], row_stats=rs("y_sumsq"),
                               workspace=ws.get("y"))
        if rows is None:
            out["y"], out["y_sumsq"] = r.D, r.row_stats

    return [("qkv", qkv), ("out", oproj), ("up", up), ("down", down)]


def llama_block_forward(t: dict, prepared: Optional[dict] = None, out: Optional[dict] = None) -> dict:
    """The block's four calls (see llama_block_calls) run in order; returns the
    outputs qkv, h, up, y and the row sums of squares h_sumsq, y_sumsq."""
    if prepared is None:
        prepared = dict(W_qkv=coda.fold_gamma(t["W_qkv"], t["gamma_attn"], "kn"),
                        W_up=coda.fold_gamma(t["W_up"], t["gamma_mlp"], "kn"))
    out = {} if out is None else out
    for _, call in llama_block_calls(t, prepared, out):
        call()
    return dict(qkv=out["qkv"], h=out["h"], up=out["up"], y=out["y"], h_sumsq=out["h_sumsq"][0],
                y_sumsq=out["y_sumsq"][0])


def row_sumsq(X: torch.Tensor) -> torch.Tensor:
    """sum_k X[i,k]^2 (fp32 [M]) of a bf16 matrix, through the library's unfused
    epilogue kernel: the statistics a residual epilogue's ROW_SUMSQ would have
    produced with X (used to seed a block's input)."""
    return coda.epilogue_apply(X, [("ROW_SUMSQ", 0)]).row_stats[0].contiguous()


def build_llama(dev="cuda", seed=0, tokens=16384, d=4096, ffn=11008, t=None) -> Step:
    t = t or inputs.make_llama_block(seed, tokens, d, ffn)
    t = {k: v.to(dev) for k, v in t.items()}
    # the block's input arrives with its row sums of squares (one layer of a stack)
    t["X_sumsq"] = row_sumsq(t["X"])
    prepared = {}

    def prep():
        prepared["W_qkv"] = coda.fold_gamma(t["W_qkv"], t["gamma_attn"], "kn", out=prepared.get("W_qkv"))
        prepared["W_up"] = coda.fold_gamma(t["W_up"], t["gamma_mlp"], "kn", out=prepared.get("W_up"))

    prep()
    T = tokens
    res_ops = [("RESIDUAL", 0, 1.0), ("ROW_SUMSQ", 0)]
    out = dict(qkv=torch.empty((T, 3 * d), dtype=torch.bfloat16, device=dev),
               h=torch.empty((T, d), dtype=torch.bfloat16, device=dev),
               up=torch.empty((T, ffn), dtype=torch.bfloat16, device=dev),
               y=torch.empty((T, d), dtype=torch.bfloat16, device=dev),
               h_sumsq=torch.empty((1, T), dtype=torch.float32, device=dev),
               y_sumsq=torch.empty((1, T), dtype=torch.float32, device=dev),
               ws=dict(h=_ws(T, d, d, res_ops, dev)[0], y=_ws(T, d, ffn, res_ops, dev)[0]))
    un = dict(xn=torch.empty((T, d), dtype=torch.bfloat16, device=dev),
              qkv=torch.empty((T, 3 * d), dtype=torch.bfloat16, device=dev),
              c_o=torch.empty((T, d), dtype=torch.bfloat16, device=dev),
              h=torch.empty((T, d), dtype=torch.bfloat16, device=dev),
              hn=torch.empty((T, d), dtype=torch.bfloat16, device=dev),
              c_up=torch.empty((T, 2 * ffn), dtype=torch.bfloat16, device=dev),
              up=torch.empty((T, ffn), dtype=torch.bfloat16, device=dev),
              c_down=torch.empty((T, d), dtype=torch.bfloat16, device=dev),
              y=torch.empty((T, d), dtype=torch.bfloat16, device=dev))

    calls = llama_block_calls(t, prepared, out)

    def fused():
        for _, call in calls:
            call()

    def unfused():
        eps = inputs.EPS_RMS
        coda.rmsnorm(t["X"], t["gamma_attn"], eps, out=un["xn"])
        coda.gemm_epilogue(un["xn"], t["W_qkv"], [], out=un["qkv"])
        coda.gemm_epilogue(t["attn_out"], t["W_o"], [], out=un["c_o"])
        coda.epilogue_apply(un["c_o"], [("RESIDUAL", 0, 1.0)], residual=t["X"], out=un["h"])
        coda.rmsnorm(un["h"], t["gamma_mlp"], eps, out=un["hn"])
        coda.gemm_epilogue(un["hn"], t["W_up"], [], out=un["c_up"])
        coda.epilogue_apply(un["c_up"], [("SWIGLU",)], out=un["up"])
        coda.gemm_epilogue(un["up"], t["W_down"], [], out=un["c_down"])
        coda.epilogue_apply(un["c_down"], [("RESIDUAL", 0, 1.0)], residual=un["h"], out=un["y"])

    part_flops = dict(qkv=2 * T * d * (3 * d), out=2 * T * d * d, up=2 * T * d * (2 * ffn), down=2 * T * ffn * d)
    flops = sum(part_flops.values())
    act = T * d * BF16
    rowvec = T * F32

    # end to end: the inputs' host-to-device copies and the outputs' read-back
    # overlapped with the block's calls.  Every step of the block is row-wise,
    # so the tokens go through in E2E_CHUNKS blocks of rows: block i's inputs
    # are copied in on one side stream while block i-1 runs, and its outputs
    # read back on another while block i+1 runs; events order them, so only the
    # first block's copy-in and the last block's read-back are exposed.
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    nchunk = E2E_CHUNKS if T % E2E_CHUNKS == 0 else 1
    blocks = [slice(i * (T // nchunk), (i + 1) * (T // nchunk)) for i in range(nchunk)]
    block_calls = [llama_block_calls(t, prepared, out, rows=b) for b in blocks]

    def e2e(h_in, h_out):
        main = torch.cuda.current_stream(dev)
        s_in.wait_stream(main)          # the previous step has read its inputs
        s_out.wait_stream(main)
        arrived = []
        with torch.cuda.stream(s_in):
            for b in blocks:
                t["X"][b].copy_(h_in["X"][b], non_blocking=True)
                t["X_sumsq"][b].copy_(h_in["X_sumsq"][b], non_blocking=True)
                t["attn_out"][b].copy_(h_in["attn_out"][b], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(s_in)
                arrived.append(ev)
        for b, calls_b, ev in zip(blocks, block_calls, arrived):
            main.wait_event(ev)
            for _, call in calls_b:
                call()
            done = torch.cuda.Event()
            done.record(main)
            s_out.wait_event(done)
            with torch.cuda.stream(s_out):
                h_out["qkv"][b].copy_(out["qkv"][b], non_blocking=True)
                h_out["y"][b].copy_(out["y"][b], non_blocking=True)
                h_out["y_sumsq"][:, b].copy_(out["y_sumsq"][:, b], non_blocking=True)
        main.wait_stream(s_out)
        main.wait_stream(s_in)

    def unfused_library():
        eps = inputs.EPS_RMS
        coda.rmsnorm(t["X"], t["gamma_attn"], eps, out=un["xn"])
        torch.matmul(un["xn"], t["W_qkv"], out=un["qkv"])
        torch.matmul(t["attn_out"], t["W_o"], out=un["c_o"])
        coda.epilogue_apply(un["c_o"], [("RESIDUAL", 0, 1.0)], residual=t["X"], out=un["h"])
        coda.rmsnorm(un["h"], t["gamma_mlp"], eps, out=un["hn"])
        torch.matmul(un["hn"], t["W_up"], out=un["c_up"])
        coda.epilogue_apply(un["c_up"], [("SWIGLU",)], out=un["up"])
        torch.matmul(un["up"], t["W_down"], out=un["c_down"])
        coda.epilogue_apply(un["c_down"], [("RESIDUAL", 0, 1.0)], residual=un["h"], out=un["y"])

    def library():
        torch.matmul(t["X"], prepared["W_qkv"], out=un["qkv"])
        torch.matmul(t["attn_out"], t["W_o"], out=un["c_o"])
        torch.matmul(un["h"], prepared["W_up"], out=un["c_up"])
        torch.matmul(un["up"], t["W_down"], out=un["c_down"])

    part_bytes = dict(qkv=act + rowvec + d * 3 * d * BF16 + T * 3 * d * BF16,
                      out=2 * act + d * d * BF16 + act + rowvec,
                      up=act + rowvec + d * 2 * ffn * BF16 + T * ffn * BF16,
                      down=T * ffn * BF16 + ffn * d * BF16 + 2 * act + rowvec)
    fb = sum(part_bytes.values())
    ub = (2 * act) + (act + d * 3 * d * BF16 + T * 3 * d * BF16) + (act + d * d * BF16 + act) + 3 * act + \
         (2 * act) + (act + d * 2 * ffn * BF16 + T * 2 * ffn * BF16) + (T * 2 * ffn * BF16 + T * ffn * BF16) + \
         (T * ffn * BF16 + ffn * d * BF16 + act) + 3 * act
    return Step("llama", flops, fb, ub, fused, unfused,
                host_inputs=dict(X=t["X"], X_sumsq=t["X_sumsq"], attn_out=t["attn_out"]),
                host_outputs=dict(y=out["y"], y_sumsq=out["y_sumsq"], qkv=out["qkv"]), kernels_per_fused=6,
                kernels_per_unfused=9, prep=prep, outputs=out, library=library,
                parts=[(name, call, part_flops[name]) for name, call in calls], parts_bytes=part_bytes, e2e=e2e,
                unfused_library=unfused_library)


BUILDERS = dict(rmsproj=build_rmsproj, lnproj=build_lnproj, swiglu=build_swiglu, dgrad=build_dgrad,
                llama=build_llama, skinny=build_skinny, wgrad=build_wgrad, fp8swiglu=build_fp8swiglu,
                mxfp8swiglu=build_mxfp8swiglu)
