"""Seeded synthetic inputs for the GEMM+epilogue workloads.

This module is shared by the tests, the benchmark and the oracle's callers.  It
holds no arithmetic of the method itself: it only draws random tensors with the
shapes and value distributions of the workloads and rounds them to bf16.

The workloads stand in for the "GPT-2 / BERT / LLaMA scale" Transformer blocks
that the CODA article (d9bl.com, "CODA：将 Transformer 模块重新表达为
GEMM+Epilogue 程序", §4.2, Fig. 8) trains on; the pages name no dataset and
print no shapes, so every shape and distribution below is the one fixed by the
workload descriptions:

  pr1      D = X@W + bias -> GELU(tanh) -> + residual, X[256,256], W[256,256],
           bias[256], residual[256,256], entries N(0,1)/sqrt(256)
  rmsproj  commuted RMSNorm projection, X[4096,2048] ~ N(0,1),
           gamma[2048] ~ U(0.5,1.5), W[2048,8192] ~ N(0, var 1/2048)
  swiglu   [G|U] = Xn @ W[4096, 2*11008], SiLU(G)*U, dropout p=0.1,
           Xn[8192,4096] ~ N(0,1), W ~ N(0, var 1/4096)
  dgrad    dX = (dY @ W^T) * GELU'(Z) and per-row sum(dX*Xhat), dY[8192,4096],
           W[16384,4096], Z and Xhat [8192,16384], all N(0,1)
  lnproj   commuted LayerNorm projection (the GPT-2 / BERT normalisation),
           the rmsproj shapes: X[4096,2048] ~ N(0,1) plus a per-row offset
           ~ N(0.5, 0.5^2), gamma ~ U(0.5,1.5), beta ~ N(0, 0.1^2),
           W[2048,8192] ~ N(0, var 1/2048)
  skinny   the LLaMA block's MLP up-projection at 128 tokens (a decode-sized
           batch): commuted RMSNorm -> SwiGLU, X[128,4096] ~ N(0,1),
           gamma ~ U(0.5,1.5), W[4096,2*11008] ~ N(0, std 0.02).  180 MB of
           weights against 23 GFLOP: bound by HBM, not by the tensor cores
  fp8swiglu the swiglu up-projection with FP8 E4M3 operands: X quantised per
           row each step, W[2*11008,4096] ([N, K]) quantised per output
           channel once; D = SiLU(G)*U of the dequantised product
  wgrad    the LLaMA MLP down-projection's weight gradient at 16384 tokens:
           dW = s * up^T @ dY + dW_old (scaled, accumulated in place) with the
           per-row sums of squares (gradient-norm partials); up[16384,11008]
           ~ N(0, 0.5^2) (a SwiGLU output), dY[16384,4096] ~ N(0, 0.01^2),
           dW_old ~ N(0, 0.01^2), s = 1/8 (eight accumulation steps)
  llama    LLaMA-7B-like non-attention block at 16384 tokens, d=4096,
           ffn=11008, weights N(0, std 0.02), gammas U(0.5,1.5)

Generation: a torch CPU generator seeded per tensor, fp32 draws, then one
round-to-nearest-even conversion to bf16.  The oracle widens those exact bf16
values to fp64, so both sides see identical inputs.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

# ---------------------------------------------------------------------------
# workload table
# ---------------------------------------------------------------------------


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    K: int
    N: int              # GEMM output width (for SwiGLU: 2 * N_out)
    b_layout: str       # "kn": B is [K,N] row-major; "nk": B is [N,K] row-major
    description: str
    extra: dict = field(default_factory=dict)

    @property
    def gemm_flops(self) -> int:
        return 2 * self.M * self.N * self.K


WORKLOADS = {
    "pr1": Workload("pr1", 256, 256, 256, "kn",
                    "D = X@W + bias -> GELU(tanh) -> + residual; X[256,256], W[256,256]"),
    "rmsproj": Workload("rmsproj", 4096, 2048, 8192, "kn",
                        "commuted RMSNorm projection D = rsqrt(mean(X^2)+1e-6) * (X @ (gamma*W)); "
                        "X[4096,2048], W[2048,8192]"),
    "lnproj": Workload("lnproj", 4096, 2048, 8192, "kn",
                       "commuted LayerNorm projection D = r (X @ (gamma*W) - mu colsum(gamma*W)) + beta@W; "
                       "X[4096,2048], W[2048,8192]"),
    "swiglu": Workload("swiglu", 8192, 4096, 2 * 11008, "kn",
                       "SwiGLU up-projection [G|U] = Xn @ W[4096,2*11008], SiLU(G)*U, dropout p=0.1"),
    "dgrad": Workload("dgrad", 8192, 4096, 16384, "nk",
                      "dgrad dX = (dY @ W^T) * GELU'(Z) + per-row sum(dX*Xhat), sum(dX); "
                      "dY[8192,4096], W[16384,4096]"),
    "skinny": Workload("skinny", 128, 4096, 2 * 11008, "kn",
                       "decode-sized MLP up-projection: rmsnorm(X[128,4096]) @ W[4096,2*11008], SiLU(G)*U"),
}

# LLaMA-7B-like non-attention block at 16384 tokens (four GEMM+epilogue calls)
LLAMA_BLOCK = dict(tokens=16384, d=4096, ffn=11008)

EPS_RMS = 1e-6
EPS_LN = 1e-5
WGRAD_SCALE = 0.125
DROPOUT_P = 0.1
DROPOUT_SEED = 0


# ---------------------------------------------------------------------------
# generators
# ---------------------------------------------------------------------------


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def randn_bf16(shape, std: float, seed: int) -> torch.Tensor:
    """N(0, std^2) drawn in fp32 on the CPU, rounded once to bf16."""
    t = torch.randn(*shape, generator=_gen(seed), dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def uniform_bf16(shape, lo: float, hi: float, seed: int) -> torch.Tensor:
    t = torch.rand(*shape, generator=_gen(seed), dtype=torch.float32)
    t.mul_(hi - lo).add_(lo)
    return t.to(torch.bfloat16)


def small_int_bf16(shape, lim: int, seed: int) -> torch.Tensor:
    """Integers in [-lim, lim], exactly representable in bf16 for lim <= 256."""
    t = torch.randint(-lim, lim + 1, shape, generator=_gen(seed), dtype=torch.int32)
    return t.to(torch.bfloat16)


def random_e4m3_codes(shape, seed: int, exp_lo: int = 7, exp_hi: int = 10) -> torch.Tensor:
    """Random FP8 E4M3 bytes: uniform sign and 3-bit mantissa, exponent field
    uniform in [exp_lo, exp_hi] (the default gives magnitudes 1 to 15.5, all
    multiples of 1/8).  Raw bit patterns: no arithmetic of the method."""
    g = _gen(seed)
    sign = torch.randint(0, 2, shape, generator=g, dtype=torch.int32) << 7
    expo = torch.randint(exp_lo, exp_hi + 1, shape, generator=g, dtype=torch.int32) << 3
    mant = torch.randint(0, 8, shape, generator=g, dtype=torch.int32)
    return (sign | expo | mant).to(torch.uint8)


def make_pr1(seed: int = 0, M: int = 256, K: int = 256, N: int = 256) -> dict:
    s = 1.0 / math.sqrt(256.0)
    return dict(
        X=randn_bf16((M, K), s, seed + 1),
        W=randn_bf16((K, N), s, seed + 2),
        bias=randn_bf16((N,), s, seed + 3),
        residual=randn_bf16((M, N), s, seed + 4),
    )


def make_rmsproj(seed: int = 0, M: int = 4096, K: int = 2048, N: int = 8192) -> dict:
    return dict(
        X=randn_bf16((M, K), 1.0, seed + 11),
        gamma=uniform_bf16((K,), 0.5, 1.5, seed + 12),
        W=randn_bf16((K, N), 1.0 / math.sqrt(2048.0), seed + 13),
    )


def make_lnproj(seed: int = 0, M: int = 4096, K: int = 2048, N: int = 8192) -> dict:
    X = torch.randn(M, K, generator=_gen(seed + 51), dtype=torch.float32)
    X += 0.5 + 0.5 * torch.randn(M, 1, generator=_gen(seed + 52), dtype=torch.float32)
    return dict(
        X=X.to(torch.bfloat16),
        gamma=uniform_bf16((K,), 0.5, 1.5, seed + 53),
        beta=randn_bf16((K,), 0.1, seed + 54),
        W=randn_bf16((K, N), 1.0 / math.sqrt(2048.0), seed + 55),
    )


def make_skinny(seed: int = 0, M: int = 128, K: int = 4096, N_out: int = 11008) -> dict:
    return dict(
        X=randn_bf16((M, K), 1.0, seed + 61),
        gamma=uniform_bf16((K,), 0.5, 1.5, seed + 62),
        W=randn_bf16((K, 2 * N_out), 0.02, seed + 63),
    )


def make_wgrad(seed: int = 0, T: int = 16384, d: int = 4096, ffn: int = 11008) -> dict:
    return dict(
        up=randn_bf16((T, ffn), 0.5, seed + 71),
        dY=randn_bf16((T, d), 0.01, seed + 72),
        dW_old=randn_bf16((ffn, d), 0.01, seed + 73),
    )


def make_swiglu(seed: int = 0, M: int = 8192, K: int = 4096, N_out: int = 11008) -> dict:
    return dict(
        X=randn_bf16((M, K), 1.0, seed + 21),
        W=randn_bf16((K, 2 * N_out), 1.0 / math.sqrt(4096.0), seed + 22),
    )


def make_dgrad(seed: int = 0, M: int = 8192, K: int = 4096, N: int = 16384) -> dict:
    return dict(
        dY=randn_bf16((M, K), 1.0, seed + 31),
        W=randn_bf16((N, K), 1.0, seed + 32),
        Z=randn_bf16((M, N), 1.0, seed + 33),
        Xhat=randn_bf16((M, N), 1.0, seed + 34),
    )


def make_llama_block(seed: int = 0, tokens: int = 16384, d: int = 4096, ffn: int = 11008) -> dict:
    w = 0.02
    return dict(
        X=randn_bf16((tokens, d), 1.0, seed + 41),
        gamma_attn=uniform_bf16((d,), 0.5, 1.5, seed + 42),
        W_qkv=randn_bf16((d, 3 * d), w, seed + 43),
        attn_out=randn_bf16((tokens, d), 1.0, seed + 44),
        W_o=randn_bf16((d, d), w, seed + 45),
        gamma_mlp=uniform_bf16((d,), 0.5, 1.5, seed + 46),
        W_up=randn_bf16((d, 2 * ffn), w, seed + 47),
        W_down=randn_bf16((ffn, d), w, seed + 48),
    )


def sample_rows(M: int, n: int, seed: int, tile: int = 128) -> list[int]:
    """Rows for sampled full-size comparison: the first and last row, both rows
    on each side of every `tile`-row boundary (128-row tiles, and so every
    256-row CTA-pair tile too), and `n` distinct random rows."""
    rows = {0, M - 1}
    for t in range(tile, M, tile):
        rows.add(t - 1)
        rows.add(t)
    g = _gen(seed)
    perm = torch.randperm(M, generator=g)[: min(n, M)].tolist()
    rows.update(perm)
    return sorted(r for r in rows if 0 <= r < M)
