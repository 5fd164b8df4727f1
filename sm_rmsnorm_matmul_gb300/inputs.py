"""Seeded synthetic inputs for the fused RMSNorm+MatMul workloads.

This module only draws random numbers and rounds them to bf16.  It holds none
of the method's arithmetic (no statistic, no normalisation, no contraction), so
the CUDA path and the fp64 CPU oracle can both be fed from it without sharing
any of the computation they are compared on.

Recipe (the same for every workload):

* one ``torch.Generator`` on the CPU, seeded with the workload's seed;
* draws are made in this fixed order, each in fp32: the X normals, then the
  per-entry outlier uniforms or the per-row scales (when the workload has
  them), then the g uniforms, then the W normals;
* every tensor is rounded once to bf16 (round to nearest even) at the end.

Distribution parameters: ``N(0, s)`` means standard deviation ``s``; g is
``U(0.5, 1.5)``; "1% of entries x20" is an independent Bernoulli(0.01) draw per
entry of X that multiplies the entry by 20; the per-row scale is
``exp(U(ln 0.1, ln 10))`` (log-uniform on [0.1, 10]) and multiplies a whole row.

The workloads are the shapes the Mirage pages' headline muGraph (RMSNorm
followed by MatMul, Mirage review page, section 3 "muGraph example") takes in
decoder-only transformer layers: decode-time QKV and gate|up projections and
prefill-time projections.  The pages name no dataset; these synthetic inputs
stand in for real activations and weights.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    K: int
    N: int
    eps: float
    seed: int
    w_std: float
    x_kind: str = "normal"  # "normal" | "outlier_entries" | "row_scaled"
    oracle_rows: int = 0    # 0: the oracle checks every row; else a row sample

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def bytes_xwy(self) -> int:
        return 2 * (self.M * self.K + self.K * self.N + self.M * self.N)

    @property
    def bytes_algorithmic(self) -> int:
        """X + W + Y + g, each moved once."""
        return self.bytes_xwy + 2 * self.K


WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny_8x1024x1024", 8, 1024, 1024, 1e-6, 0, 1.0 / math.sqrt(1024)),
        Workload("decode_qkv_16x4096x6144", 16, 4096, 6144, 1e-6, 1, 1.0 / 64,
                 x_kind="outlier_entries"),
        Workload("decode_gatedmlp_64x4096x28672", 64, 4096, 28672, 1e-5, 2, 1.0 / 64),
        Workload("prefill_qkv_4096x4096x6144", 4096, 4096, 6144, 1e-6, 3, 1.0 / 64,
                 x_kind="row_scaled"),
        Workload("large_prefill_16384x8192x8192", 16384, 8192, 8192, 1e-5, 4,
                 1.0 / math.sqrt(8192), oracle_rows=256),
    )
}

WORKLOAD_ORDER = list(WORKLOADS)

# Small cases of the prefill kernels, for profiler captures that replay a
# launch many times (inputs still larger than L2, a few hundred MB on the
# device).  `bench.py --workload` accepts them; no benchmark line uses them.
PROFILE_CASES = {
    w.name: w
    for w in (
        # paired kernel: 19 row-block pairs x 4 column tiles = 76 units, one round;
        # the unfused pair times the 256-row kernel on it
        Workload("paired_prefill_4864x8192x1024", 4864, 8192, 1024, 1e-5, 5, 1.0 / math.sqrt(8192)),
        # the 256-row kernel of the unfused pair: 16 x 16 = 256 whole tiles, two waves
        Workload("unfused_prefill_4096x8192x4096", 4096, 8192, 4096, 1e-5, 6, 1.0 / math.sqrt(8192)),
    )
}


def sample_rows(M: int, count: int = 256) -> list[int]:
    """Rows r_i = 64*i + (i mod 64) clipped to [0, M), plus the last row.

    Each residue mod 64 appears several times (it hits every lane position of
    a 128-row tile), and row 0 and row M-1 are always included.
    """
    rows = sorted({min(M - 1, 64 * i + (i % 64)) for i in range(count)} | {0, M - 1})
    return rows[:count] if len(rows) > count else rows


def generate(M: int, K: int, N: int, *, seed: int, w_std: float,
             x_kind: str = "normal"):
    """Return (X [M,K], g [K], W [K,N]) as contiguous bf16 CPU tensors."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    x = torch.randn(M, K, generator=gen, dtype=torch.float32)
    if x_kind == "outlier_entries":
        u = torch.rand(M, K, generator=gen, dtype=torch.float32)
        x = torch.where(u < 0.01, x * 20.0, x)
    elif x_kind == "row_scaled":
        u = torch.rand(M, 1, generator=gen, dtype=torch.float32)
        lo, hi = math.log(0.1), math.log(10.0)
        x = x * torch.exp(lo + (hi - lo) * u)
    elif x_kind != "normal":
        raise ValueError(f"unknown x_kind {x_kind!r}")
    g = 0.5 + torch.rand(K, generator=gen, dtype=torch.float32)
    w = torch.randn(K, N, generator=gen, dtype=torch.float32) * w_std
    return (x.to(torch.bfloat16).contiguous(), g.to(torch.bfloat16).contiguous(),
            w.to(torch.bfloat16).contiguous())


def generate_workload(w: Workload):
    return generate(w.M, w.K, w.N, seed=w.seed, w_std=w.w_std, x_kind=w.x_kind)


def random_problem(M: int, K: int, N: int, seed: int, x_kind: str = "normal"):
    """A ragged-shape problem with the same distributions (W std 1/sqrt(K))."""
    return generate(M, K, N, seed=seed, w_std=1.0 / math.sqrt(K), x_kind=x_kind)


def lora_adapter(K: int, N: int, R: int, seed: int, share: float = 1.0):
    """A low-rank adapter (A [K,R], B [R,N]) as contiguous bf16 CPU tensors:
    A ~ N(0, 1/sqrt(K)), B ~ N(0, sqrt(share/R)), so that each element of
    A @ B has variance share/K: with share = 1 the adapter's part of the output
    is of the same order as that of a W of std 1/sqrt(K)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    a = torch.randn(K, R, generator=gen, dtype=torch.float32) / math.sqrt(K)
    b = torch.randn(R, N, generator=gen, dtype=torch.float32) * math.sqrt(share / R)
    return a.to(torch.bfloat16).contiguous(), b.to(torch.bfloat16).contiguous()


def lora_problem(M: int, K: int, N: int, R: int, seed: int, x_kind: str = "row_scaled"):
    """X, g, W, A, B for RMSNorm(X) @ (W + A @ B) with unit-RMS outputs, like
    every workload above: W ~ N(0, 1/sqrt(2K)) and an adapter of share 1/2, so
    that W + A @ B has the per-element variance 1/K of a plain workload's W."""
    X, g, W = generate(M, K, N, seed=seed, w_std=1.0 / math.sqrt(2 * K), x_kind=x_kind)
    A, B = lora_adapter(K, N, R, seed=seed + 1, share=0.5)
    return X, g, W, A, B


@dataclass(frozen=True)
class AttentionWorkload:
    """QK-normalised attention over the output of a fused QKV projection:
    B sequences of S tokens, Hq query heads and Hkv key/value heads of D."""
    name: str
    B: int
    S: int
    Hq: int
    Hkv: int
    D: int
    eps: float
    causal: bool
    seed: int

    @property
    def flops(self) -> float:
        """2 S D per query-key pair for each of the two products; causal
        attention visits S (S + 1) / 2 pairs per head, full attention S^2."""
        pairs = self.S * (self.S + 1) / 2 if self.causal else self.S * self.S
        return 4.0 * self.B * self.Hq * self.D * pairs

    @property
    def bytes_algorithmic(self) -> int:
        """Q, K, V read once, O written once, bf16."""
        return 2 * self.B * self.S * self.D * (2 * self.Hq + 2 * self.Hkv)


# The prefill QKV projection's output (4096 tokens x 6144 columns) read as
# 32 query heads and 8 key/value heads of 128 (grouped-query attention).
ATTENTION_WORKLOADS = {
    "prefill_attention_1x4096_h32_kv8_d128_causal": AttentionWorkload(
        "prefill_attention_1x4096_h32_kv8_d128_causal", B=1, S=4096, Hq=32, Hkv=8, D=128,
        eps=1e-6, causal=True, seed=5),
    # the same sequence and heads with head dimension 64
    "prefill_attention_1x4096_h32_kv8_d64_causal": AttentionWorkload(
        "prefill_attention_1x4096_h32_kv8_d64_causal", B=1, S=4096, Hq=32, Hkv=8, D=64,
        eps=1e-6, causal=True, seed=6),
}


def attention_inputs(B: int, S: int, Hq: int, Hkv: int, D: int, seed: int):
    """A fused QKV projection output [B*S, (Hq + 2*Hkv)*D] as a contiguous bf16
    CPU tensor, and the gains gq, gk [D]: entries N(0, 1), every token's row
    scaled by one LogUniform(0.1, 10) factor (the spread of row norms the
    normalisation has to remove), gains U(0.5, 1.5)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    width = (Hq + 2 * Hkv) * D
    qkv = torch.randn(B * S, width, generator=gen, dtype=torch.float32)
    u = torch.rand(B * S, 1, generator=gen, dtype=torch.float32)
    qkv *= torch.exp(math.log(0.1) + u * (math.log(10.0) - math.log(0.1)))
    gq = 0.5 + torch.rand(D, generator=gen, dtype=torch.float32)
    gk = 0.5 + torch.rand(D, generator=gen, dtype=torch.float32)
    return (qkv.to(torch.bfloat16).contiguous(), gq.to(torch.bfloat16).contiguous(),
            gk.to(torch.bfloat16).contiguous())


def split_qkv(qkv, B: int, S: int, Hq: int, Hkv: int, D: int):
    """Views Q [B,S,Hq,D], K and V [B,S,Hkv,D] of a fused QKV tensor."""
    t = qkv.view(B, S, Hq + 2 * Hkv, D)
    return t[:, :, :Hq], t[:, :, Hq:Hq + Hkv], t[:, :, Hq + Hkv:]
