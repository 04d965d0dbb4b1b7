"""Seeded synthetic inputs for the attention forward.

This module only draws random numbers; it holds none of the attention
arithmetic.  Both the CUDA path (through the tests and the benchmark) and the
fp64 oracle consume what it produces.

Recipe: a CPU ``torch.Generator`` seeded with ``seed``; q, k, v drawn in that
order as float32 iid N(0, 1) of shape [B, H, S, D]; k multiplied by
``k_scale`` in float32 (the grouped-query workload stresses the softmax range
with k_scale = 3); every tensor then rounded once to bf16 (round to nearest
even).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, asdict

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H_q: int
    H_kv: int
    S_q: int
    S_kv: int
    D: int
    causal: bool
    k_scale: float = 1.0
    seed: int = 0
    path: str = "fused"   # "fused": attn_fwd; "splitkv": attn_fwd_splitkv (decoding shapes)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> float:
        """4 * B * H_q * S_q * S_kv * D, halved when causal (two GEMMs of 2*M*N*K)."""
        f = 4.0 * self.B * self.H_q * self.S_q * self.S_kv * self.D
        return f / 2.0 if self.causal else f

    @property
    def io_bytes(self) -> int:
        """Bytes the operation must move at least: Q, K, V read; O, LSE written."""
        q = self.B * self.H_q * self.S_q * self.D * 2
        kv = 2 * self.B * self.H_kv * self.S_kv * self.D * 2
        return q + kv + q + self.B * self.H_q * self.S_q * 4

    def as_dict(self) -> dict:
        d = asdict(self)
        d["scale"] = self.scale
        return d


# The headline workloads: shapes, masks and distributions of the pages'
# attention-forward microbenchmarks (long-sequence case at S = 16384).
WORKLOADS = {
    w.name: w
    for w in [
        Workload("single_head_b1_h1_s256_d64", 1, 1, 1, 256, 256, 64, False),
        Workload("batched_b4_h16_s2048_d128", 4, 16, 16, 2048, 2048, 128, False),
        Workload("causal_b2_h16_s8192_d128", 2, 16, 16, 8192, 8192, 128, True),
        Workload("long_b1_h32_s16384_d128", 1, 32, 32, 16384, 16384, 128, False),
        Workload("long_causal_b1_h32_s16384_d128", 1, 32, 32, 16384, 16384, 128, True),
        Workload("gqa_b8_hq32_hkv8_s4096_d64_k3", 8, 32, 8, 4096, 4096, 64, True, k_scale=3.0),
        # decoding: one query token per sequence against an 8192-token KV cache,
        # grouped heads of an 8B-class model (32 query heads over 8 KV heads)
        Workload("decode_b32_hq32_hkv8_sq1_skv8192_d128", 32, 32, 8, 1, 8192, 128, False,
                 path="splitkv"),
    ]
}

HEADLINE = "long_b1_h32_s16384_d128"


def make_qkv(B: int, H_q: int, H_kv: int, S_q: int, S_kv: int, D: int,
             k_scale: float = 1.0, seed: int = 0):
    """q [B,H_q,S_q,D], k and v [B,H_kv,S_kv,D], all bf16 on the CPU."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    q = torch.randn((B, H_q, S_q, D), generator=g, dtype=torch.float32)
    k = torch.randn((B, H_kv, S_kv, D), generator=g, dtype=torch.float32)
    v = torch.randn((B, H_kv, S_kv, D), generator=g, dtype=torch.float32)
    if k_scale != 1.0:
        k = k * k_scale
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def make_workload(w: Workload):
    return make_qkv(w.B, w.H_q, w.H_kv, w.S_q, w.S_kv, w.D, w.k_scale, w.seed)


# ---------------------------------------------------------------- chunk scan


@dataclass(frozen=True)
class ChunkScanWorkload:
    """Shapes of the Mamba2 chunk scan: batch B, sequence L, H heads of width
    P in G groups, chunk length Q."""
    name: str
    B: int
    L: int
    H: int = 64
    P: int = 64
    G: int = 1
    Q: int = 256
    seed: int = 0

    @property
    def nchunks(self) -> int:
        return self.L // self.Q

    @property
    def flops(self) -> float:
        """2 * P multiply-adds per (row, visible key): sum over a chunk of
        (m + 1) keys for rows m = 0..Q-1."""
        per_chunk = self.Q * (self.Q + 1) / 2
        return 2.0 * self.P * per_chunk * self.nchunks * self.B * self.H

    @property
    def io_bytes(self) -> int:
        """cb, dA_cs, dt, x read; out written."""
        cb = self.B * self.nchunks * self.G * self.Q * self.Q * 4
        vec = 2 * self.B * self.H * self.L * 4
        x = self.B * self.L * self.H * self.P * 2
        return cb + vec + 2 * x

    def as_dict(self) -> dict:
        return asdict(self)


# Mamba2-1.3B (64 heads of width 64, one group, chunk 256) at the batch and
# sequence sizes of the pages' chunk-scan microbenchmarks
CHUNK_SCAN_WORKLOADS = {
    w.name: w
    for w in [
        ChunkScanWorkload("chunkscan_b1_s1024", 1, 1024),
        ChunkScanWorkload("chunkscan_b1_s8192", 1, 8192),
        ChunkScanWorkload("chunkscan_b64_s8192", 64, 8192),
        # the CTA shape of 64 x 8192 (32 heads per CTA) at an eighth of the
        # memory: for profiling
        ChunkScanWorkload("chunkscan_b8_s8192", 8, 8192),
    ]
}

CHUNK_SCAN_HEADLINE = "chunkscan_b64_s8192"


def make_chunk_scan(B: int, L: int, H: int, P: int, G: int, Q: int, seed: int = 0,
                    device: str = "cpu"):
    """Seeded chunk-scan inputs (on `device`): cb [B, L/Q, G, Q, Q] fp32,
    dA_cs [B, H, L/Q, Q] fp32, dt [B, H, L/Q, Q] fp32, x [B, L, H, P] bf16.

    Recipe: x ~ N(0, 1) rounded to bf16; dt = softplus(0.5 N(0, 1) - 3) (about
    0.05); a per-head decay rate A_h = -exp(U(0, ln 16)); dA = dt A_h and
    dA_cs its running sum within each chunk; cb ~ N(0, 1).  Drawn in the
    order x, dt, A, cb."""
    nch = L // Q
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    kw = dict(generator=g, dtype=torch.float32, device=device)
    x = torch.randn((B, L, H, P), **kw).to(torch.bfloat16)
    dt = torch.nn.functional.softplus(0.5 * torch.randn((B, H, nch, Q), **kw) - 3.0)
    A = -torch.exp(torch.rand((H,), **kw) * math.log(16.0))
    dA_cs = torch.cumsum(dt * A.view(1, H, 1, 1), dim=-1)
    cb = torch.randn((B, nch, G, Q, Q), **kw)
    return cb, dA_cs.contiguous(), dt.contiguous(), x


def make_chunk_scan_workload(w: ChunkScanWorkload, device: str = "cpu"):
    return make_chunk_scan(w.B, w.L, w.H, w.P, w.G, w.Q, w.seed, device=device)
