"""Writes the regression fixtures in this folder.  It calls only the fp64
oracle (``oracle/``) and the seeded input generator; nothing here comes from
the CUDA path.  Inputs are stored with the outputs (bf16 as bit patterns,
fp32 as decimal strings that round-trip), so the fixtures do not depend on a
random-number generator.

    python tests/golden/make_golden.py

Rewrite a fixture only together with a change to the oracle's arithmetic,
in a commit that names the passage of the pages (or the reading of it) that
justifies the change.
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from attention_pipelining_gb300.synthetic import make_chunk_scan, make_qkv  # noqa: E402


def bf16_bits(t: torch.Tensor) -> list[int]:
    return t.contiguous().view(torch.int16).flatten().to(torch.int32).bitwise_and(0xFFFF).tolist()


def f32_list(t) -> list[str]:
    a = np.asarray(t.detach().cpu().numpy() if torch.is_tensor(t) else t, dtype=np.float32)
    return [repr(float(x)) for x in a.flatten()]


def f64_list(a) -> list[str]:
    return [repr(float(x)) for x in np.asarray(a, dtype=np.float64).flatten()]


def attention_cases():
    out = []
    for causal in (False, True):
        B, Hq, Hkv, Sq, Skv, D = 1, 2, 1, 5, 7, 8
        q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=11)
        scale = 0.35
        g = torch.Generator().manual_seed(12)
        dout = torch.randn((B, Hq, Sq, D), generator=g).to(torch.bfloat16)
        o, lse = oracle.attn_fwd(q, k, v, causal, scale)
        dq, dk, dv = oracle.attn_bwd(q, k, v, dout, causal, scale)
        out.append({
            "shape": [B, Hq, Hkv, Sq, Skv, D], "causal": causal, "scale": scale,
            "q_bf16": bf16_bits(q), "k_bf16": bf16_bits(k), "v_bf16": bf16_bits(v),
            "dout_bf16": bf16_bits(dout),
            "o": f64_list(o), "lse": f64_list(lse),
            "dq": f64_list(dq), "dk": f64_list(dk), "dv": f64_list(dv),
        })
    return out


def chunk_scan_case():
    B, L, H, P, G, Q = 1, 16, 2, 4, 1, 8
    cb, dA_cs, dt, x = make_chunk_scan(B, L, H, P, G, Q, seed=13)
    out = oracle.chunk_scan_default().chunk_scan(cb, dA_cs, dt, x)
    return {
        "shape": [B, L, H, P, G, Q],
        "cb": f32_list(cb), "dA_cs": f32_list(dA_cs), "dt": f32_list(dt), "x_bf16": bf16_bits(x),
        "out": f64_list(out),
    }


def main():
    with open(os.path.join(HERE, "attention_small.json"), "w") as f:
        json.dump({"about": "fp64 oracle forward (O, LSE) and backward (dQ, dK, dV) of two small "
                            "grouped-query problems; see README.md",
                   "cases": attention_cases()}, f, indent=0)
    with open(os.path.join(HERE, "chunk_scan_small.json"), "w") as f:
        json.dump({"about": "fp64 chunk-scan oracle on one small problem; see README.md",
                   "case": chunk_scan_case()}, f, indent=0)


if __name__ == "__main__":
    main()
