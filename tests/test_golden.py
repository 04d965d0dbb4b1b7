"""The fp64 oracles against the regression fixtures in tests/golden/ (written
by tests/golden/make_golden.py from the oracles alone; see its README): a
change to an oracle's arithmetic shows up here."""
import json
import os

import numpy as np
import torch

import oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
RTOL = 1e-12


def _bf16(bits, shape):
    a = np.asarray(bits, dtype=np.int32).astype(np.uint16).view(np.int16)
    return torch.from_numpy(a.copy()).view(torch.bfloat16).reshape(shape)


def _f64(xs):
    return np.asarray([float(x) for x in xs], dtype=np.float64)


def _close(got, want, what):
    got = np.asarray(got, dtype=np.float64).flatten()
    assert got.shape == want.shape, what
    err = np.abs(got - want).max()
    assert err <= RTOL * max(1.0, np.abs(want).max()), f"{what}: max error {err}"


def test_attention_fixture():
    with open(os.path.join(HERE, "attention_small.json")) as f:
        cases = json.load(f)["cases"]
    assert len(cases) == 2
    for c in cases:
        B, Hq, Hkv, Sq, Skv, D = c["shape"]
        q = _bf16(c["q_bf16"], (B, Hq, Sq, D))
        k = _bf16(c["k_bf16"], (B, Hkv, Skv, D))
        v = _bf16(c["v_bf16"], (B, Hkv, Skv, D))
        dout = _bf16(c["dout_bf16"], (B, Hq, Sq, D))
        o, lse = oracle.attn_fwd(q, k, v, c["causal"], c["scale"])
        _close(o, _f64(c["o"]), "O")
        _close(lse, _f64(c["lse"]), "LSE")
        dq, dk, dv = oracle.attn_bwd(q, k, v, dout, c["causal"], c["scale"])
        _close(dq, _f64(c["dq"]), "dQ")
        _close(dk, _f64(c["dk"]), "dK")
        _close(dv, _f64(c["dv"]), "dV")


def test_chunk_scan_fixture():
    with open(os.path.join(HERE, "chunk_scan_small.json")) as f:
        c = json.load(f)["case"]
    B, L, H, P, G, Q = c["shape"]
    nch = L // Q
    cb = torch.tensor(_f64(c["cb"]), dtype=torch.float32).reshape(B, nch, G, Q, Q)
    dA = torch.tensor(_f64(c["dA_cs"]), dtype=torch.float32).reshape(B, H, nch, Q)
    dt = torch.tensor(_f64(c["dt"]), dtype=torch.float32).reshape(B, H, nch, Q)
    x = _bf16(c["x_bf16"], (B, L, H, P))
    out = oracle.chunk_scan_default().chunk_scan(cb, dA, dt, x)
    _close(out, _f64(c["out"]), "chunk scan out")
