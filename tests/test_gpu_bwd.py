"""Parity of the CUDA backward (attn_bwd) against the fp64 oracle.

Inputs: seeded q, k, v (synthetic.make_qkv) and dO drawn the same way; the
GPU backward consumes the GPU forward's O and LSE, the oracle forms its own
exact softmax.  Tolerance (derived, the pages fix none for the backward):
each gradient is a sum of products that carry at most three bf16 roundings
(P or dS before its GEMM, O in D_i, the output), 3 * 2^-9 relative per term;
dQ and dK also cancel (every row of dS sums to zero), so errors are measured
against the gradient's norm: relative Frobenius error <= 2^-6 and every
element within 2^-4 of the tensor's largest magnitude.
"""
import math

import numpy as np
import pytest
import torch

import attention_pipelining_gb300 as ap
import oracle
from attention_pipelining_gb300.synthetic import make_qkv

pytestmark = pytest.mark.gpu

REL_FRO = 2.0 ** -6
REL_MAX = 2.0 ** -4


@pytest.fixture(scope="module", autouse=True)
def _built():
    ap.build()
    ap.device_status(reset=True)
    yield


def make_dout(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def gpu_bwd(q, k, v, dout, causal, scale):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, dout))
    o, lse = ap.attn_fwd(qd, kd, vd, causal, scale)
    dq, dk, dv = ap.attn_bwd(qd, kd, vd, o, lse, dod, causal, scale)
    torch.cuda.synchronize()
    assert ap.device_status(reset=True) == 0
    return dq.float().cpu().numpy(), dk.float().cpu().numpy(), dv.float().cpu().numpy()


def assert_close(name, got, ref):
    ref = np.asarray(ref, np.float64)
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    err = np.abs(got - ref)
    fro = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)
    mx = err.max() / max(np.abs(ref).max(), 1e-30)
    assert fro <= REL_FRO and mx <= REL_MAX, (
        f"{name}: relative Frobenius error {fro:.3e} (<= {REL_FRO:.3e}), "
        f"max error / max |ref| {mx:.3e} (<= {REL_MAX:.3e})")


SHAPES = [
    # B, H_q, H_kv, S_q, S_kv, D, causal
    (1, 2, 2, 128, 128, 128, False),
    (1, 2, 2, 256, 256, 128, True),
    (1, 2, 1, 200, 300, 64, True),      # ragged, grouped heads, S_kv > S_q
    (2, 4, 2, 256, 384, 128, False),
    (1, 3, 1, 77, 150, 64, False),      # three heads per group, tiny S_q
    (1, 1, 1, 513, 129, 128, True),     # S_kv < S_q, ragged tails
    (2, 2, 2, 640, 640, 64, True),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_bwd_matches_oracle(shape):
    B, Hq, Hkv, Sq, Skv, D, causal = shape
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=11)
    dout = make_dout(q.shape, 12)
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = gpu_bwd(q, k, v, dout, causal, scale)
    rq, rk, rv = oracle.attn_bwd(q, k, v, dout, causal, scale)
    assert_close("dq", dq, rq)
    assert_close("dk", dk, rk)
    assert_close("dv", dv, rv)


def test_bwd_medium_causal_full():
    B, Hq, Hkv, Sq, Skv, D = 1, 4, 2, 1024, 1024, 128
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=13)
    dout = make_dout(q.shape, 14)
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = gpu_bwd(q, k, v, dout, True, scale)
    rq, rk, rv = oracle.attn_bwd(q, k, v, dout, True, scale)
    assert_close("dq", dq, rq)
    assert_close("dk", dk, rk)
    assert_close("dv", dv, rv)


def test_bwd_k_scaled_by_3():
    """A near one-hot softmax (the grouped-query workload's K x 3)."""
    B, Hq, Hkv, Sq, Skv, D = 1, 4, 1, 256, 256, 64
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, k_scale=3.0, seed=15)
    dout = make_dout(q.shape, 16)
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = gpu_bwd(q, k, v, dout, True, scale)
    rq, rk, rv = oracle.attn_bwd(q, k, v, dout, True, scale)
    assert_close("dq", dq, rq)
    assert_close("dk", dk, rk)
    assert_close("dv", dv, rv)


@pytest.mark.parametrize("name", ["batched_b4_h16_s2048_d128", "gqa_b8_hq32_hkv8_s4096_d64_k3",
                                  "long_b1_h32_s16384_d128", "long_causal_b1_h32_s16384_d128"])
def test_bwd_workload_sampled_rows(name):
    """Workload-size run: sampled query rows (dQ) and key rows (dK, dV) against
    the oracle, plus identities that hold at any size."""
    from attention_pipelining_gb300.synthetic import WORKLOADS, make_workload
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    dout = make_dout(q.shape, 17)
    dq, dk, dv = gpu_bwd(q, k, v, dout, w.causal, w.scale)
    rng = np.random.default_rng(18)
    nq = w.B * w.H_q * w.S_q
    qrows = np.unique(np.concatenate([[0, nq - 1], rng.integers(0, nq, 62)]))
    bo = oracle.bwd_default()
    ref_q = bo.dq_rows(q, k, v, dout, qrows, w.causal, w.scale)
    assert_close("dq rows", dq.reshape(-1, w.D)[qrows], ref_q)
    # key rows of two groups (each needs all of its group's softmax rows)
    groups = [0, w.B * w.H_kv - 1]
    krows = np.concatenate([g * w.S_kv + rng.integers(0, w.S_kv, 8) for g in groups])
    krows = np.unique(np.concatenate([krows, [0, w.B * w.H_kv * w.S_kv - 1]]))
    ref_k, ref_v = bo.dkv_rows(q, k, v, dout, krows, w.causal, w.scale)
    assert_close("dk rows", dk.reshape(-1, w.D)[krows], ref_k)
    assert_close("dv rows", dv.reshape(-1, w.D)[krows], ref_v)
    # sum_j dV_j = sum of dO over the group's rows; sum_j dK_j = 0
    rep = w.H_q // w.H_kv
    do_group = dout.double().numpy().reshape(w.B, w.H_kv, rep, w.S_q, w.D).sum(axis=(2, 3))
    sv = dv.astype(np.float64).sum(axis=2)
    assert np.abs(sv - do_group).max() <= 0.02 * np.abs(do_group).max() + 0.05
    sk = dk.astype(np.float64).sum(axis=2)
    assert np.abs(sk).max() <= 0.02 * np.abs(dk).astype(np.float64).sum(axis=2).max()


def test_bwd_deterministic_and_rejects_bad_workspace():
    B, Hq, Hkv, S, D = 1, 2, 1, 256, 128
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, S, S, D, seed=19))
    dout = make_dout(q.shape, 20).cuda()
    scale = 1.0 / math.sqrt(D)
    o, lse = ap.attn_fwd(q, k, v, True, scale)
    a = ap.attn_bwd(q, k, v, o, lse, dout, True, scale)
    b = ap.attn_bwd(q, k, v, o, lse, dout, True, scale)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ap.AttnError):
        ap.attn_bwd(q, k, v, o, lse, dout, True, scale, workspace=small)
    assert ap.device_status(reset=True) == 0


HOST_BWD_SHAPES = [
    # B, H_q, H_kv, S, D, causal: the first two are cut into chunks (inputs >= 32 MiB)
    (1, 16, 16, 8192, 128, False),
    (4, 8, 2, 4096, 64, True),
    (1, 2, 2, 256, 128, True),      # one chunk
]


@pytest.mark.parametrize("shape", HOST_BWD_SHAPES, ids=[str(s) for s in HOST_BWD_SHAPES])
def test_bwd_host_entry_matches_device_entry(shape):
    """attn_bwd_host (pinned host buffers, chunked copies and kernels on its
    own streams) gives the same bits as attn_bwd on device buffers, called
    twice in a row on a side stream."""
    B, Hq, Hkv, S, D, causal = shape
    q, k, v = make_qkv(B, Hq, Hkv, S, S, D, seed=21)
    dout = make_dout(q.shape, 22)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, dout))
    o, lse = ap.attn_fwd(qd, kd, vd, causal, scale)
    ref = ap.attn_bwd(qd, kd, vd, o, lse, dod, causal, scale)
    torch.cuda.synchronize()
    host_in = [t.pin_memory() for t in (q, k, v, o.cpu(), lse.cpu(), dout)]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in ref]
    dev_in = [torch.empty_like(t) for t in (qd, kd, vd, o, lse, dod)]
    dev_out = [torch.empty_like(t) for t in ref]
    ws = torch.empty(ap.bwd_workspace_bytes(B, Hq, Hkv, S), dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    for _ in range(2):
        for t in host_out:
            t.fill_(0)
        ap.attn_bwd_host(*host_in, *host_out, *dev_in, *dev_out, causal, scale, ws, stream=side)
        side.synchronize()
        assert ap.device_status(reset=True) == 0
        for name, got, want in zip(("dq", "dk", "dv"), host_out, ref):
            assert torch.equal(got, want.cpu()), name
