"""Parity of the CUDA backward (attn_bwd, and attn_bwd_deterministic) against
the fp64 oracle.

Inputs: seeded q, k, v (synthetic.make_qkv) and dO drawn the same way; the
GPU backward consumes the GPU forward's O and LSE, the oracle forms its own
exact softmax.  Tolerance (derived, the pages fix none for the backward):
per element, 8 standard deviations of the rounding model of the GPU path (P,
dS and O rounded to bf16, independent roundings summed over each gradient's
terms; tests/bwd_bound.py) plus the output's own bf16 rounding, and the RMS
of the errors in units of that model's deviation at most 1.5.  Every check
prints the achieved errors.
"""
import math

import numpy as np
import pytest
import torch

import attention_pipelining_gb300 as ap
import oracle
from attention_pipelining_gb300.synthetic import make_qkv
from tests import bwd_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ap.build()
    ap.device_status(reset=True)
    yield


def make_dout(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def gpu_bwd(q, k, v, dout, causal, scale, deterministic=False):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, dout))
    o, lse = ap.attn_fwd(qd, kd, vd, causal, scale)
    dq, dk, dv = ap.attn_bwd(qd, kd, vd, o, lse, dod, causal, scale, deterministic=deterministic)
    torch.cuda.synchronize()
    assert ap.device_status(reset=True) == 0
    return dq.float().cpu().numpy(), dk.float().cpu().numpy(), dv.float().cpu().numpy()


def check_rows(q, k, v, dout, causal, scale, got, ref, qrows=None, krows=None, what=""):
    """got / ref: (dq, dk, dv) at the flat rows qrows (dq) and krows (dk, dv),
    all rows when None; each [n, D] or the full tensors."""
    D = q.shape[-1]
    nq = q.numel() // D
    nk = k.numel() // D
    qrows = np.arange(nq) if qrows is None else qrows
    krows = np.arange(nk) if krows is None else krows
    sq, aq = bwd_bound.dq_sigma(q, k, v, dout, qrows, causal, scale)
    sk, ak, sv, av = bwd_bound.dkv_sigma(q, k, v, dout, krows, causal, scale)
    for name, g, r, s_, a_ in (("dq", got[0], ref[0], sq, aq), ("dk", got[1], ref[1], sk, ak),
                               ("dv", got[2], ref[2], sv, av)):
        bwd_bound.check(f"{what} {name}", np.reshape(g, (-1, D)), np.reshape(r, (-1, D)), s_, a_)


SHAPES = [
    # B, H_q, H_kv, S_q, S_kv, D, causal
    (1, 2, 2, 128, 128, 128, False),
    (1, 2, 2, 256, 256, 128, True),
    (1, 2, 1, 200, 300, 64, True),      # ragged, grouped heads, S_kv > S_q
    (2, 4, 2, 256, 384, 128, False),
    (1, 3, 1, 77, 150, 64, False),      # three heads per group, tiny S_q
    (1, 1, 1, 513, 129, 128, True),     # S_kv < S_q, ragged tails
    (2, 2, 2, 640, 640, 64, True),
    (1, 8, 1, 40, 96, 128, True),       # eight heads per group, one ragged key block
    (2, 1, 1, 1, 33, 64, False),        # one query row: the second half block holds none
    (1, 4, 4, 64, 64, 128, True),       # exactly one half block of rows per head
    # causal with S_q a multiple of 128 (visible query blocks computed per
    # head): keys past the last position (no query block sees key block 2),
    # and more positions than keys
    (1, 2, 1, 256, 384, 128, True),
    (1, 4, 2, 384, 256, 64, True),
]


@pytest.mark.parametrize("deterministic", [False, True], ids=["default", "deterministic"])
@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_bwd_matches_oracle(shape, deterministic):
    """The default path computes dQ inside the dK/dV kernel (fp32 partials
    added in L2), the deterministic one by its own kernel."""
    B, Hq, Hkv, Sq, Skv, D, causal = shape
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=11)
    dout = make_dout(q.shape, 12)
    scale = 1.0 / math.sqrt(D)
    got = gpu_bwd(q, k, v, dout, causal, scale, deterministic)
    ref = oracle.attn_bwd(q, k, v, dout, causal, scale)
    check_rows(q, k, v, dout, causal, scale, got, ref, what=f"{shape} det={deterministic}")


def test_bwd_medium_causal_full():
    B, Hq, Hkv, Sq, Skv, D = 1, 4, 2, 1024, 1024, 128
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=13)
    dout = make_dout(q.shape, 14)
    scale = 1.0 / math.sqrt(D)
    got = gpu_bwd(q, k, v, dout, True, scale)
    ref = oracle.attn_bwd(q, k, v, dout, True, scale)
    check_rows(q, k, v, dout, True, scale, got, ref, what=f"{(B, Hq, Hkv, Sq, Skv, D)}")


def test_bwd_k_scaled_by_3():
    """A near one-hot softmax (the grouped-query workload's K x 3)."""
    B, Hq, Hkv, Sq, Skv, D = 1, 4, 1, 256, 256, 64
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, k_scale=3.0, seed=15)
    dout = make_dout(q.shape, 16)
    scale = 1.0 / math.sqrt(D)
    got = gpu_bwd(q, k, v, dout, True, scale)
    ref = oracle.attn_bwd(q, k, v, dout, True, scale)
    check_rows(q, k, v, dout, True, scale, got, ref, what=f"{(B, Hq, Hkv, Sq, Skv, D)}")


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_negative_scale(causal):
    B, Hq, Hkv, Sq, Skv, D = 1, 4, 2, 300, 300, 64
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=31)
    dout = make_dout(q.shape, 32)
    scale = -0.125
    got = gpu_bwd(q, k, v, dout, causal, scale)
    ref = oracle.attn_bwd(q, k, v, dout, causal, scale)
    check_rows(q, k, v, dout, causal, scale, got, ref, what=f"negative scale causal={causal}")


@pytest.mark.parametrize("name,deterministic", [
    ("batched_b4_h16_s2048_d128", False), ("batched_b4_h16_s2048_d128", True),
    ("gqa_b8_hq32_hkv8_s4096_d64_k3", False), ("long_b1_h32_s16384_d128", False),
    ("long_causal_b1_h32_s16384_d128", False)])
def test_bwd_workload_sampled_rows(name, deterministic):
    """Workload-size run: sampled query rows (dQ) and key rows (dK, dV) against
    the oracle, plus identities that hold at any size."""
    from attention_pipelining_gb300.synthetic import WORKLOADS, make_workload
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    dout = make_dout(q.shape, 17)
    dq, dk, dv = gpu_bwd(q, k, v, dout, w.causal, w.scale, deterministic)
    rng = np.random.default_rng(18)
    nq = w.B * w.H_q * w.S_q
    qrows = np.unique(np.concatenate([[0, nq - 1], rng.integers(0, nq, 62)]))
    bo = oracle.bwd_default()
    ref_q = bo.dq_rows(q, k, v, dout, qrows, w.causal, w.scale)
    # key rows of two groups (each needs all of its group's softmax rows)
    groups = [0, w.B * w.H_kv - 1]
    krows = np.concatenate([g * w.S_kv + rng.integers(0, w.S_kv, 8) for g in groups])
    krows = np.unique(np.concatenate([krows, [0, w.B * w.H_kv * w.S_kv - 1]]))
    ref_k, ref_v = bo.dkv_rows(q, k, v, dout, krows, w.causal, w.scale)
    got = (dq.reshape(-1, w.D)[qrows], dk.reshape(-1, w.D)[krows], dv.reshape(-1, w.D)[krows])
    check_rows(q, k, v, dout, w.causal, w.scale, got, (ref_q, ref_k, ref_v), qrows=qrows,
               krows=krows, what=name)
    # sum_j dV_j = sum of dO over the group's rows; sum_j dK_j = 0
    rep = w.H_q // w.H_kv
    do_group = dout.double().numpy().reshape(w.B, w.H_kv, rep, w.S_q, w.D).sum(axis=(2, 3))
    sv = dv.astype(np.float64).sum(axis=2)
    assert np.abs(sv - do_group).max() <= 0.02 * np.abs(do_group).max() + 0.05
    sk = dk.astype(np.float64).sum(axis=2)
    assert np.abs(sk).max() <= 0.02 * np.abs(dk).astype(np.float64).sum(axis=2).max()


def bf16_ulps(a, b):
    """Largest difference of two bf16 tensors in units of the last place of
    the larger magnitude (0 where both are equal), counting an element only
    above 2^-10 of the tensor's largest magnitude: a gradient element that is
    a sum with cancellation carries the rounding of its terms, which
    reordered fp32 additions move by more than its own last place."""
    a, b = a.float(), b.float()
    mag = torch.maximum(a.abs(), b.abs())
    floor = 2.0 ** -10 * mag.max().clamp_min(2.0 ** -126)
    ulp = torch.exp2(torch.floor(torch.log2(torch.maximum(mag, floor))) - 7)
    return ((a - b).abs() / ulp).max().item()


def test_bwd_deterministic_and_rejects_bad_workspace():
    B, Hq, Hkv, S, D = 1, 2, 1, 256, 128
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, S, S, D, seed=19))
    dout = make_dout(q.shape, 20).cuda()
    scale = 1.0 / math.sqrt(D)
    o, lse = ap.attn_fwd(q, k, v, True, scale)
    a = ap.attn_bwd(q, k, v, o, lse, dout, True, scale, deterministic=True)
    b = ap.attn_bwd(q, k, v, o, lse, dout, True, scale, deterministic=True)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    for det in (False, True):
        with pytest.raises(ap.AttnError):
            ap.attn_bwd(q, k, v, o, lse, dout, True, scale, workspace=small, deterministic=det)
    assert ap.device_status(reset=True) == 0


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_fused_dq_repeatable(causal, D):
    """The default path, 20 runs over 16 key blocks per group:
    dK and dV are the same bits every time; dQ, whose fp32 partials are added
    in L2 in an order that varies, stays within one bf16 unit in the last
    place of the first run (the fp32 sums differ only by rounding).  Against
    the deterministic path, which adds the query blocks in another order
    (without the mask the fused path starts each key block at its own query
    block), all three agree within four units in the last place."""
    B, Hq, Hkv, S = 2, 8, 2, 2048
    q, k, v = (t.cuda() for t in make_qkv(B, Hq, Hkv, S, S, D, seed=41))
    dout = make_dout(q.shape, 42).cuda()
    scale = 1.0 / math.sqrt(D)
    o, lse = ap.attn_fwd(q, k, v, causal, scale)
    ws = torch.empty(ap.bwd_workspace_bytes(B, Hq, Hkv, S, D), dtype=torch.uint8, device="cuda")
    first = [t.clone() for t in ap.attn_bwd(q, k, v, o, lse, dout, causal, scale, workspace=ws)]
    worst = 0.0
    for _ in range(20):
        dq, dk, dv = ap.attn_bwd(q, k, v, o, lse, dout, causal, scale, workspace=ws)
        assert torch.equal(dk, first[1]) and torch.equal(dv, first[2])
        worst = max(worst, bf16_ulps(dq, first[0]))
    det = ap.attn_bwd(q, k, v, o, lse, dout, causal, scale, deterministic=True)
    torch.cuda.synchronize()
    assert ap.device_status(reset=True) == 0
    print(f"fused dQ run-to-run: {worst} ulp; against the deterministic path: "
          f"dq {bf16_ulps(first[0], det[0])} dk {bf16_ulps(first[1], det[1])} "
          f"dv {bf16_ulps(first[2], det[2])} ulp")
    assert worst <= 1.0
    for got, want in zip(first, det):
        assert bf16_ulps(got, want) <= 4.0


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
    ws = torch.empty(ap.bwd_workspace_bytes(B, Hq, Hkv, S, D), dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    for _ in range(2):
        for t in host_out:
            t.fill_(0)
        ap.attn_bwd_host(*host_in, *host_out, *dev_in, *dev_out, causal, scale, ws, stream=side)
        side.synchronize()
        assert ap.device_status(reset=True) == 0
        for name, got, want in zip(("dq", "dk", "dv"), host_out, ref):
            if name == "dq":
                # the fused dQ's fp32 partials are added in a varying order
                assert bf16_ulps(got, want.cpu()) <= 1.0, name
            else:
                assert torch.equal(got, want.cpu()), name
