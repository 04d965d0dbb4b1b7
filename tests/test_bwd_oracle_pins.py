"""Pins of the fp64 backward oracle (CPU only).

The oracle's dQ, dK, dV are checked against things that do not share its
formulas: central finite differences of the forward definition (L = sum O dO
differentiated numerically), torch's float64 autograd through an explicit
softmax attention (a library special case), and identities the exact
gradients satisfy:
  * sum_j dK_j = 0 per key/value head (each row of dS sums to zero),
  * sum_j dV_j = sum of dO over the head group's rows,
  * sum_i q_i . dQ_i = sum_j k_j . dK_j (both are dL/dalpha for s -> alpha s),
  * sum_j v_j . dV_j = L = sum O . dO (L is linear in V).
tests/test_bwd_oracle_mutants.py plants mistakes in copies of the C source and
checks that these pins catch each.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_pipelining_gb300.synthetic import make_qkv

SHAPES = [
    # B, H_q, H_kv, S_q, S_kv, D, causal
    (1, 2, 1, 4, 5, 3, False),
    (1, 2, 1, 5, 5, 4, True),
    (2, 4, 2, 3, 6, 3, True),
    (1, 1, 1, 6, 3, 2, True),   # S_kv < S_q: later rows see every key
    (1, 3, 3, 1, 7, 5, False),
]


def _rand(shape, seed):
    B, Hq, Hkv, Sq, Skv, D, _ = shape
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, Sq, D))
    k = rng.standard_normal((B, Hkv, Skv, D))
    v = rng.standard_normal((B, Hkv, Skv, D))
    do = rng.standard_normal((B, Hq, Sq, D))
    return q, k, v, do


def loss(bo, q, k, v, do, causal, scale):
    o, _ = bo.attn_fwd_f64(q, k, v, causal, scale)
    return float((o * do).sum())


def finite_difference(bo, q, k, v, do, causal, scale, h=1e-6):
    """Central differences of L with respect to every element of q, k, v."""
    grads = []
    for which in range(3):
        args = [q.copy(), k.copy(), v.copy()]
        x = args[which]
        g = np.empty_like(x)
        flat, gflat = x.reshape(-1), g.reshape(-1)
        for t in range(flat.size):
            keep = flat[t]
            flat[t] = keep + h
            lp = loss(bo, *args, do, causal, scale)
            flat[t] = keep - h
            lm = loss(bo, *args, do, causal, scale)
            flat[t] = keep
            gflat[t] = (lp - lm) / (2 * h)
        grads.append(g)
    return grads


def check_finite_difference(bo, shape, seed=0, scale=0.8):
    q, k, v, do = _rand(shape, seed)
    causal = shape[-1]
    dq, dk, dv = bo.attn_bwd_f64(q, k, v, do, causal, scale)
    fq, fk, fv = finite_difference(bo, q, k, v, do, causal, scale)
    for name, a, b in (("dq", dq, fq), ("dk", dk, fk), ("dv", dv, fv)):
        err = np.abs(a - b).max()
        assert err <= 2e-7 * max(1.0, np.abs(b).max()), f"{name} vs finite differences: {err}"


def check_torch(bo, shape, seed=1, scale=0.6):
    q, k, v, do = _rand(shape, seed)
    B, Hq, Hkv, Sq, Skv, D, causal = shape
    dq, dk, dv = bo.attn_bwd_f64(q, k, v, do, causal, scale)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    rep = Hq // Hkv
    kk = tk.repeat_interleave(rep, dim=1)
    vv = tv.repeat_interleave(rep, dim=1)
    # explicit fp64 attention with a top-left causal mask (key j <= query i)
    s = torch.einsum("bhid,bhjd->bhij", tq, kk) * scale
    if causal:
        mask = torch.ones(Sq, Skv, dtype=torch.bool).tril()
        s = s.masked_fill(~mask, float("-inf"))
    o = torch.softmax(s, dim=-1) @ vv
    (o * torch.tensor(do)).sum().backward()
    for name, a, b in (("dq", dq, tq.grad), ("dk", dk, tk.grad), ("dv", dv, tv.grad)):
        err = np.abs(a - b.numpy()).max()
        assert err <= 1e-12 * max(1.0, np.abs(a).max()), f"{name} vs torch autograd: {err}"


def check_identities(bo, shape, seed=2, scale=0.9):
    q, k, v, do = _rand(shape, seed)
    B, Hq, Hkv, Sq, Skv, D, causal = shape
    dq, dk, dv = bo.attn_bwd_f64(q, k, v, do, causal, scale)
    o, _ = bo.attn_fwd_f64(q, k, v, causal, scale)
    rep = Hq // Hkv
    tol = 1e-12
    # each row of dS sums to zero
    assert np.abs(dk.sum(axis=2)).max() <= tol * max(1.0, np.abs(dk).max())
    # dV collects dO through a stochastic P
    do_group = do.reshape(B, Hkv, rep, Sq, D).sum(axis=(2, 3))
    assert np.abs(dv.sum(axis=2) - do_group).max() <= tol * max(1.0, np.abs(do_group).max())
    # scaling every score: dL/dalpha seen from Q and from K
    lhs, rhs = float((q * dq).sum()), float((k * dk).sum())
    assert abs(lhs - rhs) <= tol * max(1.0, abs(lhs))
    # linearity in V
    lv, lo = float((v * dv).sum()), float((o * do).sum())
    assert abs(lv - lo) <= tol * max(1.0, abs(lo))


@pytest.fixture(scope="module")
def bo():
    return oracle.bwd_default()


@pytest.mark.parametrize("shape", SHAPES)
def test_finite_differences(bo, shape):
    check_finite_difference(bo, shape)


@pytest.mark.parametrize("shape", SHAPES)
def test_torch_autograd(bo, shape):
    check_torch(bo, shape)


@pytest.mark.parametrize("shape", SHAPES)
def test_identities(bo, shape):
    check_identities(bo, shape)


def test_zero_upstream_gradient(bo):
    q, k, v, do = _rand(SHAPES[2], 3)
    for g in bo.attn_bwd_f64(q, k, v, np.zeros_like(do), True, 0.5):
        assert not np.any(g)


def test_bf16_entry_equals_widened_f64(bo):
    """The bf16 entry point is the fp64 one on exactly widened inputs."""
    q, k, v = make_qkv(2, 4, 2, 33, 40, 8, seed=4)
    g = torch.Generator().manual_seed(5)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    a = bo.attn_bwd(q, k, v, do, True, 0.35)
    b = bo.attn_bwd_f64(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                        do.double().numpy(), True, 0.35)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_row_entries_match_full(bo):
    """Sampled query rows (dQ) and key rows (dK, dV) equal the full result."""
    B, Hq, Hkv, Sq, Skv, D = 2, 4, 2, 37, 45, 16
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=6)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    scale = 1 / math.sqrt(D)
    for causal in (False, True):
        dq, dk, dv = bo.attn_bwd(q, k, v, do, causal, scale)
        qrows = np.array([0, 5, 36, 37 * 3 + 11, B * Hq * Sq - 1])
        got = bo.dq_rows(q, k, v, do, qrows, causal, scale)
        assert np.allclose(got, dq.reshape(-1, D)[qrows], rtol=1e-13, atol=1e-14)
        krows = np.array([0, 44, 45 + 3, 2 * 45 + 20, B * Hkv * Skv - 1])
        gk, gv = bo.dkv_rows(q, k, v, do, krows, causal, scale)
        assert np.allclose(gk, dk.reshape(-1, D)[krows], rtol=1e-12, atol=1e-13)
        assert np.allclose(gv, dv.reshape(-1, D)[krows], rtol=1e-12, atol=1e-13)


def test_rejects_bad_arguments(bo):
    q, k, v, do = _rand(SHAPES[0], 0)
    with pytest.raises(ValueError):
        bo.attn_bwd_f64(q, k, v, do[:, :, :, :2], False, 1.0)
    q3 = np.zeros((1, 3, 4, 3))   # 3 query heads cannot share 2 key/value heads
    k2 = np.zeros((1, 2, 5, 3))
    with pytest.raises(ValueError):
        bo.attn_bwd_f64(q3, k2, k2, q3, False, 1.0)
