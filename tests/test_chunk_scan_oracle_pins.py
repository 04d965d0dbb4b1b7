"""Pins of the fp64 chunk-scan oracle (CPU only).

The oracle's sum out[m] = sum_{k <= m} cb[m, k] exp(dA_cs[m] - dA_cs[k]) dt[k]
x[k] is checked against things that do not share its formula: the state-space
recurrence it unrolls (h_t = exp(dA_t) h_{t-1} + dt_t x_t B_t^T, y_t = h_t C_t,
zero state at each chunk start, cb = C B^T), closed forms for a single
non-zero key and for constant cb, the invariance of the decay to a constant
shift of dA_cs, and dt = 0.  tests/test_chunk_scan_oracle_mutants.py plants
mistakes in copies of the C source and checks that these pins catch each.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_pipelining_gb300.synthetic import make_chunk_scan


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def check_recurrence(cs, seed=0, B=2, nch=2, H=4, G=2, P=3, Q=8, N=5):
    """Unrolled SSM recurrence per (batch, head, chunk), zero initial state."""
    rng = np.random.default_rng(seed)
    L = nch * Q
    x = bf16(rng.standard_normal((B, L, H, P)))
    xd = x.double().numpy()
    dt = rng.uniform(0.01, 0.3, (B, H, nch, Q)).astype(np.float32)
    A = -rng.uniform(0.5, 4.0, H)
    dA = (dt.astype(np.float64) * A[None, :, None, None]).astype(np.float32)
    # C, B per (batch, chunk, group, position); cb = C B^T given in fp32
    Cm = rng.standard_normal((B, nch, G, Q, N))
    Bm = rng.standard_normal((B, nch, G, Q, N))
    cb = np.einsum("bcgmn,bcgkn->bcgmk", Cm, Bm).astype(np.float32)
    dA_cs = np.cumsum(dA.astype(np.float64), axis=-1).astype(np.float32)
    got = cs.chunk_scan(cb, dA_cs, dt, x)
    want = np.zeros_like(got)
    rep = H // G
    for b in range(B):
        for h in range(H):
            g = h // rep
            for c in range(nch):
                state = np.zeros((P, N))
                prev = 0.0
                for t in range(Q):
                    # the per-step decay recovered from the running sums, so
                    # both sides see the same fp32 dA_cs values
                    step = float(dA_cs[b, h, c, t]) - prev
                    prev = float(dA_cs[b, h, c, t])
                    state = np.exp(step) * state + float(dt[b, h, c, t]) * np.outer(
                        xd[b, c * Q + t, h], Bm[b, c, g, t])
                    want[b, c * Q + t, h] = state @ Cm[b, c, g, t]
    # the oracle is given cb = C B^T rounded to fp32; the recurrence uses the
    # exact C and B
    assert np.allclose(got, want, rtol=1e-5, atol=1e-6), \
        f"oracle vs recurrence: {np.abs(got - want).max()}"


def check_single_key(cs, seed=1, Q=16, P=4):
    """x non-zero at one key k0 only: out[m] = cb[m,k0] e^{dA_m - dA_k0} dt_k0 x_k0
    for m >= k0 and 0 before it."""
    rng = np.random.default_rng(seed)
    B, nch, H, G = 1, 2, 2, 1
    L = nch * Q
    k0 = 5
    x = np.zeros((B, L, H, P), np.float32)
    x[0, Q + k0] = rng.standard_normal((H, P))   # in the second chunk
    x = bf16(x)
    cb = rng.standard_normal((B, nch, G, Q, Q)).astype(np.float32)
    dt = rng.uniform(0.05, 0.5, (B, H, nch, Q)).astype(np.float32)
    dA_cs = -np.cumsum(rng.uniform(0.0, 0.3, (B, H, nch, Q)), axis=-1).astype(np.float32)
    got = cs.chunk_scan(cb, dA_cs, dt, x)
    xd = x.double().numpy()
    for h in range(H):
        for m in range(Q):
            row = got[0, Q + m, h]
            if m < k0:
                assert not np.any(row), "a key after the row contributed"
            else:
                w = float(cb[0, 1, 0, m, k0]) * np.exp(float(dA_cs[0, h, 1, m]) - float(dA_cs[0, h, 1, k0])) \
                    * float(dt[0, h, 1, k0])
                assert np.allclose(row, w * xd[0, Q + k0, h], rtol=1e-13, atol=1e-15)
    assert not np.any(got[0, :Q]), "the first chunk sees the second chunk's key"


def check_constant_cb_groups(cs, Q=8, P=3):
    """dA = 0, dt = 1, cb = c_g constant per group: out[m] = c_g sum_{k<=m} x_k,
    with head h on group h // (H / G)."""
    B, nch, H, G = 1, 1, 4, 2
    rng = np.random.default_rng(2)
    x = bf16(rng.standard_normal((B, Q, H, P)))
    cb = np.empty((B, nch, G, Q, Q), np.float32)
    cb[:, :, 0] = 1.0
    cb[:, :, 1] = 2.0
    dt = np.ones((B, H, nch, Q), np.float32)
    dA_cs = np.zeros((B, H, nch, Q), np.float32)
    got = cs.chunk_scan(cb, dA_cs, dt, x)
    pref = np.cumsum(x.double().numpy(), axis=1)
    for h in range(H):
        c = 1.0 if h < 2 else 2.0
        assert np.allclose(got[:, :, h], c * pref[:, :, h], rtol=1e-14, atol=1e-14)


def check_shift_and_zero(cs, seed=3):
    cb, dA_cs, dt, x = make_chunk_scan(1, 64, 4, 8, 2, 32, seed=seed)
    base = cs.chunk_scan(cb, dA_cs, dt, x)
    shifted = cs.chunk_scan(cb, dA_cs + 1.5, dt, x)   # exactly representable shift
    assert np.allclose(base, shifted, rtol=1e-5, atol=1e-6), "decay depends on more than differences"
    zero = cs.chunk_scan(cb, dA_cs, torch.zeros_like(dt), x)
    assert not np.any(zero)


@pytest.fixture(scope="module")
def cs():
    return oracle.chunk_scan_default()


def test_recurrence(cs):
    check_recurrence(cs)


def test_single_key_and_mask(cs):
    check_single_key(cs)


def test_constant_cb_and_groups(cs):
    check_constant_cb_groups(cs)


def test_shift_invariance_and_zero_dt(cs):
    check_shift_and_zero(cs)


def test_rows_match_full(cs):
    cb, dA_cs, dt, x = make_chunk_scan(2, 512, 4, 64, 2, 256, seed=4)
    full = cs.chunk_scan(cb, dA_cs, dt, x)
    rows = np.array([0, 1, 255 * 4 + 3, 256 * 4, 2 * 512 * 4 - 1])
    got = cs.rows(cb, dA_cs, dt, x, rows)
    assert np.array_equal(got, full.reshape(-1, 64)[rows])


def test_rejects_bad_arguments(cs):
    cb, dA_cs, dt, x = make_chunk_scan(1, 64, 4, 8, 2, 32, seed=5)
    with pytest.raises(ValueError):
        cs.chunk_scan(cb[:, :1], dA_cs, dt, x)
    with pytest.raises(ValueError):
        cs.chunk_scan(cb, dA_cs[:, :2], dt, x)
