"""Parity of the CUDA chunk scan (chunk_scan_fwd) against the fp64 oracle.

Tolerance (derived, the pages fix none): each output element is a sum of up
to Q products whose scaled-cb factor is rounded to bf16 (2^-9 relative) with
bf16 x, accumulated in fp32, then rounded to bf16 once more; terms of both
signs partly cancel, so the error is measured against the tensor's scale:
relative Frobenius error <= 2^-7 and every element within 2^-5 of the
largest magnitude.
"""
import numpy as np
import pytest
import torch

import attention_pipelining_gb300 as ap
import oracle
from attention_pipelining_gb300.synthetic import (CHUNK_SCAN_WORKLOADS, make_chunk_scan,
                                                  make_chunk_scan_workload)

pytestmark = pytest.mark.gpu

REL_FRO = 2.0 ** -7
REL_MAX = 2.0 ** -5


@pytest.fixture(scope="module", autouse=True)
def _built():
    ap.build()
    ap.device_status(reset=True)
    yield


def assert_close(name, got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    err = np.abs(got - ref)
    fro = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)
    mx = err.max() / max(np.abs(ref).max(), 1e-30)
    assert fro <= REL_FRO and mx <= REL_MAX, (
        f"{name}: relative Frobenius error {fro:.3e} (<= {REL_FRO:.3e}), "
        f"max error / max |ref| {mx:.3e} (<= {REL_MAX:.3e})")


def run(cb, dA_cs, dt, x):
    out = ap.chunk_scan(cb.cuda(), dA_cs.cuda(), dt.cuda(), x.cuda())
    torch.cuda.synchronize()
    assert ap.device_status(reset=True) == 0
    return out.float().cpu().numpy()


SHAPES = [
    # B, L, H, P, G, Q
    (1, 256, 4, 64, 1, 256),
    (2, 512, 4, 64, 2, 256),
    (1, 384, 3, 64, 1, 128),
    (2, 256, 6, 64, 3, 128),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_chunk_scan_matches_oracle(shape):
    B, L, H, P, G, Q = shape
    cb, dA_cs, dt, x = make_chunk_scan(B, L, H, P, G, Q, seed=31)
    got = run(cb, dA_cs, dt, x)
    ref = oracle.chunk_scan_default().chunk_scan(cb, dA_cs, dt, x)
    assert_close("out", got, ref)


def test_chunk_scan_single_key_and_zero_dt():
    """Closed forms on the GPU: dt = 0 gives 0; x non-zero at one key gives
    nothing before that key within its chunk and nothing in other chunks."""
    B, L, H, P, G, Q = 1, 512, 2, 64, 1, 256
    cb, dA_cs, dt, x = make_chunk_scan(B, L, H, P, G, Q, seed=32)
    assert not np.any(run(cb, dA_cs, torch.zeros_like(dt), x))
    x1 = torch.zeros_like(x)
    k0 = Q + 70
    x1[0, k0] = x[0, k0]
    got = run(cb, dA_cs, dt, x1)
    assert not np.any(got[0, :k0])
    ref = oracle.chunk_scan_default().chunk_scan(cb, dA_cs, dt, x1)
    assert_close("single key", got, ref)


@pytest.mark.parametrize("name", ["chunkscan_b1_s8192"])
def test_chunk_scan_workload_sampled_rows(name):
    w = CHUNK_SCAN_WORKLOADS[name]
    cb, dA_cs, dt, x = make_chunk_scan_workload(w)
    got = run(cb, dA_cs, dt, x)
    rng = np.random.default_rng(33)
    total = w.B * w.L * w.H
    rows = np.unique(np.concatenate([[0, total - 1], rng.integers(0, total, 400)]))
    ref = oracle.chunk_scan_default().rows(cb, dA_cs, dt, x, rows)
    assert_close("rows", got.reshape(-1, w.P)[rows], ref)


def test_chunk_scan_rejects_bad_arguments():
    cb, dA_cs, dt, x = (t.cuda() for t in make_chunk_scan(1, 256, 2, 64, 1, 256, seed=34))
    with pytest.raises(ap.AttnError):   # P = 32 is not supported
        ap.chunk_scan(cb, dA_cs, dt, x[..., :32].contiguous())
    assert ap.device_status(reset=True) == 0


def test_chunk_scan_rising_decay():
    """dA_cs that rises somewhere in a chunk (not Mamba2's case, where dt > 0
    and A < 0 make it fall), or falls by 100 within 16 keys, next to heads
    where it falls gently, in one launch: where it rises the kernel keeps one
    exponential per (row, key), elsewhere it splits the decay into a row and a
    key factor."""
    B, L, H, P, G, Q = 2, 512, 8, 64, 2, 256
    cb, dA_cs, dt, x = make_chunk_scan(B, L, H, P, G, Q, seed=35)
    g = torch.Generator().manual_seed(36)
    walk = torch.cumsum(0.05 * torch.randn(B, H, L // Q, Q, generator=g), dim=-1)
    dA_cs[:, 1] = walk[:, 1]                     # a random walk: rises and falls
    dA_cs[0, 2, 1, 100:] += 0.3                  # one step up at key 100 of one chunk
    dA_cs[1, 6, 0, 255] += 1e-3                  # a rise at the chunk's last key only
    dA_cs[1, 3, 0, 40:] -= 100.0                 # a fall of 100 inside one 16-key portion
    got = run(cb, dA_cs, dt, x)
    ref = oracle.chunk_scan_default().chunk_scan(cb, dA_cs, dt, x)
    assert_close("out", got, ref)


@pytest.mark.parametrize("shape", [(4, 8192, 64, 64, 1, 256)], ids=["b4_s8192"])
def test_chunk_scan_large_head_blocks_sampled_rows(shape):
    """Enough row tiles that a CTA takes 32 heads; sampled rows."""
    B, L, H, P, G, Q = shape
    cb, dA_cs, dt, x = make_chunk_scan(B, L, H, P, G, Q, seed=37)
    got = run(cb, dA_cs, dt, x)
    rng = np.random.default_rng(38)
    total = B * L * H
    rows = np.unique(np.concatenate([[0, total - 1], rng.integers(0, total, 400)]))
    ref = oracle.chunk_scan_default().rows(cb, dA_cs, dt, x, rows)
    assert_close("rows", got.reshape(-1, P)[rows], ref)


def test_chunk_scan_headline_workload_sampled_rows():
    """The 64 x 8192 workload as the benchmark times it (inputs drawn on the
    device): sampled rows against the oracle."""
    w = CHUNK_SCAN_WORKLOADS["chunkscan_b64_s8192"]
    cb, dA_cs, dt, x = make_chunk_scan_workload(w, device="cuda")
    out = ap.chunk_scan(cb, dA_cs, dt, x)
    torch.cuda.synchronize()
    assert ap.device_status(reset=True) == 0
    rng = np.random.default_rng(39)
    total = w.B * w.L * w.H
    rows = np.unique(np.concatenate([[0, total - 1], rng.integers(0, total, 300)]))
    got = out.reshape(-1, w.P)[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    cpu = [t.cpu() for t in (cb, dA_cs, dt, x)]
    del cb, dA_cs, dt, x, out
    ref = oracle.chunk_scan_default().rows(*cpu, rows)
    assert_close("rows", got, ref)


@pytest.mark.parametrize("shape", [(4, 8192, 64, 64, 1, 256), (1, 512, 4, 64, 1, 256)],
                         ids=["b4_s8192_chunked", "b1_s512_one_chunk"])
def test_chunk_scan_host_entry_matches_device_entry(shape):
    """chunk_scan_fwd_host (pinned host buffers; the first shape is cut into
    chunks of batch entries on the entry's own streams) gives the same bits
    as chunk_scan_fwd, called twice in a row on a side stream."""
    B, L, H, P, G, Q = shape
    cb, dA_cs, dt, x = make_chunk_scan(B, L, H, P, G, Q, seed=51)
    dev = [t.cuda() for t in (cb, dA_cs, dt, x)]
    ref = ap.chunk_scan(*dev)
    torch.cuda.synchronize()
    host_in = [t.pin_memory() for t in (cb, dA_cs, dt, x)]
    host_out = torch.empty(x.shape, dtype=x.dtype).pin_memory()
    dev_in = [torch.empty_like(t) for t in dev]
    dev_out = torch.empty_like(ref)
    side = torch.cuda.Stream()
    for _ in range(2):
        host_out.fill_(0)
        ap.chunk_scan_host(*host_in, host_out, *dev_in, dev_out, stream=side)
        side.synchronize()
        assert ap.device_status(reset=True) == 0
        assert torch.equal(host_out, ref.cpu())
