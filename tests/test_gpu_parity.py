"""The CUDA path against the fp64 oracle, element by element on small and odd
shapes, and on sampled rows at the full sizes of the benchmark workloads."""
import math

import numpy as np
import pytest
import torch

import attention_pipelining_gb300 as ap
import oracle
from attention_pipelining_gb300.synthetic import WORKLOADS, make_qkv, make_workload
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ap.build()
    ap.device_status(reset=True)
    yield
    assert ap.device_status(reset=True) == 0, "a kernel wait timed out during the tests"


def run_gpu(q, k, v, causal, scale):
    o, lse = ap.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal, scale)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


SMALL = [
    # B, H_q, H_kv, S_q, S_kv, D, causal, k_scale
    (1, 1, 1, 256, 256, 64, False, 1.0),   # the single-head workload, full size
    (1, 2, 2, 128, 128, 128, False, 1.0),
    (1, 2, 2, 128, 128, 128, True, 1.0),
    (2, 4, 4, 1024, 1024, 128, False, 1.0),
    (2, 4, 4, 1024, 1024, 128, True, 1.0),
    (2, 8, 2, 512, 512, 64, True, 3.0),    # grouped heads, K x 3
    (1, 4, 1, 512, 512, 128, False, 1.0),
    (3, 2, 1, 130, 130, 128, True, 1.0),
    (1, 2, 2, 200, 77, 128, True, 1.0),    # S_q > S_kv
    (1, 2, 2, 200, 77, 128, False, 1.0),
    (1, 2, 2, 77, 300, 64, True, 1.0),     # S_q < S_kv
    (1, 2, 2, 77, 300, 64, False, 1.0),
    (1, 3, 3, 40, 1, 128, False, 1.0),     # a single key
    (1, 3, 3, 40, 1, 64, True, 1.0),
    # 160 tiles of 32 KV blocks on 152 SMs: the last round's 8 tiles are
    # split across CTA pairs (each half of the KV blocks, merged through the
    # cluster); plain heads and grouped heads
    (1, 40, 40, 1024, 4096, 64, False, 1.0),
    (10, 8, 2, 512, 4096, 64, False, 1.0),
]
ODD_S = [1, 17, 127, 129, 255, 257, 383, 513]


def _check(B, Hq, Hkv, Sq, Skv, D, causal, kscale, seed=0):
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, k_scale=kscale, seed=seed)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_gpu(q, k, v, causal, scale)
    o64, lse64 = oracle.attn_fwd(q, k, v, causal, scale)
    return assert_parity(o, lse, o64, lse64, f"{(B, Hq, Hkv, Sq, Skv, D, causal, kscale)}")


@pytest.mark.parametrize("case", SMALL, ids=[str(c) for c in SMALL])
def test_small_shapes(case):
    _check(*case)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", ODD_S)
def test_ragged_lengths(S, causal, D):
    _check(1, 2, 1, S, S, D, causal, 1.0, seed=S)


def test_v_ones_gives_ones():
    q, k, _ = make_qkv(1, 4, 2, 300, 300, 128, seed=3)
    v = torch.ones((1, 2, 300, 128), dtype=torch.bfloat16)
    for causal in (False, True):
        o, _ = run_gpu(q, k, v, causal, 1 / math.sqrt(128))
        assert np.abs(o.double().numpy() - 1.0).max() <= 1e-2


def test_zero_scale_gives_mean_of_v():
    q, k, v = make_qkv(1, 2, 2, 260, 260, 64, seed=4)
    for causal in (False, True):
        o, lse = run_gpu(q, k, v, causal, 0.0)
        o64, lse64 = oracle.attn_fwd(q, k, v, causal, 0.0)
        assert_parity(o, lse, o64, lse64, f"scale=0 causal={causal}")


@pytest.mark.parametrize("case", [
    # B, H_q, H_kv, S_q, S_kv, D, causal, scale
    (1, 2, 2, 300, 300, 128, False, -0.125),
    (1, 2, 2, 300, 300, 128, True, -0.125),
    (2, 8, 2, 512, 512, 64, True, -1.0 / 8),     # grouped heads
    (1, 4, 1, 77, 1000, 64, False, -0.4),        # a large negative scale, ragged
    (1, 2, 2, 260, 260, 64, True, -0.0),
])
def test_negative_scale(case):
    """The definition admits any real scale: with a negative one the row max
    is the smallest raw score times the scale, and masked keys must still
    drop out."""
    B, Hq, Hkv, Sq, Skv, D, causal, scale = case
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=80 + Sq)
    o, lse = run_gpu(q, k, v, causal, scale)
    o64, lse64 = oracle.attn_fwd(q, k, v, causal, scale)
    assert_parity(o, lse, o64, lse64, f"negative scale {case}")


def test_negative_scale_split_tail():
    """A negative scale through the split tail (the pair merge by LSE)."""
    q, k, v = make_qkv(1, 40, 40, 1024, 4096, 64, seed=81)
    o, lse = run_gpu(q, k, v, False, -0.125)
    o64, lse64 = oracle.attn_fwd(q, k, v, False, -0.125)
    assert_parity(o, lse, o64, lse64, "negative scale, split tail")


def test_deterministic():
    q, k, v = make_qkv(2, 4, 2, 700, 700, 128, seed=9)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = ap.attn_fwd(q, k, v, True, 0.1)
    o2, l2 = ap.attn_fwd(q, k, v, True, 0.1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_split_tail_repeatable():
    """A grid whose last round is split across CTA pairs (each CTA's
    partial for the sub-tile its partner writes crosses by a bulk copy into
    the partner's shared memory), run 20 times: every launch gives the same
    bits and no wait runs out, so the exchange has no race that shows up
    from one launch to the next."""
    q, k, v = make_qkv(1, 40, 40, 1024, 4096, 64, seed=61)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o0, l0 = ap.attn_fwd(qd, kd, vd, False, 0.125)
    outs = [ap.attn_fwd(qd, kd, vd, False, 0.125) for _ in range(20)]
    torch.cuda.synchronize()
    assert ap.device_status(reset=True) == 0
    for o, lse in outs:
        assert torch.equal(o, o0) and torch.equal(lse, l0)


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("D", [64, 128])
def test_split_tail_ragged_rows(D):
    """A split tail that holds ragged tiles: one head per row group, S_q = 400
    (a group's second tile has rows 256..399, its second sub-tile only 16
    rows), 32 KV blocks, and SMs / 2 + 4 heads, so the grid's last round is
    the last four groups' eight tiles, each split across a CTA pair."""
    sms = _sms()
    H, Sq, Skv = sms // 2 + 4, 400, 4096
    assert ap.fwd_tail_pairs(1, H, H, Sq, Skv, D, False) == 8
    _check(1, H, H, Sq, Skv, D, False, 1.0, seed=70 + D)


@pytest.mark.parametrize("D", [64, 128])
def test_split_tail_one_subtile_and_ragged_keys(D):
    """A split tail at the shortest split tiles (S_kv = 2000: 16 KV blocks,
    the last one ragged, so each half holds 8 and the second half the ragged
    block) whose tiles alternate between two sub-tiles (one CTA of the pair
    writes each) and one (S_q = 384: a group's second tile is 128 rows, so
    the second CTA only sends and the first only writes)."""
    sms = _sms()
    H, Sq, Skv = sms // 2 + 4, 384, 2000
    assert ap.fwd_tail_pairs(1, H, H, Sq, Skv, D, False) == 8
    _check(1, H, H, Sq, Skv, D, False, 1.0 / math.sqrt(D), seed=90 + D)


def test_split_tail_plan():
    """The shapes the split-tail tests rely on do split their tail; causal,
    short-KV and whole-round shapes do not."""
    sms = _sms()
    assert ap.fwd_tail_pairs(1, 40, 40, 1024, 4096, 64, False) == 160 - sms
    assert ap.fwd_tail_pairs(10, 8, 2, 512, 4096, 64, False) == 160 - sms
    assert ap.fwd_tail_pairs(1, 32, 32, 16384, 16384, 128, False) == 2048 % sms
    assert ap.fwd_tail_pairs(1, 40, 40, 1024, 4096, 64, True) == 0       # causal
    assert ap.fwd_tail_pairs(1, 40, 40, 1024, 2048, 64, False) == 160 - sms  # 16 KV blocks
    assert ap.fwd_tail_pairs(4, 16, 16, 2048, 2048, 128, False) == 512 % sms
    assert ap.fwd_tail_pairs(1, 40, 40, 1024, 1920, 64, False) == 0      # 15 KV blocks
    assert ap.fwd_tail_pairs(1, sms // 2, sms // 2, 512, 4096, 64, False) == 0  # whole rounds


def test_side_stream_and_host_entry():
    q, k, v = make_qkv(1, 2, 2, 300, 300, 128, seed=5)
    scale = 1 / math.sqrt(128)
    o64, lse64 = oracle.attn_fwd(q, k, v, False, scale)
    s = torch.cuda.Stream()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        o, lse = ap.attn_fwd(qd, kd, vd, False, scale, stream=s)
    s.synchronize()
    assert_parity(o, lse, o64, lse64, "side stream")
    # host buffers in, host buffers out
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    oh = torch.empty_like(q).pin_memory()
    lh = torch.empty((1, 2, 300), dtype=torch.float32).pin_memory()
    od, ld = torch.empty_like(qd), torch.empty((1, 2, 300), dtype=torch.float32, device="cuda")
    ap.attn_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, False, scale)
    torch.cuda.synchronize()
    assert_parity(oh, lh, o64, lse64, "host entry")


HOST_PIPE_SHAPES = [
    # B, H_q, H_kv, S, D, causal: copies longer than the kernels (8 chunks)
    (2, 8, 4, 4096, 128, False),
    (2, 8, 4, 4096, 128, True),
    # kernels longer than the copies: 16 chunks of one row group each
    (1, 16, 16, 16384, 128, False),
]


@pytest.mark.parametrize("shape", HOST_PIPE_SHAPES, ids=[str(c) for c in HOST_PIPE_SHAPES])
def test_host_entry_pipelined_matches_device(shape):
    """Inputs of 32 MiB or more: the host entry splits the row groups into
    chunks whose copies overlap the other chunks' kernels (on the caller's
    side stream here).  In these shapes neither the one call (256 and 1024
    tiles) nor a chunk (fewer tiles than SMs) splits its last round across
    CTA pairs, so every row is computed by the same tiles and the outputs
    are bit-identical to one attn_fwd call."""
    B, Hq, Hkv, S, D, causal = shape
    q, k, v = make_qkv(B, Hq, Hkv, S, S, D, seed=7)
    scale = 1 / math.sqrt(D)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_ref, lse_ref = ap.attn_fwd(qd, kd, vd, causal, scale)
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    oh = torch.full_like(q, float("nan")).pin_memory()
    lh = torch.full((B, Hq, S), float("nan"), dtype=torch.float32).pin_memory()
    od = torch.full_like(qd, float("nan"))
    ld = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device="cuda")
    qd2, kd2, vd2 = torch.zeros_like(qd), torch.zeros_like(kd), torch.zeros_like(vd)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    for _ in range(2):  # twice: the second call reuses the cached streams and events
        ap.attn_fwd_host(qh, kh, vh, oh, lh, qd2, kd2, vd2, od, ld, causal, scale, stream=s)
    s.synchronize()
    assert ap.device_status(reset=True) == 0
    assert torch.equal(oh, o_ref.cpu())
    assert torch.equal(lh, lse_ref.cpu())


def test_host_entry_where_one_call_splits_its_tail():
    """512 tiles in one call (its last 56 split across CTA pairs) against
    chunks of 32 tiles (none split): the same result within the rounding of
    the split tiles' merge, and parity against the oracle on sampled rows."""
    B, Hq, Hkv, S, D = 1, 32, 32, 4096, 128
    q, k, v = make_qkv(B, Hq, Hkv, S, S, D, seed=71)
    scale = 1 / math.sqrt(D)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_ref, lse_ref = ap.attn_fwd(qd, kd, vd, False, scale)
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    oh = torch.empty_like(q).pin_memory()
    lh = torch.empty((B, Hq, S), dtype=torch.float32).pin_memory()
    od, ld = torch.empty_like(qd), torch.empty((B, Hq, S), dtype=torch.float32, device="cuda")
    ap.attn_fwd_host(qh, kh, vh, oh, lh, torch.empty_like(qd), torch.empty_like(kd),
                     torch.empty_like(vd), od, ld, False, scale)
    torch.cuda.synchronize()
    assert ap.device_status(reset=True) == 0
    assert (oh.float() - o_ref.cpu().float()).abs().max().item() <= 2e-2
    assert (lh - lse_ref.cpu()).abs().max().item() <= 1e-4
    rng = np.random.default_rng(72)
    rows = np.unique(np.concatenate([rng.integers(0, Hq * S, 48),
                                     Hq * S - 1 - rng.integers(0, 2048, 16)]))
    o64, lse64 = oracle.attn_rows(q, k, v, rows, False, scale)
    idx = torch.from_numpy(rows)
    assert_parity(oh.reshape(-1, D)[idx], lh.reshape(-1)[idx], o64, lse64, "host, split tail")
    assert_parity(o_ref.cpu().reshape(-1, D)[idx], lse_ref.cpu().reshape(-1)[idx], o64, lse64,
                  "device, split tail")


def _sample_rows(w, n_heads=6, seed=0):
    """Flat row indices into [B, H_q, S_q]: tile edges, sequence ends, random rows."""
    rng = np.random.default_rng(seed)
    heads = {(0, 0), (w.B - 1, w.H_q - 1)}
    while len(heads) < min(n_heads, w.B * w.H_q):
        heads.add((int(rng.integers(w.B)), int(rng.integers(w.H_q))))
    pos = {0, 1, 127, 128, 255, 256, w.S_q - 1, w.S_q - 2, w.S_q // 2}
    pos |= set(int(x) for x in rng.integers(0, w.S_q, 24))
    pos = sorted(p for p in pos if 0 <= p < w.S_q)
    return np.array([(b * w.H_q + h) * w.S_q + i for (b, h) in sorted(heads) for i in pos], np.int64)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_sampled_rows(name):
    """Full-size workloads in the benchmark's launch configuration, checked on
    sampled rows that the oracle computes one by one."""
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    if w.path == "splitkv":
        o, lse = ap.attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), w.causal, w.scale)
        torch.cuda.synchronize()
        o, lse = o.cpu(), lse.cpu()
    else:
        o, lse = run_gpu(q, k, v, w.causal, w.scale)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    rows = _sample_rows(w)
    o64, lse64 = oracle.attn_rows(q, k, v, rows, w.causal, w.scale)
    og = o.reshape(-1, w.D)[torch.from_numpy(rows)]
    lg = lse.reshape(-1)[torch.from_numpy(rows)]
    assert_parity(og, lg, o64, lse64, name)


FULL_HEAD = [n for n in ("long_b1_h32_s16384_d128", "long_causal_b1_h32_s16384_d128",
                         "causal_b2_h16_s8192_d128", "batched_b4_h16_s2048_d128",
                         "gqa_b8_hq32_hkv8_s4096_d64_k3", "single_head_b1_h1_s256_d64")]


@pytest.mark.parametrize("name", FULL_HEAD)
def test_full_size_one_whole_head(name):
    """Full-size workloads: every row of one query head, element by element.
    The head is the last one of the last batch entry: its tiles come last in
    the tile list, so it is wholly inside the
    split tail (every one of its tiles split across a CTA pair) on the
    non-causal long sequence and batched shapes, and on the
    grouped-query shape it is the last head of the last KV group."""
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    o, lse = run_gpu(q, k, v, w.causal, w.scale)
    if name in ("long_b1_h32_s16384_d128", "batched_b4_h16_s2048_d128"):
        tiles = w.B * w.H_q * w.S_q // 256
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        tail = ap.fwd_tail_pairs(w.B, w.H_q, w.H_kv, w.S_q, w.S_kv, w.D, w.causal)
        assert tail == tiles % sms and tail >= w.S_q // 256   # the last head is all tail
    b, h = w.B - 1, w.H_q - 1
    first = (b * w.H_q + h) * w.S_q
    rows = np.arange(first, first + w.S_q)
    o64, lse64 = oracle.attn_rows(q, k, v, rows, w.causal, w.scale)
    assert_parity(o[b, h], lse[b, h], o64.reshape(w.S_q, w.D), lse64.reshape(w.S_q), name)


def test_trace_instantiation_matches_and_stamps():
    """The trace instantiation computes the same result and stamps every role
    (S = 512: every traced tile has both 128-row sub-tiles)."""
    q, k, v = make_qkv(1, 2, 2, 512, 600, 128, seed=8)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = ap.attn_fwd(qd, kd, vd, False, 0.09)
    o2, lse2, tr = ap.attn_fwd_trace(qd, kd, vd, False, 0.09, ctas=2)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    n = (600 + 127) // 128
    t = tr.numpy()
    assert tr.shape[0] == 2
    for ev in ("sm0_wake", "sm0_done", "sm1_wake", "sm1_done", "mma_pv0", "mma_pv1",
               "mma_s0", "mma_s1", "load_k", "load_v"):
        e = ap.TRACE_EVENTS.index(ev)
        assert (t[:, e, :n] > 0).all(), ev
    sm0w, sm0d = t[:, 0, :n], t[:, 2, :n]
    assert (sm0d >= sm0w).all() and (np.diff(sm0w, axis=1) > 0).all()
