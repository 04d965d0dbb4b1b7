"""Long sequences against the fp64 oracle, on sampled rows: the forward at
131072 keys (1024 KV blocks per tile, plain and causal, grouped heads, both
head widths) and split-KV decoding over 262144 keys at the largest split
count the entry point accepts (128) and at its default one.  These run the
online softmax over far more blocks than the benchmark workloads, where the
running row sums and the rescaled accumulators have the most blocks to drift
over."""
import math

import numpy as np
import pytest
import torch

import attention_pipelining_gb300 as ap
import oracle
from attention_pipelining_gb300.synthetic import make_qkv
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ap.build()
    ap.device_status(reset=True)
    yield
    assert ap.device_status(reset=True) == 0, "a kernel wait timed out during the tests"


def sample_rows(B, Hq, Sq, n, seed):
    """Flat row indices into [B, H_q, S_q]: the first and last rows of every
    head, rows on both sides of 128-row block edges, and random rows."""
    rng = np.random.default_rng(seed)
    pos = {0, 1, 127, 128, 129, Sq // 2 - 1, Sq // 2, Sq - 129, Sq - 128, Sq - 2, Sq - 1}
    pos |= set(int(x) for x in rng.integers(0, Sq, n))
    pos = sorted(p for p in pos if 0 <= p < Sq)
    return np.array([(b * Hq + h) * Sq + i for b in range(B) for h in range(Hq) for i in pos],
                    np.int64)


LONG = [
    # B, H_q, H_kv, S, D, causal
    (1, 2, 1, 131072, 128, False),
    (1, 2, 1, 131072, 128, True),
    (1, 4, 2, 65536, 64, True),
]


@pytest.mark.parametrize("case", LONG, ids=[str(c) for c in LONG])
def test_long_sequence_sampled_rows(case):
    B, Hq, Hkv, S, D, causal = case
    q, k, v = make_qkv(B, Hq, Hkv, S, S, D, seed=41)
    scale = 1.0 / math.sqrt(D)
    o, lse = ap.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal, scale)
    torch.cuda.synchronize()
    o, lse = o.cpu(), lse.cpu()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    rows = sample_rows(B, Hq, S, 24, seed=42)
    o64, lse64 = oracle.attn_rows(q, k, v, rows, causal, scale)
    idx = torch.from_numpy(rows)
    assert_parity(o.reshape(-1, D)[idx], lse.reshape(-1)[idx], o64, lse64, str(case))


DECODE = (1, 32, 8, 1, 262144, 128)   # B, H_q, H_kv, S_q, S_kv, D


@pytest.fixture(scope="module")
def decode_case():
    """Inputs on the device and the oracle's result, made once."""
    B, Hq, Hkv, Sq, Skv, D = DECODE
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=43)
    scale = 1.0 / math.sqrt(D)
    o64, lse64 = oracle.attn_fwd(q, k, v, False, scale)
    return q.cuda(), k.cuda(), v.cuda(), scale, o64, lse64


@pytest.mark.parametrize("splits", [128, 0], ids=["max_splits", "default_splits"])
def test_long_decode_splitkv(decode_case, splits):
    """One query row per head over 262144 keys (grouped heads packed per
    tile): every row against the oracle."""
    q, k, v, scale, o64, lse64 = decode_case
    o, lse = ap.attn_fwd_splitkv(q, k, v, False, scale, num_splits=splits)
    torch.cuda.synchronize()
    assert_parity(o.cpu(), lse.cpu(), o64, lse64, f"decode {DECODE} splits={splits}")
