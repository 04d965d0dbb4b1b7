"""Split-KV forward against the fp64 oracle: decoding shapes (one query row per
head, grouped heads packed into one tile), ragged key lengths, causal and
non-causal, explicit and default split counts."""
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
    assert ap.device_status(reset=True) == 0


CASES = [
    # B, H_q, H_kv, S_q, S_kv, D, causal, splits
    (4, 32, 8, 1, 4096, 128, False, 0),      # decode, grouped heads packed 4 per tile
    (2, 32, 8, 1, 1000, 128, False, 7),      # ragged KV length
    (3, 8, 8, 1, 777, 64, False, 3),
    (1, 16, 2, 3, 2048, 128, False, 5),      # few query rows, 8 heads per group
    (1, 4, 4, 200, 1536, 128, True, 4),      # causal: late splits are empty for early rows
    (2, 8, 2, 300, 900, 64, True, 0),
    (1, 2, 2, 512, 512, 128, False, 1),      # one split = the plain forward
    (1, 4, 1, 17, 5000, 64, False, 16),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_splitkv_parity(case):
    B, Hq, Hkv, Sq, Skv, D, causal, splits = case
    q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=31)
    scale = 1.0 / math.sqrt(D)
    o, lse = ap.attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), causal, scale, num_splits=splits)
    torch.cuda.synchronize()
    o64, lse64 = oracle.attn_fwd(q, k, v, causal, scale)
    assert_parity(o.cpu(), lse.cpu(), o64, lse64, str(case))


def test_splitkv_matches_plain_forward():
    q, k, v = make_qkv(2, 8, 2, 64, 3000, 128, seed=32)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = ap.attn_fwd(qd, kd, vd, False, 0.09)
    o2, l2 = ap.attn_fwd_splitkv(qd, kd, vd, False, 0.09, num_splits=6)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (l1 - l2).abs().max().item() <= 1e-4


def test_packed_groups_in_plain_forward():
    """Grouped heads with one query row each, through the plain forward."""
    q, k, v = make_qkv(3, 16, 4, 1, 700, 64, seed=33)
    o, lse = ap.attn_fwd(q.cuda(), k.cuda(), v.cuda(), False, 0.125)
    torch.cuda.synchronize()
    o64, lse64 = oracle.attn_fwd(q, k, v, False, 0.125)
    assert_parity(o.cpu(), lse.cpu(), o64, lse64, "packed plain")


def test_one_split_on_a_grid_whose_plain_forward_splits_its_tail():
    """160 tiles of 32 KV blocks: the plain forward splits its last round
    across CTA pairs; the split-KV entry with one split must not (its tiles
    write partials for the merge kernel).  Both against the oracle."""
    q, k, v = make_qkv(1, 40, 40, 1024, 4096, 64, seed=33)
    scale = 1.0 / math.sqrt(64)
    o64, lse64 = oracle.attn_fwd(q, k, v, False, scale)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, l1 = ap.attn_fwd_splitkv(qd, kd, vd, False, scale, num_splits=1)
    o2, l2 = ap.attn_fwd(qd, kd, vd, False, scale)
    torch.cuda.synchronize()
    assert ap.device_status(reset=True) == 0
    assert_parity(o1.cpu(), l1.cpu(), o64, lse64, "split KV, one split")
    assert_parity(o2.cpu(), l2.cpu(), o64, lse64, "plain, split tail")
