"""The allocation-free split-KV entry point (for callers that cannot allocate
device memory) against the workspace entry point, through the C ABI, on two
calls in a row.  This file sorts last so that a run stopping at the first
failure has run every other test before it; it also passes on its own."""
import ctypes
import math

import pytest
import torch

import attention_pipelining_gb300 as ap
import oracle
from attention_pipelining_gb300.synthetic import make_qkv
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, k, v, causal, scale, splits):
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    rc = lib.attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), B, Hq, Hkv, Sq, Skv, D, int(causal),
                                      ctypes.c_float(scale), splits,
                                      torch.cuda.current_stream().cuda_stream)
    return rc, o, lse


def test_noalloc_matches_workspace_entry_on_two_calls():
    ap.build()
    lib = ap._load()
    assert lib.attn_splitkv_noalloc_capacity() == 16 << 20
    shapes = [
        # B, H_q, H_kv, S_q, S_kv, D, causal, splits
        (4, 32, 8, 1, 4096, 128, False, 8),
        (2, 16, 4, 5, 3000, 64, True, 0),
    ]
    for (B, Hq, Hkv, Sq, Skv, D, causal, splits), seed in zip(shapes, (41, 42)):
        qc, kc, vc = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=seed)
        q, k, v = qc.cuda(), kc.cuda(), vc.cuda()
        scale = 1.0 / math.sqrt(D)
        used = splits if splits > 0 else lib.attn_splitkv_default_splits(B, Hq, Hkv, Sq, Skv,
                                                                         int(causal))
        o_ref, lse_ref = ap.attn_fwd_splitkv(q, k, v, causal, scale, num_splits=used)
        # two calls in a row: the second finds the first one's partials in the
        # shared array and must not be affected by them
        for _ in range(2):
            rc, o, lse = _noalloc(lib, q, k, v, causal, scale, splits)
            torch.cuda.synchronize()
            assert rc == 0, ap.status_string(rc)
            # the same kernels on the same tiles with the same split count:
            # only the scratch memory differs, so the bits must agree
            assert torch.equal(o, o_ref)
            assert torch.equal(lse, lse_ref)
        o64, lse64 = oracle.attn_fwd(qc, kc, vc, causal, scale)
        assert_parity(o, lse, o64, lse64, "noalloc vs oracle")
    assert ap.device_status(reset=True) == 0


def test_noalloc_refuses_more_than_its_scratch():
    ap.build()
    lib = ap._load()
    # 64 x 64 x 64 rows x 129 floats x 16 splits is far beyond 16 MiB
    q, k, v = (torch.zeros((64, 64, 64, 128), dtype=torch.bfloat16, device="cuda") for _ in range(3))
    rc, _, _ = _noalloc(lib, q, k, v, False, 0.1, 16)
    assert rc == 2          # ATTN_ERR_UNSUPPORTED, nothing launched
