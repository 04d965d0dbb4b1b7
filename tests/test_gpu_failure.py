"""Failure detection on the GPU without a fault: a kernel wait is made to run
out (a signal is withheld that nothing else sets: one "P ready", the split
tail's hand-off between the CTAs of a cluster, or the backward's "P^T, dS^T
stored") with a short wait budget; the
kernel must return, the device status word must read ATTN_ERR_TIMEOUT, and
the same CUDA context must keep working."""
import math

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
    ap.device_status(reset=True)


@pytest.mark.parametrize("D", [64, 128])
def test_wait_runs_out_and_context_survives(D):
    q, k, v = make_qkv(1, 2, 2, 512, 512, D, seed=21)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    assert ap.device_status(reset=True) == 0
    ap.fwd_timeout_test(qd, kd, vd, False, scale, drop_block=1, wait_budget_ns=20_000_000)
    torch.cuda.synchronize()
    assert ap.device_status(reset=True) == 5        # ATTN_ERR_TIMEOUT
    # the context is intact: a normal call right after is correct and clean
    o, lse = ap.attn_fwd(qd, kd, vd, False, scale)
    torch.cuda.synchronize()
    o64, lse64 = oracle.attn_fwd(q, k, v, False, scale)
    assert_parity(o.cpu(), lse.cpu(), o64, lse64, f"after timeout D={D}")
    assert ap.device_status(reset=True) == 0


def test_withheld_signal_beyond_last_block_is_harmless():
    """A drop block past the end of every CTA's KV loop changes nothing."""
    q, k, v = make_qkv(1, 2, 1, 300, 300, 128, seed=22)
    scale = 1.0 / math.sqrt(128)
    o, lse = ap.fwd_timeout_test(q.cuda(), k.cuda(), v.cuda(), True, scale, drop_block=50)
    torch.cuda.synchronize()
    assert ap.device_status(reset=True) == 0
    o64, lse64 = oracle.attn_fwd(q, k, v, True, scale)
    assert_parity(o.cpu(), lse.cpu(), o64, lse64, "drop beyond end")


@pytest.mark.parametrize("D", [64, 128])
def test_split_tail_handoff_runs_out_and_context_survives(D):
    """No CTA of a split tail pair sends its staged partial: each CTA's
    cluster-scope wait for the partner's runs out; both reach the exit
    barrier."""
    q, k, v = make_qkv(1, 40, 40, 1024, 4096, D, seed=23)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    assert ap.fwd_tail_pairs(1, 40, 40, 1024, 4096, D, False) > 0
    assert ap.device_status(reset=True) == 0
    ap.fwd_tail_timeout_test(qd, kd, vd, False, scale, wait_budget_ns=20_000_000)
    torch.cuda.synchronize()
    assert ap.device_status(reset=True) == 5        # ATTN_ERR_TIMEOUT
    o, lse = ap.attn_fwd(qd, kd, vd, False, scale)
    torch.cuda.synchronize()
    assert ap.device_status(reset=True) == 0
    o64, lse64 = oracle.attn_fwd(q, k, v, False, scale)
    assert_parity(o.cpu(), lse.cpu(), o64, lse64, f"after hand-off timeout D={D}")


def test_split_tail_handoff_test_needs_a_split_tail():
    q, k, v = make_qkv(1, 2, 2, 512, 512, 64, seed=24)
    with pytest.raises(ap.AttnError):
        ap.fwd_tail_timeout_test(q.cuda(), k.cuda(), v.cuda(), False, 0.125)


@pytest.mark.parametrize("D", [64, 128])
def test_bwd_wait_runs_out_and_context_survives(D):
    """The backward's dK/dV kernel with dQ: one "P^T, dS^T stored" signal is
    withheld at the second query block of every CTA, the issuer's wait runs
    out, every role unwinds (the dQ read-out warps included) and a normal
    backward right after agrees with the deterministic path."""
    from tests.test_gpu_bwd import bf16_ulps, make_dout
    q, k, v = (t.cuda() for t in make_qkv(1, 4, 2, 512, 512, D, seed=24))
    dout = make_dout(q.shape, 25).cuda()
    scale = 1.0 / math.sqrt(D)
    o, lse = ap.attn_fwd(q, k, v, False, scale)
    torch.cuda.synchronize()
    assert ap.device_status(reset=True) == 0
    ap.bwd_timeout_test(q, k, v, o, lse, dout, False, scale, drop_item=1,
                        wait_budget_ns=20_000_000)
    torch.cuda.synchronize()
    assert ap.device_status(reset=True) == 5        # ATTN_ERR_TIMEOUT
    got = ap.attn_bwd(q, k, v, o, lse, dout, False, scale)
    want = ap.attn_bwd(q, k, v, o, lse, dout, False, scale, deterministic=True)
    torch.cuda.synchronize()
    assert ap.device_status(reset=True) == 0
    for g, w_ in zip(got, want):
        assert bf16_ulps(g, w_) <= 4.0
