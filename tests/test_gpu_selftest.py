"""GPU checks of the kernel's building blocks: TMA with 128-byte swizzle, the
shared-memory and instruction descriptors of tcgen05.mma, and the tensor-
memory layouts, each on one 128-row tile against a CPU product."""
import numpy as np
import pytest
import torch

import attention_pipelining_gb300 as ap

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ap.build()
    ap.device_status(reset=True)
    yield
    assert ap.device_status(reset=True) == 0


def _f64(t):
    return t.detach().cpu().double().numpy()


@pytest.mark.parametrize("D", [64, 128])
def test_qk_tile(D):
    g = torch.Generator().manual_seed(D)
    q = torch.randn((128, D), generator=g).to(torch.bfloat16)
    k = torch.randn((128, D), generator=g).to(torch.bfloat16)
    s = ap.selftest_qk(q.cuda(), k.cuda())
    torch.cuda.synchronize()
    want = _f64(q) @ _f64(k).T
    bound = np.abs(_f64(q)) @ np.abs(_f64(k)).T * 2e-6 + 1e-6   # fp32 accumulation of exact products
    assert np.all(np.abs(_f64(s) - want) <= bound), np.abs(_f64(s) - want).max()


@pytest.mark.parametrize("D", [64, 128])
def test_qk_tile_structured(D):
    """Index patterns that expose a transposed or mis-strided operand exactly."""
    q = torch.zeros((128, D))
    k = torch.zeros((128, D))
    for i in range(128):
        q[i, i % D] = 1.0 + (i // D)
        k[i, (3 * i) % D] = float(i % 7 + 1)
    q, k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    s = ap.selftest_qk(q.cuda(), k.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(_f64(s), _f64(q) @ _f64(k).T)


@pytest.mark.parametrize("D", [64, 128])
def test_pv_tile(D):
    g = torch.Generator().manual_seed(100 + D)
    p = torch.rand((128, 128), generator=g).to(torch.bfloat16)
    v = torch.randn((128, D), generator=g).to(torch.bfloat16)
    o = ap.selftest_pv(p.cuda(), v.cuda())
    torch.cuda.synchronize()
    want = _f64(p) @ _f64(v)
    bound = np.abs(_f64(p)) @ np.abs(_f64(v)) * 2e-6 + 1e-6
    assert np.all(np.abs(_f64(o) - want) <= bound), np.abs(_f64(o) - want).max()


@pytest.mark.parametrize("D", [64, 128])
def test_pv_tile_structured(D):
    """P a permutation-like 0/1 matrix: O must be exact rows of V, so a wrong
    packing order of P in tensor memory or a wrong V stride shows at once."""
    p = torch.zeros((128, 128))
    for i in range(128):
        p[i, (5 * i + 3) % 128] = 1.0
    v = torch.arange(128 * D, dtype=torch.float32).reshape(128, D) % 251 - 125
    p, v = p.to(torch.bfloat16), v.to(torch.bfloat16)
    o = ap.selftest_pv(p.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(_f64(o), _f64(p) @ _f64(v))
