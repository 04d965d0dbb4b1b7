"""The fp64 oracle against what the definition of attention fixes (CPU only)."""
import pytest

import oracle
from tests import pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    errs = pin(orc)
    assert not errs, "\n".join(errs[:10])


def test_rows_match_full(orc):
    """The sampled-row entry point gives the same numbers as the full forward."""
    import numpy as np
    from attention_pipelining_gb300.synthetic import make_qkv
    q, k, v = make_qkv(2, 4, 2, 37, 41, 16, seed=2)
    for causal in (False, True):
        o, lse = orc.attn_fwd(q, k, v, causal, 0.25)
        rows = np.array([0, 5, 36, 37, 100, 2 * 4 * 37 - 1])
        o_r, l_r = orc.attn_rows(q, k, v, rows, causal, 0.25)
        assert np.array_equal(o.reshape(-1, 16)[rows], o_r)
        assert np.array_equal(lse.reshape(-1)[rows], l_r)


def test_rejects_bad_arguments(orc):
    from attention_pipelining_gb300.synthetic import make_qkv
    q, k, v = make_qkv(1, 3, 2, 4, 4, 8)   # 3 query heads over 2 kv heads
    with pytest.raises(ValueError):
        orc.attn_fwd(q, k, v, False, 1.0)
