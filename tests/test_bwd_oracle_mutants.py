"""Plant plausible mistakes in copies of the backward oracle and check that the
pins of tests/test_bwd_oracle_pins.py catch each one.  The mistakes are
planted in the C source of the oracle (on the CPU), never in the CUDA path."""
import os

import pytest

import oracle
from tests import test_bwd_oracle_pins as bp

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_bwd_oracle.c")

# (name, original text, planted text); each site occurs exactly once
MUTANTS = [
    ("D term dropped", "double ds = p[j] * (dp - delta);\n                            for (int d = 0; d < D; ++d) {\n                                dqi",
     "double ds = p[j] * dp;\n                            for (int d = 0; d < D; ++d) {\n                                dqi"),
    ("dK without scale", "dkb[j * D + d] += scale * ds * qi[d];", "dkb[j * D + d] += ds * qi[d];"),
    ("dQ without scale", "dqi[d] += scale * ds * kb[j * D + d];", "dqi[d] += ds * kb[j * D + d];"),
    ("dQ from V", "dqi[d] += scale * ds * kb[j * D + d];", "dqi[d] += scale * ds * vb[j * D + d];"),
    ("dV from Q", "dvb[j * D + d] += p[j] * doi[d];", "dvb[j * D + d] += p[j] * qi[d];"),
    ("dK from dO", "dkb[j * D + d] += scale * ds * qi[d];", "dkb[j * D + d] += scale * ds * doi[d];"),
    ("D_i from dO only", "dl += doi[d] * o[d];", "dl += doi[d] * doi[d];"),
    ("P not normalised", "p[j] /= l;", "p[j] /= 1.0;"),
    ("dP from K", "dp += doi[d] * vb[j * D + d];\n                            double ds = p[j] * (dp - delta);\n                            for (int d = 0; d < D; ++d) {\n                                dqi",
     "dp += doi[d] * kb[j * D + d];\n                            double ds = p[j] * (dp - delta);\n                            for (int d = 0; d < D; ++d) {\n                                dqi"),
    ("grouped heads interleaved", "int64_t hkv = h / (Hq / Hkv);\n    const double *qi",
     "int64_t hkv = h % Hkv;\n    const double *qi"),
    ("causal j < i", "return (i + 1 < (int64_t)Skv) ? (i + 1) : (int64_t)Skv;",
     "return (i < (int64_t)Skv) ? i : (int64_t)Skv;"),
    ("scale dropped from scores", "p[j] = scale * dot;", "p[j] = dot;"),
]


@pytest.mark.parametrize("name,orig,planted", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, orig, planted):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation site for '{name}' not found exactly once"
    mut_c = tmp_path / "mutant.c"
    mut_c.write_text(src.replace(orig, planted))
    lib = oracle.compile_source(str(mut_c), str(tmp_path / "libmutant.so"))
    bo = oracle.BwdOracle(lib)
    caught = []
    for check in (bp.check_finite_difference, bp.check_torch, bp.check_identities):
        for shape in (bp.SHAPES[1], bp.SHAPES[2]):
            try:
                check(bo, shape)
            except Exception as e:  # a failed assertion or a crash counts as caught
                caught.append(f"{check.__name__}: {str(e)[:60]}")
    assert caught, f"no pin caught the planted mistake '{name}'"
