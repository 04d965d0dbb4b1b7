"""Plant plausible mistakes in copies of the chunk-scan oracle and check that
the pins of tests/test_chunk_scan_oracle_pins.py catch each one.  The mistakes
are planted in the C source of the oracle (on the CPU), never in the CUDA
path."""
import os

import pytest

import oracle
from tests import test_chunk_scan_oracle_pins as cp

SRC = os.path.join(os.path.dirname(oracle.__file__), "chunk_scan_oracle.c")

# (name, original text, planted text); each site occurs exactly once
MUTANTS = [
    ("decay sign flipped", "exp((double)da[m] - (double)da[k])", "exp((double)da[k] - (double)da[m])"),
    ("mask k < m", "for (int64_t k = 0; k <= m; ++k) {", "for (int64_t k = 0; k < m; ++k) {"),
    ("mask dropped", "for (int64_t k = 0; k <= m; ++k) {", "for (int64_t k = 0; k < Q; ++k) {"),
    ("dt of the row", "* (double)dtc[k];", "* (double)dtc[m];"),
    ("cb transposed", "double w = (double)cb_row[k]",
     "double w = (double)cb[(((b * nch + c) * G + g) * (int64_t)Q + k) * Q + m]"),
    ("groups interleaved", "int64_t g = h / (H / G);", "int64_t g = h % G;"),
    ("x without chunk offset", "const uint16_t *xk = x + ((b * L + c * Q + k) * H + h) * (int64_t)P;",
     "const uint16_t *xk = x + ((b * L + k) * H + h) * (int64_t)P;"),
    ("dA of the first chunk", "const float *da = dA_cs + ((b * H + h) * nch + c) * (int64_t)Q;",
     "const float *da = dA_cs + ((b * H + h) * nch) * (int64_t)Q;"),
]


@pytest.mark.parametrize("name,orig,planted", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, orig, planted):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation site for '{name}' not found exactly once"
    mut_c = tmp_path / "mutant.c"
    mut_c.write_text(src.replace(orig, planted))
    lib = oracle.compile_source(str(mut_c), str(tmp_path / "libmutant.so"))
    cs = oracle.ChunkScanOracle(lib)
    caught = []
    for check in (cp.check_recurrence, cp.check_single_key, cp.check_constant_cb_groups,
                  cp.check_shift_and_zero):
        try:
            check(cs)
        except Exception as e:  # a failed assertion or a crash counts as caught
            caught.append(f"{check.__name__}: {str(e)[:60]}")
    assert caught, f"no pin caught the planted mistake '{name}'"
