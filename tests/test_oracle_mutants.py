"""Plant plausible mistakes in copies of the oracle and check that the pins catch
each one.  The mistakes are planted in the C source of the oracle (on the CPU),
never in the CUDA path."""
import os

import pytest

import oracle
from tests import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

# (name, original text, planted text)
MUTANTS = [
    ("scale dropped", "s[j] = scale * dot;", "s[j] = dot;"),
    ("causal j < i", "return (i + 1 < (int64_t)Skv) ? (i + 1) : (int64_t)Skv;",
     "return (i < (int64_t)Skv) ? i : (int64_t)Skv;"),
    ("causal j <= i + 1", "return (i + 1 < (int64_t)Skv) ? (i + 1) : (int64_t)Skv;",
     "return (i + 2 < (int64_t)Skv) ? (i + 2) : (int64_t)Skv;"),
    ("K transposed", "bf16_bits_to_double(kb[j * D + d])",
     "bf16_bits_to_double(kb[d * (int64_t)Skv + j])"),
    ("grouped heads interleaved", "int64_t hkv = h / (Hq / Hkv);", "int64_t hkv = h % Hkv;"),
    ("LSE in log2", "*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
    ("LSE without max", "*lse_out = m + log(l);", "*lse_out = log(l);"),
    ("no normalisation", "double pj = s[j] / l;", "double pj = s[j];"),
    ("V reversed", "o_row[d] += pj * bf16_bits_to_double(vb[j * D + d]);",
     "o_row[d] += pj * bf16_bits_to_double(vb[(nvis - 1 - j) * D + d]);"),
    ("exp sign flipped", "s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    ("query head from kv head", "const uint16_t *qi = q + ((b * Hq + h)",
     "const uint16_t *qi = q + ((b * Hq + hkv)"),
    ("max not subtracted in LSE path", "s[j] = exp(s[j] - m);", "s[j] = exp(s[j]);"),
]


@pytest.mark.parametrize("name,orig,planted", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, orig, planted):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation site for '{name}' not found exactly once"
    mut_c = tmp_path / "mutant.c"
    mut_c.write_text(src.replace(orig, planted))
    lib = oracle.compile_source(str(mut_c), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            errs = pin(orc)
        except Exception as e:  # a crash in the checks also counts as caught
            errs = [repr(e)]
        if errs:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake '{name}'"
