"""Accuracy of the FMA-pipe exp2 in ptx.cuh (exp2_poly_x2), evaluated on the
CPU with the kernel's own fp32 steps: the coefficients are read from the
CUDA header, the rounding split and the exponent add are done on float32
bits, and each fused multiply-add is one rounding of the exact product plus
the addend.  The routine is the measured-and-not-adopted alternative to
MUFU ex2 for part of the softmax's exponentials."""
import os
import re

import numpy as np

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "attention_pipelining_gb300", "csrc", "ptx.cuh")


def _coefficients():
    src = open(HDR).read()
    body = src[src.index("exp2_poly_x2"):]
    vals = dict(re.findall(r"(kC[0-3]) = ([0-9.eE+-]+)f", body[:2000]))
    return [np.float32(vals[f"kC{i}"]) for i in range(4)]


def _fma32(a, b, c):
    # a*b is exact in float64 for float32 inputs; one rounding to float32
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def exp2_poly(x):
    c0, c1, c2, c3 = _coefficients()
    x = np.maximum(np.asarray(x, np.float32), np.float32(-126.0))
    k = np.float32(12582912.0)
    t = (x + k).astype(np.float32)
    n = (t - k).astype(np.float32)
    r = _fma32(n, np.full_like(n, -1.0), x)
    q = _fma32(np.full_like(r, c3), r, np.full_like(r, c2))
    q = _fma32(q, r, np.full_like(r, c1))
    q = _fma32(q, r, np.full_like(r, c0))
    bits = q.view(np.uint32) + (t.view(np.uint32) << np.uint32(23))
    return bits.astype(np.uint32).view(np.float32)


def test_relative_error_against_fp64():
    rng = np.random.default_rng(0)
    # (below -125 the results approach the subnormal range, where fp32
    # itself loses relative precision; they vanish in bf16 P and in the sums)
    x = np.concatenate([np.linspace(-125, 8, 400001, dtype=np.float32),
                        rng.uniform(-40, 8, 400000).astype(np.float32),
                        np.arange(-125, 9, dtype=np.float32)])
    y = exp2_poly(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y - ref) / ref
    assert rel.max() <= 2.0 ** -12.5, rel.max()
    # far below bf16's rounding of P (2^-8) and well inside the LSE tolerance
    assert np.abs(np.log(y / ref)).max() <= 1e-4


def test_against_float32_exp2_and_clamp():
    x = np.linspace(-20, 8, 10001, dtype=np.float32)
    y = exp2_poly(x)
    ref32 = np.exp2(x)  # the C library's single-precision exp2
    assert (np.abs(y - ref32) / ref32).max() <= 2.0 ** -12.5
    # at and below the clamp: tiny, finite and non-negative (no wrapped
    # exponent field)
    z = exp2_poly(np.array([-200.0, -1e30, -127.0, -126.9, -126.5, -126.0, -125.6], np.float32))
    assert np.all(np.isfinite(z)) and np.all(z >= 0) and np.all(z <= 2.0 ** -125)
