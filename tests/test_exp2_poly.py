"""The forward's FMA-pipe exp2 (exp2_poly2 in csrc/ptx.cuh), emulated step by step in fp32.

The method: x = n + f with n = round(x) taken from the low mantissa bits of
x + 1.5 * 2^23, f in [-1/2, 1/2]; a degree-3 polynomial for 2^f; n added to the
exponent field.  The coefficients are read from the header, and the result must stay
within 1e-4 relative error of 2^x over the range the kernel feeds it ([-125, 8]),
far below the 2^-9 rounding of the bf16 probabilities it produces.
"""
import os
import re

import numpy as np

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "exact_attention_bwd_gb300",
                   "csrc", "ptx.cuh")


def coefficients():
    src = open(HDR).read()
    body = src[src.index("exp2_poly2"):]
    body = body[:body.index("return make_float2")]
    vals = [float(v) for v in re.findall(r"make_float2\(([-0-9.e]+)f, \1f\)", body)]
    # the last four constants of the function, in source order: c3, c2 (first fma), c1, c0
    return vals[-4:]


def emulate(x):
    x = np.asarray(x, np.float32)
    c3, c2, c1, c0 = (np.float32(v) for v in coefficients())
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    n = (t - magic).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = (c3 * f + c2).astype(np.float32)
    p = (p * f + c1).astype(np.float32)
    p = (p * f + c0).astype(np.float32)
    bits = (p.view(np.uint32).astype(np.uint64) + ((t.view(np.uint32).astype(np.uint64) << 23) & 0xFFFFFFFF))
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def test_coefficients_found():
    assert len(coefficients()) == 4


def test_relative_error_over_kernel_range():
    x = np.concatenate([np.linspace(-125.0, 8.0, 2_000_001), np.arange(-125, 9, dtype=np.float64)]).astype(np.float32)
    got = emulate(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(got - ref) / ref
    assert rel.max() < 1e-4, rel.max()


def test_monotone_and_exact_at_zero():
    x = np.linspace(-20, 0, 200001).astype(np.float32)
    y = emulate(x)
    assert np.all(np.diff(y.astype(np.float64)) >= -1e-12 * y[1:])
    assert abs(float(emulate(np.float32(0.0))) - 1.0) < 1e-4
