"""The fp16 input rounding against torch's float16 conversion and against the binary16
format's definition (exact patterns, ties to even, subnormals, overflow)."""
import numpy as np
import pytest

from exact_attention_bwd_gb300 import inputs


def test_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = inputs.rng(7).standard_normal(200000).astype(np.float32) * np.float32(3.0)
    x = np.concatenate([x, inputs.rng(8).standard_normal(20000).astype(np.float32) * np.float32(1e-5)])
    ours = inputs.f16_bits(x)
    ref = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("x,bits", [
    (1.0, 0x3C00), (-2.0, 0xC000), (0.5, 0x3800), (-0.0, 0x8000), (65504.0, 0x7BFF),
    (65520.0, 0x7C00),                            # halfway to 2^16: ties to even -> inf
    (2.0 ** -24, 0x0001), (2.0 ** -25, 0x0000),    # smallest subnormal; half of it ties to 0
    (3 * 2.0 ** -25, 0x0002), (2.0 ** -14, 0x0400),
    (1 + 2.0 ** -11, 0x3C00), (1 + 3 * 2.0 ** -11, 0x3C02),   # ties to the even neighbour
    (1 + 2.0 ** -10, 0x3C01),
])
def test_exact_patterns(x, bits):
    assert int(inputs.f16_bits(np.float32([x]))[0]) == bits


def test_round_trip_and_spacing():
    allb = np.arange(1 << 16, dtype=np.uint16)
    vals = inputs.f16_to_f64(allb)
    finite = np.isfinite(vals)
    assert finite.sum() == (1 << 16) - 2 * 1024     # exponent 31: 2 infinities + 2046 NaNs
    assert np.array_equal(inputs.f16_bits(vals[finite].astype(np.float32)), allb[finite])
    # the spacing of [1, 2) is 2^-10
    ones = inputs.f16_to_f64(np.arange(0x3C00, 0x4000, dtype=np.uint16))
    assert np.allclose(np.diff(ones), 2.0 ** -10, rtol=0, atol=0)


def test_make_f16_uses_the_same_draws():
    w = dict(wid=3, variant=1, B=1, s_q=40, s_kv=40, h_q=2, h_kv=1, d=64, causal=False, window=(-1, -1),
             sinks=False, varlen=False)
    a = inputs.make(dict(w))
    b = inputs.make(dict(w, dtype="f16"))
    assert a["dtype"] == "bf16" and b["dtype"] == "f16"
    for key in ("q", "k", "v", "dout"):
        xa, xb = inputs.bf16_to_f64(a[key]), inputs.f16_to_f64(b[key])
        # two roundings of one fp32 draw: within bf16's half ulp of each other
        assert np.all(np.abs(xa - xb) <= 2.0 ** -8 * np.abs(xb) + 1e-7)
        assert not np.array_equal(xa, xb)
