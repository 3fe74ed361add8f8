"""The e4m3 input encoder against torch's float8_e4m3fn conversion and the format's own
definition (special values, spacing, saturation)."""
import numpy as np
import pytest

from exact_attention_bwd_gb300 import inputs


def test_encoder_matches_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    x = inputs.rng(5).standard_normal(200000).astype(np.float32) * np.float32(40.0)
    x = np.concatenate([x, np.float32([0.0, -0.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 448.0, -448.0, 1.0625,
                                       1.1875, 240.0, 232.0, 0.015625])])
    ours = inputs.e4m3_bits(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_round_trip_and_special_values():
    allb = np.arange(256, dtype=np.uint8)
    vals = inputs.e4m3_to_f64(allb)
    finite = ~np.isnan(vals)
    assert finite.sum() == 254                      # 0x7F and 0xFF are NaN
    assert np.nanmax(vals) == 448.0 and np.nanmin(vals) == -448.0
    # every finite pattern decodes and encodes back to itself (0x80 is -0, kept as such)
    back = inputs.e4m3_bits(np.where(allb[finite] == 0x80, -0.0, vals[finite]))
    assert np.array_equal(back, allb[finite])
    assert inputs.e4m3_to_f64(np.uint8(1)) == 2.0 ** -9   # smallest subnormal
    assert inputs.e4m3_to_f64(np.uint8(8)) == 2.0 ** -6   # smallest normal
    # ties go to even mantissas, values beyond 448 saturate
    assert inputs.e4m3_to_f64(inputs.e4m3_bits(1.0625)) == 1.0
    assert inputs.e4m3_to_f64(inputs.e4m3_bits(1.1875)) == 1.25
    assert inputs.e4m3_to_f64(inputs.e4m3_bits(1000.0)) == 448.0
    assert inputs.e4m3_to_f64(inputs.e4m3_bits(-1000.0)) == -448.0


def test_descales_range():
    d = inputs.descales(3, 4, 8)
    assert d.dtype == np.float32 and d.shape == (32,)
    assert np.all(d >= 0.5 / 32 - 1e-9) and np.all(d <= 2.0 / 32 + 1e-9)
