"""The seeded input generators: bf16 rounding and packed-batch lengths."""
import numpy as np
import pytest
import torch

from exact_attention_bwd_gb300 import inputs


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 7
    x[:6] = [0.0, -0.0, 1.0, 1.00390625, 1.01171875, -3.5e-39]   # ties and a denormal
    ours = inputs.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    back = inputs.bf16_to_f32(ours)
    np.testing.assert_array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_varlen_lengths_recipe():
    L = inputs.varlen_lengths(inputs.seed_of(4, 0, inputs.LENGTHS))
    assert L.dtype == np.int32 and len(L) == 256
    assert int(L.sum()) == 32768
    assert int((L == 0).sum()) == 26          # round(0.1 * 256)
    assert int(L[L > 0].min()) >= 1
    cu = inputs.cu_seqlens(L)
    assert cu[0] == 0 and cu[-1] == 32768 and np.all(np.diff(cu) >= 0)


def test_draws_are_seeded():
    a = inputs.normal_bf16(7, (3, 4))
    b = inputs.normal_bf16(7, (3, 4))
    c = inputs.normal_bf16(8, (3, 4))
    assert np.array_equal(a, b) and not np.array_equal(a, c)


@pytest.mark.parametrize("name", sorted(inputs.WORKLOADS))
def test_workload_shapes(name):
    w = inputs.workload(name)
    if w.get("varlen"):
        assert w["T"] == 32768
    else:
        assert w["h_q"] % w["h_kv"] == 0
