"""GPU tests of the deterministic backward (FA_FLAG_DETERMINISTIC).

With the flag, dQ is summed over key blocks in a fixed order and the sink gradient in a
fixed per-head reduction, so two runs on the same inputs give the same bits (the pages'
deterministic backward option, vllm-project/flash-attention README, changelog 2.4).  The
results must still match the fp64 oracle like the default backward, and agree with it
within the same tolerance.  The shapes cover d = 64, 128, 192 and 256, causal and window bands
(whose key blocks see different query-tile ranges, so the order has gaps and ends),
grouped-query heads, packed batches with empty sequences, and the benchmark's full size.
"""
import numpy as np
import pytest

import oracle
from exact_attention_bwd_gb300 import inputs
from gpu_helpers import check, dev_inputs, f64, from_dev, oracle_args

pytestmark = pytest.mark.gpu


def case(variant, **kw):
    base = dict(wid=130, variant=variant, B=2, s_q=300, s_kv=300, h_q=4, h_kv=2, d=64, causal=True,
                window=(-1, -1), sinks=False, varlen=False)
    base.update(kw)
    if "lengths" in base:
        base["varlen"] = True
        base["B"] = len(base["lengths"])
    return inputs.make(base)


def run_bwd(w, d, flags):
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    kw = dict(causal=w["causal"], window=w["window"], softmax_scale=w["scale"], sinks=d["sinks"], cu_q=d["cu_q"],
              cu_k=d["cu_k"])
    o, lse, _ = fa.forward(d["q"], d["k"], d["v"], **kw)
    dq, dk, dv, ds, ws = fa.backward(d["q"], d["k"], d["v"], o, lse, d["dout"], **kw, flags=flags)
    torch.cuda.synchronize()
    assert fa.device_status(ws) == fa.FA_OK
    out = [dq, dk, dv] + ([] if ds is None else [ds])
    return [x.detach().cpu().clone() for x in out]


def bitwise_equal(a, b):
    import torch
    return all(torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x, y.view(torch.int16)
                           if y.dtype == torch.bfloat16 else y) for x, y in zip(a, b))


CASES = [
    dict(d=64),
    dict(d=128),
    dict(d=128, causal=False, window=(130, 40), h_q=8, h_kv=2, sinks=True),
    dict(d=64, s_q=700, s_kv=700, h_q=16, h_kv=2, window=(127, 0), sinks=True),
    dict(d=128, s_q=200, s_kv=650, h_q=6, h_kv=2),
    dict(d=128, s_q=650, s_kv=200, h_q=4, h_kv=4, causal=True),
    dict(d=128, lengths=[17, 283, 128, 0, 1, 0, 300, 129], h_q=4, h_kv=2),
    dict(d=64, lengths=[400, 3, 0, 250], h_q=8, h_kv=2, causal=False, window=(50, 20), sinks=True),
    # the wide-head kernel (64-key blocks)
    dict(d=256),
    dict(d=192, causal=False, window=(130, 40), h_q=8, h_kv=2, sinks=True),
    dict(d=256, lengths=[17, 283, 128, 0, 1, 0, 300, 129], h_q=4, h_kv=2),
    dict(d=192, s_q=200, s_kv=650, h_q=6, h_kv=2),
]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_deterministic_matches_oracle_and_repeats(i):
    from exact_attention_bwd_gb300 import binding as fa
    w = case(i, **CASES[i])
    d = dev_inputs(w)
    a = run_bwd(w, d, fa.FA_FLAG_DETERMINISTIC)
    b = run_bwd(w, d, fa.FA_FLAG_DETERMINISTIC)
    assert bitwise_equal(a, b), "two deterministic runs differ"
    q, k, v, do = f64(w, "q"), f64(w, "k"), f64(w, "v"), f64(w, "dout")
    dq, dk, dv, ds = oracle.bwd(q, k, v, do, **oracle_args(w))
    check("dQ", from_dev(a[0]), dq)
    check("dK", from_dev(a[1]), dk)
    check("dV", from_dev(a[2]), dv)
    if ds is not None:
        err = float(np.abs(a[3].numpy().astype(np.float64) - ds).max())
        assert err <= 2e-2 * max(1.0, float(np.abs(ds).max()))
    # the default (arrival-order) backward agrees within the oracle tolerance
    c = run_bwd(w, d, 0)
    for x, y in zip(a[:3], c[:3]):
        check("default vs deterministic", from_dev(y), from_dev(x))


def test_deterministic_full_size():
    """The benchmark's workload (B=2, s=8192, h=16, d=128, causal): bitwise-equal reruns,
    and within tolerance of the default backward."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    w = inputs.workload("sweep_s8192_causal")
    sd = lambda t: inputs.seed_of(w["wid"], w["variant"], t)  # noqa: E731
    dev = torch.device("cuda", 0)
    shape = (w["B"], w["s_q"], w["h_q"], w["d"])
    d = dict(q=inputs.normal_bf16_torch(sd(inputs.Q), shape, dev), k=inputs.normal_bf16_torch(sd(inputs.K), shape, dev),
             v=inputs.normal_bf16_torch(sd(inputs.V), shape, dev),
             dout=inputs.normal_bf16_torch(sd(inputs.DO), shape, dev), sinks=None, cu_q=None, cu_k=None)
    w = dict(w, scale=1.0 / np.sqrt(w["d"]))
    a = run_bwd(w, d, fa.FA_FLAG_DETERMINISTIC)
    b = run_bwd(w, d, fa.FA_FLAG_DETERMINISTIC)
    assert bitwise_equal(a, b), "two deterministic runs differ"
    c = run_bwd(w, d, 0)
    for x, y in zip(a, c):
        check("default vs deterministic", from_dev(y), from_dev(x))
