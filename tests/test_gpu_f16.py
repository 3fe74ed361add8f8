"""GPU parity of the fp16 inputs against the fp64 oracle.

The pages take bf16 or fp16 tensors (dew-flash-attn PyPI page, usage; fa4-jax PyPI page,
restrictions: fp16/bf16).  fp16 runs the bf16 kernels' fp16 instantiations: the tensor
cores read fp16 operands, P, dS and the outputs are rounded to fp16, accumulation and the
statistics stay fp32.  The same tolerances as bf16 apply; fp16's 10-bit mantissa should
beat bf16's 7-bit one by a wide margin, and one test checks that it does on the same fp32
draws — a kernel that read fp16 bits as bf16 (or rounded to bf16 on the way) would not.

Shapes reach every kernel with a 16-bit path: the d = 64 / 128 forward and backward
(masks, grouped-query heads, sinks, packed batches with empty sequences, s_q != s_kv),
the d = 256 forward, the split tensor-core forward with its combine, the CUDA-core decode
kernel on dense and paged caches, and the deterministic backward.
"""
import numpy as np
import pytest

import oracle
from exact_attention_bwd_gb300 import inputs
from gpu_helpers import check, check_lse, dev_inputs, f64, from_dev, oracle_args, run_gpu, to_dev

pytestmark = pytest.mark.gpu

WID = 140


def case(variant, dtype="f16", **kw):
    w = dict(wid=WID, variant=variant, B=2, s_q=300, s_kv=300, h_q=4, h_kv=2, d=128, causal=True,
             window=(-1, -1), sinks=False, varlen=False, dtype=dtype)
    w.update(kw)
    if "lengths" in w:
        w["varlen"] = True
        w["B"] = len(w["lengths"])
    return inputs.make(w)


def errors(w, bwd=True, flags=0):
    """Runs the library on w, checks every output against the oracle and returns the
    mean-abs error of each."""
    got = run_gpu(w, bwd=bwd, flags=flags)
    q, k, v, do = f64(w, "q"), f64(w, "k"), f64(w, "v"), f64(w, "dout")
    kw = oracle_args(w)
    o, lse, _ = oracle.fwd(q, k, v, **kw)
    out = dict(o=check("O", got["o"], o)[1])
    check_lse("LSE", got["lse"], lse)
    if bwd:
        dq, dk, dv, ds = oracle.bwd(q, k, v, do, **kw)
        out.update(dq=check("dQ", got["dq"], dq)[1], dk=check("dK", got["dk"], dk)[1],
                   dv=check("dV", got["dv"], dv)[1])
        if ds is not None:
            err = float(np.abs(got["dsinks"] - ds).max())
            assert err <= 2e-2 * max(1.0, float(np.abs(ds).max())), f"dsink max-abs {err:.3e}"
    return out


CASES = [
    dict(d=64),
    dict(d=128),
    dict(d=64, causal=False),
    dict(d=128, causal=False, window=(130, 40), h_q=8, h_kv=2, sinks=True),
    dict(d=64, s_q=200, s_kv=650, h_q=6, h_kv=2),
    dict(d=128, s_q=650, s_kv=200, h_q=4, h_kv=4),
    dict(d=128, lengths=[17, 283, 128, 0, 1, 0, 300, 129]),
    dict(d=64, lengths=[400, 3, 0, 250], h_q=8, h_kv=2, causal=False, window=(50, 20), sinks=True),
    # dense grouped-query window at d = 64: the forward's 64-key tiles, two CTAs per SM
    dict(d=64, s_q=700, s_kv=700, h_q=16, h_kv=2, causal=True, window=(127, 0), sinks=True),
]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_forward_backward(i):
    errors(case(i, **CASES[i]))


@pytest.mark.parametrize("causal", [False, True])
def test_forward_d256(causal):
    errors(case(20 + causal, d=256, s_q=300, s_kv=300, h_q=4, h_kv=2, causal=causal), bwd=False)


def test_forward_split_keys():
    """64 queries against 6000 keys: the tensor-core forward splits the key range and the
    combine kernel merges the fp32 partials into fp16 rows; NO_SPLIT gives the same
    problem in one pass."""
    from exact_attention_bwd_gb300 import binding as fa
    w = case(30, B=1, s_q=64, s_kv=6000, h_q=8, h_kv=2, d=128)
    errors(w, bwd=False)
    errors(w, bwd=False, flags=fa.FA_FLAG_NO_SPLIT)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_decode(d):
    """One query per sequence (the CUDA-core decode kernel and the combine)."""
    errors(case(40 + d, B=3, s_q=1, s_kv=3000, h_q=8, h_kv=2, d=d), bwd=False)


def test_paged_decode():
    """A paged fp16 cache: key j of sequence b is row j % 128 of page table[b][j // 128];
    the oracle sees the dense cache the pages stand for."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    B, s_kv, h_q, h_kv, d, ps = 3, 1000, 8, 2, 128, 128
    sd = lambda t: inputs.seed_of(WID, 50, t)  # noqa: E731
    max_blocks = -(-s_kv // ps)
    num_pages = B * max_blocks + 2
    table = inputs.page_table(sd(7), B, max_blocks, num_pages)
    q = inputs.f16_bits(inputs.normal_f32(sd(inputs.Q), (B, 1, h_q, d)))
    kp = inputs.f16_bits(inputs.normal_f32(sd(inputs.K), (num_pages, ps, h_kv, d)))
    vp = inputs.f16_bits(inputs.normal_f32(sd(inputs.V), (num_pages, ps, h_kv, d)))
    o, lse, ws = fa.forward(to_dev(q, "f16"), to_dev(kp, "f16"), to_dev(vp, "f16"), causal=True,
                            block_table=torch.from_numpy(table).cuda(), s_kv=s_kv)
    torch.cuda.synchronize()
    assert fa.device_status(ws) == fa.FA_OK
    assert o.dtype == torch.float16
    j = np.arange(s_kv)
    kd = inputs.f16_to_f64(kp)[table[:, j // ps], j % ps]
    vd = inputs.f16_to_f64(vp)[table[:, j // ps], j % ps]
    ro, rl, _ = oracle.fwd(inputs.f16_to_f64(q), kd, vd, scale=1.0 / np.sqrt(d), causal=True)
    check("O", from_dev(o), ro)
    check_lse("LSE", lse.cpu().numpy().astype(np.float64), rl)


def test_deterministic_backward_repeats():
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    w = case(60, d=128, h_q=8, h_kv=2, causal=False, window=(130, 40), sinks=True)
    errors(w, flags=fa.FA_FLAG_DETERMINISTIC)
    d = dev_inputs(w)
    kw = dict(causal=w["causal"], window=w["window"], softmax_scale=w["scale"], sinks=d["sinks"])
    o, lse, _ = fa.forward(d["q"], d["k"], d["v"], **kw)
    runs = []
    for _ in range(2):
        dq, dk, dv, ds, ws = fa.backward(d["q"], d["k"], d["v"], o, lse, d["dout"], **kw,
                                         flags=fa.FA_FLAG_DETERMINISTIC)
        torch.cuda.synchronize()
        assert fa.device_status(ws) == fa.FA_OK
        runs.append([x.view(torch.int16).cpu().clone() for x in (dq, dk, dv)] + [ds.cpu().clone()])
    assert all(torch.equal(a, b) for a, b in zip(*runs))


@pytest.mark.parametrize("d", [64, 128])
def test_f16_beats_bf16_precision(d):
    """On the same fp32 draws, the fp16 path's mean error is well below the bf16 path's
    (fp16 keeps 3 more mantissa bits in the inputs, P, dS and the outputs)."""
    kw = dict(d=d, h_q=8, h_kv=2, sinks=True)
    e16 = errors(case(70 + d, dtype="f16", **kw))
    ebf = errors(case(70 + d, dtype="bf16", **kw))
    for key in ("o", "dq", "dk", "dv"):
        assert e16[key] <= 0.5 * ebf[key], f"{key}: fp16 mean error {e16[key]:.3e} vs bf16 {ebf[key]:.3e}"


def test_outputs_have_input_type():
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    w = case(80, d=64, B=1, s_q=130, s_kv=130, h_q=2, h_kv=2)
    d = dev_inputs(w)
    o, lse, _ = fa.forward(d["q"], d["k"], d["v"], causal=True)
    dq, dk, dv, _, _ = fa.backward(d["q"], d["k"], d["v"], o, lse, d["dout"], causal=True)
    torch.cuda.synchronize()
    assert {t.dtype for t in (o, dq, dk, dv)} == {torch.float16}
    assert lse.dtype == torch.float32
