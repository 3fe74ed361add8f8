"""Failure paths of the C ABI on a GPU: the device-side offset check and the bounded waits.

The pages leave packed-batch offsets unchecked (fa4-jax PyPI page, "Varlen semantics")
and ask that the restrictions be checked with clear errors (same page, Restrictions).
Here:

- FA_FLAG_VALIDATE_CU: offsets that break the rules (not starting at 0, decreasing,
  not ending at the token count) but stay inside the tensors, so nothing could go out of
  bounds even without the check.  The status word must read FA_ERR_DEVICE_CHECK and
  every output must keep the canary bytes it started with: no kernel after the check
  may touch them.
- wait_limit_ns = 1: the first wait of a kernel's pipeline that is not complete when it
  starts runs out at once, so the CTA takes its give-up path (record FA_ERR_TIMEOUT, let its
  copies and MMAs land, free its tensor memory, return); the cases are shaped so that such
  a wait comes early (a consumer waits for the first copies or MMAs, a producer for ring
  slots).  The status word must read FA_ERR_TIMEOUT, and the next call
  with the default limit, on the same device and streams, must match the oracle: a CTA
  that had left tensor memory allocated or a copy in flight would break it.
No GPU fault, trap or hang is involved: the waits are bounded and the offsets in range.
"""
import numpy as np
import pytest

import oracle
from exact_attention_bwd_gb300 import inputs
from gpu_helpers import Guarded, check, check_lse, dev_inputs, f64, oracle_args

pytestmark = pytest.mark.gpu


def _packed(variant, lengths, d=64, h_q=4, h_kv=2, causal=True, sinks=False):
    w = dict(wid=120, variant=variant, B=len(lengths), s_q=0, s_kv=0, h_q=h_q, h_kv=h_kv, d=d, causal=causal,
             window=(-1, -1), sinks=sinks, varlen=True, lengths=lengths)
    return inputs.make(w)


BAD_OFFSETS = {
    # T = 100 tokens in every case; each list breaks one rule and stays within [0, T]
    "decreasing": [0, 40, 20, 100],
    "not_from_zero": [1, 30, 60, 100],
    "short_of_total": [0, 30, 60, 90],
}


@pytest.mark.parametrize("case", sorted(BAD_OFFSETS))
@pytest.mark.parametrize("which", ["q", "k"])
def test_validate_cu_stops_every_kernel(case, which):
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    w = _packed(0, [30, 30, 40], sinks=True)
    d = dev_inputs(w)
    bad = torch.tensor(BAD_OFFSETS[case], dtype=torch.int32, device="cuda")
    cu_q, cu_k = (bad, d["cu_k"]) if which == "q" else (d["cu_q"], bad)
    kw = dict(causal=True, softmax_scale=w["scale"], sinks=d["sinks"], cu_q=cu_q, cu_k=cu_k,
              flags=fa.FA_FLAG_VALIDATE_CU)
    q, k, v, do = d["q"], d["k"], d["v"], d["dout"]
    g_o, g_lse = Guarded(q.shape, q.dtype), Guarded((4, 100), torch.float32)
    _, _, ws = fa.forward(q, k, v, **kw, out=g_o.t, lse=g_lse.t)
    assert fa.device_status(ws) == fa.FA_ERR_DEVICE_CHECK
    for name, g in (("O", g_o), ("LSE", g_lse)):
        g.check(name)
        assert torch.all(g.buf == 0xFF), f"{name} was written after the offset check failed"
    # the backward, with finite o / lse stand-ins (never read either)
    o, lse = torch.zeros_like(q), torch.zeros((4, 100), dtype=torch.float32, device="cuda")
    g_dq, g_dk, g_dv = Guarded(q.shape, q.dtype), Guarded(k.shape, k.dtype), Guarded(v.shape, v.dtype)
    ds = torch.full((4,), 7.0, device="cuda")
    _, _, _, ds_out, ws2 = fa.backward(q, k, v, o, lse, do, **kw, grads=(g_dq.t, g_dk.t, g_dv.t, ds))
    assert fa.device_status(ws2) == fa.FA_ERR_DEVICE_CHECK
    for name, g in (("dQ", g_dq), ("dK", g_dk), ("dV", g_dv)):
        g.check(name)
        assert torch.all(g.buf == 0xFF), f"{name} was written after the offset check failed"
    # the sink gradient is cleared on the host side of the call and stays zero
    assert torch.all(ds_out == 0)


def test_validate_cu_passes_good_offsets():
    """The same flag with valid offsets (an empty sequence included) changes nothing."""
    from exact_attention_bwd_gb300 import binding as fa
    from gpu_helpers import run_gpu
    w = _packed(1, [30, 0, 70, 1], d=128, sinks=True)
    got = run_gpu(w, bwd=True, flags=fa.FA_FLAG_VALIDATE_CU)
    q, k, v, do = f64(w, "q"), f64(w, "k"), f64(w, "v"), f64(w, "dout")
    o, lse, _ = oracle.fwd(q, k, v, **oracle_args(w))
    dq, dk, dv, _ = oracle.bwd(q, k, v, do, **oracle_args(w))
    check("O", got["o"], o)
    check_lse("LSE", got["lse"], lse)
    check("dQ", got["dq"], dq)
    check("dK", got["dk"], dk)
    check("dV", got["dv"], dv)


def _dense(variant, **kw):
    base = dict(wid=121, variant=variant, B=2, s_q=300, s_kv=300, h_q=4, h_kv=2, d=64, causal=True, window=(-1, -1),
                sinks=False, varlen=False)
    base.update(kw)
    return inputs.make(base)


# (name, workload overrides, backward flags or None for a forward-only case)
TIMEOUT_CASES = [
    ("fwd_d64", dict(d=64), None),
    ("fwd_d128_two_tiles", dict(d=128, s_q=600, s_kv=600), None),
    ("fwd_d256", dict(d=256), None),
    ("fwd_split_keys", dict(d=128, s_q=64, s_kv=4100, h_q=8), None),
    # a long cache in few units: each split streams many key tiles, so the producer
    # waits for ring slots (with one tile per split nothing ever waits)
    ("decode", dict(d=128, B=1, s_q=1, s_kv=65536, h_q=8), None),
    ("bwd_d64", dict(d=64, sinks=True), 0),
    ("bwd_d128", dict(d=128, s_q=600, s_kv=600), 0),
    ("bwd_d128_deterministic", dict(d=128, s_q=600, s_kv=600), 4),
    ("bwd_d256", dict(d=256), 0),
]


@pytest.mark.parametrize("name,over,bwd_flags", TIMEOUT_CASES, ids=[c[0] for c in TIMEOUT_CASES])
def test_wait_limit_gives_up_cleanly(name, over, bwd_flags):
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    w = _dense(TIMEOUT_CASES.index((name, over, bwd_flags)), **over)
    d = dev_inputs(w)
    kw = dict(causal=w["causal"], window=w["window"], softmax_scale=w["scale"], sinks=d["sinks"])
    q, k, v, do = d["q"], d["k"], d["v"], d["dout"]
    if bwd_flags is None:
        _, _, ws = fa.forward(q, k, v, **kw, wait_limit_ns=1)
        assert fa.device_status(ws) == fa.FA_ERR_TIMEOUT
    else:
        o, lse, _ = fa.forward(q, k, v, **kw)
        *_, ws2 = fa.backward(q, k, v, o, lse, do, **kw, flags=bwd_flags, wait_limit_ns=1)
        assert fa.device_status(ws2) == fa.FA_ERR_TIMEOUT
    torch.cuda.synchronize()
    # the device is healthy afterwards: the same problem with the default limit is exact
    o, lse, ws = fa.forward(q, k, v, **kw)
    assert fa.device_status(ws) == fa.FA_OK
    qf, kf, vf, dof = f64(w, "q"), f64(w, "k"), f64(w, "v"), f64(w, "dout")
    ro, rl, _ = oracle.fwd(qf, kf, vf, **oracle_args(w))
    check("O", o.float().cpu().numpy(), ro)
    check_lse("LSE", lse.cpu().numpy(), rl)
    if bwd_flags is not None:
        dq, dk, dv, _, ws2 = fa.backward(q, k, v, o, lse, do, **kw, flags=bwd_flags)
        assert fa.device_status(ws2) == fa.FA_OK
        rdq, rdk, rdv, _ = oracle.bwd(qf, kf, vf, dof, **oracle_args(w))
        check("dQ", dq.float().cpu().numpy(), rdq)
        check("dK", dk.float().cpu().numpy(), rdk)
        check("dV", dv.float().cpu().numpy(), rdv)


def test_wait_limit_gives_up_cleanly_e4m3():
    """The FP8 forward's give-up path, then a normal FP8 call on the same inputs that
    must agree bit for bit with one made before the failure."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    rng = np.random.default_rng(inputs.seed_of(122, 0, 0))
    B, s, h, dd = 1, 384, 2, 128
    mk = lambda: torch.from_numpy(inputs.e4m3_bits(rng.standard_normal((B, s, h, dd)).astype(np.float32) * 4)).cuda()  # noqa: E731
    q, k, v = mk(), mk(), mk()
    ref, _, ws = fa.forward(q, k, v, causal=True)
    assert fa.device_status(ws) == fa.FA_OK
    ref = ref.clone()
    _, _, ws = fa.forward(q, k, v, causal=True, wait_limit_ns=1)
    assert fa.device_status(ws) == fa.FA_ERR_TIMEOUT
    again, _, ws = fa.forward(q, k, v, causal=True)
    assert fa.device_status(ws) == fa.FA_OK
    assert torch.equal(again.view(torch.int16), ref.view(torch.int16))
