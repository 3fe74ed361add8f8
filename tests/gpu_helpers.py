"""Shared helpers of the GPU parity tests: upload seeded bf16 bits, run the library,
compare with the fp64 oracle.

Tolerances against fp64: bf16 outputs O, dQ, dK, dV have mean-abs error <= 2e-3 and,
element by element, error <= 2e-2 + 2^-8 |ref|.  The 2e-2 absolute bound is the stated
one; the relative term is the bf16 format's own rounding (half an ulp is at most 2^-8 of
the value), which alone exceeds 2e-2 once |ref| > 5.12 — large dV / dK entries of long
grouped-query sums get there.  LSE: <= 1e-3 on finite entries, -inf entries equal.  The
sink gradient (a sum over every row of the head): <= 2e-2 relative to its magnitude.
"""
from __future__ import annotations

import numpy as np

from exact_attention_bwd_gb300 import inputs

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
BF16_HALF_ULP = 2.0 ** -8
LSE_ABS = 1e-3


def to_dev(bits, dtype="bf16"):
    """uint16 bit patterns -> a CUDA tensor of bf16 (or fp16 for dtype "f16")."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16).cuda()


def from_dev(t) -> np.ndarray:
    import torch
    return t.detach().float().cpu().numpy().astype(np.float64)


def dev_inputs(w):
    import torch
    t = w.get("dtype", "bf16")
    d = dict(q=to_dev(w["q"], t), k=to_dev(w["k"], t), v=to_dev(w["v"], t), dout=to_dev(w["dout"], t))
    d["sinks"] = None if w["sinks"] is None else torch.from_numpy(w["sinks"]).cuda()
    d["cu_q"] = None if w["cu_q"] is None else torch.from_numpy(w["cu_q"]).cuda()
    d["cu_k"] = None if w["cu_k"] is None else torch.from_numpy(w["cu_k"]).cuda()
    return d


def oracle_args(w):
    return dict(scale=w["scale"], causal=w["causal"], window=w["window"],
                sinks=None if w["sinks"] is None else w["sinks"].astype(np.float64),
                cu_q=w["cu_q"], cu_k=w["cu_k"])


def check(name, got, ref, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - ref)
    if not err.size:
        return 0.0, 0.0
    bound = max_abs + BF16_HALF_ULP * np.abs(ref)
    worst = int(np.argmax(err - bound))
    mx, mn = float(err.max()), float(err.mean())
    assert err.flat[worst] <= bound.flat[worst], (
        f"{name}: error {err.flat[worst]:.3e} at |ref| {abs(ref.flat[worst]):.3f} exceeds "
        f"{bound.flat[worst]:.3e}; max-abs {mx:.3e}")
    assert mn <= mean_abs, f"{name}: mean-abs {mn:.3e} > {mean_abs}"
    return mx, mn


def check_lse(name, got, ref, tol=LSE_ABS):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape
    fin = np.isfinite(ref)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), f"{name}: -inf pattern differs"
    if fin.any():
        err = float(np.abs(got[fin] - ref[fin]).max())
        assert err <= tol, f"{name}: max-abs {err:.3e} > {tol}"


def run_gpu(w, bwd=True, flags=0):
    """fa_fwd (+ fa_bwd) through the binding; returns numpy fp64 results."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    d = dev_inputs(w)
    kw = dict(causal=w["causal"], window=w["window"], softmax_scale=w["scale"], sinks=d["sinks"],
              cu_q=d["cu_q"], cu_k=d["cu_k"], flags=flags)
    o, lse, ws = fa.forward(d["q"], d["k"], d["v"], **kw)
    torch.cuda.synchronize()
    st = fa.device_status(ws)
    assert st == fa.FA_OK, f"device status {st} after the forward"
    out = dict(o=from_dev(o), lse=lse.cpu().numpy().astype(np.float64))
    if bwd:
        dq, dk, dv, ds, ws2 = fa.backward(d["q"], d["k"], d["v"], o, lse, d["dout"], **kw)
        torch.cuda.synchronize()
        st = fa.device_status(ws2)
        assert st == fa.FA_OK, f"device status {st} after the backward"
        out.update(dq=from_dev(dq), dk=from_dev(dk), dv=from_dev(dv),
                   dsinks=None if ds is None else ds.cpu().numpy().astype(np.float64))
    return out


def f64(w, key):
    return (inputs.f16_to_f64 if w.get("dtype") == "f16" else inputs.bf16_to_f64)(w[key])
