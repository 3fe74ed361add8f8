"""Shared helpers of the GPU parity tests: upload seeded bf16 bits, run the library,
compare with the fp64 oracle.

Tolerances against fp64: bf16 outputs O, dQ, dK, dV have mean-abs error <= 2e-3 and,
element by element, error <= 2e-2 + 2^-8 |ref|.  The 2e-2 absolute bound is the stated
one; the relative term is the bf16 format's own rounding (half an ulp is at most 2^-8 of
the value), which alone exceeds 2e-2 once |ref| > 5.12 — large dV / dK entries of long
grouped-query sums get there.  LSE: <= 1e-3 on finite entries, -inf entries equal.  The
sink gradient (a sum over every row of the head): <= 2e-2 relative to its magnitude.

Guard regions: run_gpu places every output (O, LSE, dQ, dK, dV, dsink) and both workspaces
inside a larger buffer filled with 0xFF bytes (a NaN in bf16, fp16 and fp32) and checks,
after each call, that the GUARD bytes before and after are untouched (no write out of
bounds) and, through the finiteness checks of the comparison, that every element inside
was written.  This stands in for a memory checker on the GPU.
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


def dev_inputs(w, share_cu=True):
    """Device copies of a workload's inputs.  When the query and key offsets are equal,
    one device array serves as both (unless share_cu is False), which is how a caller
    signals queries and keys packed alike and what lets the d <= 128 kernels tile the
    packed token axis; separate arrays with equal contents take the per-sequence tiles."""
    import torch
    t = w.get("dtype", "bf16")
    d = dict(q=to_dev(w["q"], t), k=to_dev(w["k"], t), v=to_dev(w["v"], t), dout=to_dev(w["dout"], t))
    d["sinks"] = None if w["sinks"] is None else torch.from_numpy(w["sinks"]).cuda()
    d["cu_q"] = None if w["cu_q"] is None else torch.from_numpy(w["cu_q"]).cuda()
    d["cu_k"] = None if w["cu_k"] is None else torch.from_numpy(w["cu_k"]).cuda()
    if share_cu and d["cu_q"] is not None and np.array_equal(w["cu_q"], w["cu_k"]):
        d["cu_k"] = d["cu_q"]
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


GUARD = 4096  # canary bytes before and after every guarded buffer


class Guarded:
    """A tensor of `shape` and `dtype` at byte offset GUARD of a buffer that is GUARD bytes
    longer on each side; the whole buffer starts as 0xFF bytes."""

    def __init__(self, shape, dtype, device="cuda"):
        import torch
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.nbytes = n
        self.buf = torch.full((n + 2 * GUARD,), 0xFF, dtype=torch.uint8, device=device)
        self.t = self.buf[GUARD:GUARD + n].view(dtype).view(tuple(shape)) if n else \
            torch.empty(tuple(shape), dtype=dtype, device=device)

    def check(self, name):
        import torch
        torch.cuda.synchronize()
        head = self.buf[:GUARD].cpu().numpy()
        tail = self.buf[GUARD + self.nbytes:].cpu().numpy()
        assert np.all(head == 0xFF), f"{name}: a write landed before the buffer (first at byte {np.argmax(head != 0xFF) - GUARD})"
        assert np.all(tail == 0xFF), f"{name}: a write landed past the end (first at byte +{np.argmax(tail != 0xFF)})"


def run_gpu(w, bwd=True, flags=0, share_cu=True):
    """fa_fwd (+ fa_bwd) through the binding, every output and workspace guarded; returns
    numpy fp64 results."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    d = dev_inputs(w, share_cu=share_cu)
    kw = dict(causal=w["causal"], window=w["window"], softmax_scale=w["scale"], sinks=d["sinks"],
              cu_q=d["cu_q"], cu_k=d["cu_k"], flags=flags)
    q, k, v = d["q"], d["k"], d["v"]
    p = fa.make_params(q, k, causal=kw["causal"], window=kw["window"], softmax_scale=kw["softmax_scale"],
                       sinks=kw["sinks"], cu_q=kw["cu_q"], cu_k=kw["cu_k"], flags=flags,
                       dtype=fa._type_code(q.dtype))
    lse_shape = (p.B, p.h_q, p.s_q) if d["cu_q"] is None else (p.h_q, p.s_q)
    g_o, g_lse = Guarded(q.shape, q.dtype), Guarded(lse_shape, torch.float32)
    g_ws = Guarded((fa.fa_fwd_workspace_size(p),), torch.uint8)
    o, lse, ws = fa.forward(q, k, v, **kw, out=g_o.t, lse=g_lse.t, workspace=g_ws.t)
    torch.cuda.synchronize()
    st = fa.device_status(ws)
    assert st == fa.FA_OK, f"device status {st} after the forward"
    for name, g in (("O", g_o), ("LSE", g_lse), ("forward workspace", g_ws)):
        g.check(name)
    out = dict(o=from_dev(o), lse=lse.cpu().numpy().astype(np.float64))
    if bwd:
        g_dq, g_dk, g_dv = Guarded(q.shape, q.dtype), Guarded(k.shape, k.dtype), Guarded(v.shape, v.dtype)
        g_ds = None if d["sinks"] is None else Guarded(d["sinks"].shape, torch.float32)
        g_ws2 = Guarded((fa.fa_bwd_workspace_size(p),), torch.uint8)
        grads = (g_dq.t, g_dk.t, g_dv.t, None if g_ds is None else g_ds.t)
        dq, dk, dv, ds, ws2 = fa.backward(q, k, v, o, lse, d["dout"], **kw, grads=grads, workspace=g_ws2.t)
        torch.cuda.synchronize()
        st = fa.device_status(ws2)
        assert st == fa.FA_OK, f"device status {st} after the backward"
        for name, g in (("dQ", g_dq), ("dK", g_dk), ("dV", g_dv), ("dsink", g_ds), ("backward workspace", g_ws2)):
            if g is not None:
                g.check(name)
        out.update(dq=from_dev(dq), dk=from_dev(dk), dv=from_dev(dv),
                   dsinks=None if ds is None else ds.cpu().numpy().astype(np.float64))
    return out


def f64(w, key):
    return (inputs.f16_to_f64 if w.get("dtype") == "f16" else inputs.bf16_to_f64)(w[key])
