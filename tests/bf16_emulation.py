"""CPU emulation of the tensor-core path's rounding points, for the pages' secondary rule.

The flash-attention test rule (vllm-project/flash-attention README and the FA2 README
copy, "Tests": the kernel's max error must be at most twice that of a reference run in
the same low precision) needs a low-precision reference.  This one takes the bf16
inputs, accumulates in fp32 and rounds to bf16 exactly where a bf16 tensor-core GEMM
must: P before P V and P^T dO, dS before dS^T Q and dS K, and every output.  It is not
the oracle (the oracle is fp64 and exact); it only calibrates how much error bf16
operands alone cause.  Dense tensors only.
"""
import numpy as np

from exact_attention_bwd_gb300 import inputs


def _r(x):
    return inputs.bf16_to_f32(inputs.bf16_bits(np.asarray(x, np.float32)))


def keep_mask(s_q, s_kv, causal, left, right):
    i = np.arange(s_q)[:, None]
    j = np.arange(s_kv)[None, :]
    off = s_kv - s_q
    m = np.ones((s_q, s_kv), bool)
    if causal:
        m &= j <= i + off
    if left >= 0:
        m &= j >= i + off - left
    if right >= 0:
        m &= j <= i + off + right
    return m


def fwd_bwd(q, k, v, do, *, scale, causal, window, sinks=None):
    """q, k, v, do: fp32 arrays holding bf16 values, [B, S, H, D]; returns bf16-rounded outputs."""
    B, s_q, h_q, d = q.shape
    _, s_kv, h_kv, _ = k.shape
    G = h_q // h_kv
    keep = keep_mask(s_q, s_kv, causal, *window)
    o = np.zeros_like(q)
    dq = np.zeros_like(q)
    dk = np.zeros((B, s_kv, h_kv, d), np.float32)
    dv = np.zeros((B, s_kv, h_kv, d), np.float32)
    for b in range(B):
        for h in range(h_q):
            g = h // G
            s = (q[b, :, h] @ k[b, :, g].T).astype(np.float32) * np.float32(scale)
            s = np.where(keep, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            if sinks is not None:
                m = np.maximum(m, sinks[h])
            m = np.where(np.isfinite(m), m, 0.0)
            e = np.exp(s - m)
            z = e.sum(axis=1, keepdims=True) + (np.exp(sinks[h] - m) if sinks is not None else 0.0)
            zz = np.where(z > 0, z, 1.0)
            p = (e / zz).astype(np.float32)
            ob = _r(_r(p) @ v[b, :, g])
            o[b, :, h] = ob
            delta = (do[b, :, h] * ob).sum(axis=1, keepdims=True)
            dp = do[b, :, h] @ v[b, :, g].T
            ds = (p * (dp - delta)).astype(np.float32)
            dv[b, :, g] += _r(p).T @ do[b, :, h]
            dk[b, :, g] += np.float32(scale) * (_r(ds).T @ q[b, :, h])
            dq[b, :, h] = _r(np.float32(scale) * (_r(ds) @ k[b, :, g]))
    return dict(o=o, dq=dq, dk=_r(dk), dv=_r(dv))
