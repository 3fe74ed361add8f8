"""CPU emulation of the e4m3 forward's one lossy rounding point, for the pages' test rule.

The flash-attention test rule (vllm-project/flash-attention README, "Tests": the kernel's
maximum error at most twice that of a baseline run in the same low precision) needs a
baseline with the same low-precision step.  With e4m3 inputs the products of S = Q K^T are
exact and only fp32 summation rounds; the lossy step is P, rounded to e4m3 before P V.
Which values get rounded depends on the reference maximum P is taken against, so this
emulation follows the kernel's: per row, the running maximum over 128-key tiles, set by the
first tile that has an allowed key and moved only when a later tile raises it by more than
2^8 (in the exp2 domain).  Each key's P = 2^(s c - m_ref) is rounded to e4m3 (so the row's
largest P is usually not exactly 1 and carries a rounding error too), weighted by
2^(m_ref - m_final) as the kernel's rescaling of O does, normalised by the unrounded
weighted sum, and O is rounded to bf16.  It is not the oracle; it calibrates how much error
the e4m3 P alone causes.  Dense tensors only; kv_len optionally limits each batch entry's keys.
"""
import numpy as np

from exact_attention_bwd_gb300 import inputs
from bf16_emulation import keep_mask


def _ref_max(x, tile=128, lazy=8.0):
    """Per-key reference maximum of the kernel's online softmax for rows x [rows, keys]
    (exp2 domain, -inf = masked): the running max of 128-key tiles, moved only when a tile
    exceeds it by more than `lazy`.  Returns (m_ref [rows, keys], m_final [rows, 1])."""
    rows, n = x.shape
    m = np.full(rows, -np.inf)
    m_ref = np.full((rows, n), -np.inf)
    for t0 in range(0, n, tile):
        tm = x[:, t0:t0 + tile].max(axis=1) if n > t0 else np.full(rows, -np.inf)
        first = np.isneginf(m)
        grow = ~first & (tm > m + lazy)
        m = np.where(first, tm, np.where(grow, tm, m))
        m_ref[:, t0:t0 + tile] = m[:, None]
    return m_ref, m[:, None]


def fwd(q, k, v, *, scale, causal, window, sinks=None, kv_len=None):
    """q, k, v: fp32 true values [B, S, H, D]; returns O (bf16 values as fp32)."""
    B, s_q, h_q, d = q.shape
    _, s_kv, h_kv, _ = k.shape
    G = h_q // h_kv
    c = np.float32(scale * np.log2(np.e))
    o = np.zeros_like(q)
    for b in range(B):
        nk = s_kv if kv_len is None else int(kv_len[b])
        keep = keep_mask(s_q, nk, causal, *window)
        for h in range(h_q):
            g = h // G
            x = (q[b, :, h] @ k[b, :nk, g].T).astype(np.float32) * c
            x = np.where(keep, x, -np.inf)
            m_ref, m_fin = _ref_max(x.astype(np.float64))
            base = np.where(np.isfinite(m_ref), m_ref, 0.0).astype(np.float32)
            praw = np.exp2(x - base).astype(np.float32)
            pq = inputs.e4m3_to_f64(inputs.e4m3_bits(praw)).astype(np.float32)
            fin = np.where(np.isfinite(m_fin), m_fin, 0.0)
            w = np.where(np.isfinite(m_ref), np.exp2(base - fin), 0.0).astype(np.float32)
            z = (praw * w).sum(axis=1, keepdims=True)
            if sinks is not None:
                z = z + np.exp2(np.float32(sinks[h]) * np.float32(np.log2(np.e)) - fin) * (np.isfinite(m_fin))
                z = np.where(np.isfinite(m_fin), z, 1.0)  # rows without keys: O = 0
            zz = np.where(z > 0, z, 1.0)
            ob = ((pq * w) @ v[b, :nk, g]) / zz
            o[b, :, h] = inputs.bf16_to_f32(inputs.bf16_bits(ob.astype(np.float32)))
    return o
