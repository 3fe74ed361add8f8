"""Work accounting for the benchmark: allowed (query, key) pairs and FLOPs.

The FLOP convention is the one the throughput tables on the pages use: the
forward counts 4 * d FLOPs per allowed (query, key) pair and head (two
multiply-adds per element for Q K^T and for P V), the backward 2.5 times that,
and forward+backward 3.5 times (jax-flash-attn3 README, the benchmark table).
"""
from __future__ import annotations

import numpy as np


def fwd_pairs(w: dict) -> int:
    """Number of allowed (query, key) pairs summed over sequences and query heads.

    Pure counting of the mask's interval sizes per row; the FLOP convention is
    4 * d * pairs for the forward and 2.5x that for the backward.
    """
    causal, (left, right) = w["causal"], w["window"]
    if w.get("varlen") or w.get("cu_q") is not None:
        cu_q, cu_k = w["cu_q"], w["cu_k"]
        seqs = [(int(cu_q[b + 1] - cu_q[b]), int(cu_k[b + 1] - cu_k[b])) for b in range(len(cu_q) - 1)]
    else:
        seqs = [(w["s_q"], w["s_kv"])] * w["B"]
    total = 0
    for nq, nk in seqs:
        i = np.arange(nq, dtype=np.int64)
        off = nk - nq
        hi = np.full(nq, nk - 1, np.int64)
        lo = np.zeros(nq, np.int64)
        if causal:
            hi = np.minimum(hi, i + off)
        if right >= 0:
            hi = np.minimum(hi, i + off + right)
        if left >= 0:
            lo = np.maximum(lo, i + off - left)
        total += int(np.maximum(hi - lo + 1, 0).sum())
    return total * w["h_q"]


def fwd_flops(w: dict) -> float:
    return 4.0 * w["d"] * fwd_pairs(w)


def bwd_flops(w: dict) -> float:
    return 2.5 * fwd_flops(w)


def _tokens(w: dict):
    """(query rows, key rows) over the batch: B s_q and B s_kv, or the packed totals."""
    if w.get("varlen") or w.get("cu_q") is not None:
        return int(w["cu_q"][-1]) if w.get("cu_q") is not None else w["T"], \
            int(w["cu_k"][-1]) if w.get("cu_k") is not None else w["T"]
    return w["B"] * w["s_q"], w["B"] * w["s_kv"]


def fwd_bytes(w: dict, elem: int = 2) -> float:
    """Algorithmic HBM bytes of the forward: Q, K, V read once, O written (16-bit elements)
    and the fp32 LSE written."""
    tq, tk = _tokens(w)
    return elem * (2 * tq * w["h_q"] * w["d"] + 2 * tk * w["h_kv"] * w["d"]) + 4 * tq * w["h_q"]


def bwd_bytes(w: dict, elem: int = 2) -> float:
    """Algorithmic HBM bytes of the backward: Q, O, dO read and dQ written; K, V read and
    dK, dV written (16-bit elements); the fp32 LSE read."""
    tq, tk = _tokens(w)
    return elem * (4 * tq * w["h_q"] * w["d"] + 4 * tk * w["h_kv"] * w["d"]) + 4 * tq * w["h_q"]
