"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module holds none of the attention arithmetic: it draws random numbers,
rounds them to bf16 (or fp16, e4m3) bit patterns and builds packed-sequence offsets.  The same
bits are uploaded to the GPU and widened to fp64 for the oracle, so both sides
see identical inputs.

Seed recipe: tensor seed = 1000 * workload + 10 * variant + tensor index, with
tensor index Q=0, K=1, V=2, dO=3, sinks=4, lengths=5.  Every draw uses numpy's
``Generator(PCG64(seed))``.
"""
from __future__ import annotations

import math

import numpy as np

Q, K, V, DO, SINKS, LENGTHS = range(6)


def seed_of(workload: int, variant: int, tensor: int) -> int:
    return 1000 * workload + 10 * variant + tensor


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def bf16_bits(x) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); returns uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    return r.astype(np.uint16)


def bf16_to_f32(bits) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def bf16_to_f64(bits) -> np.ndarray:
    return bf16_to_f32(bits).astype(np.float64)


def normal_bf16(seed: int, shape) -> np.ndarray:
    """i.i.d. N(0, 1) draws in fp32, rounded to bf16 bit patterns."""
    return bf16_bits(rng(seed).standard_normal(size=shape, dtype=np.float32))


def f16_bits(x) -> np.ndarray:
    """Round fp32 values to IEEE binary16 (round to nearest, ties to even; overflow to inf);
    returns uint16 bit patterns.  numpy's float32 -> float16 cast rounds this way."""
    with np.errstate(over="ignore"):  # overflow to inf is the format's rule
        return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def f16_to_f64(bits) -> np.ndarray:
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def normal_f32(seed: int, shape) -> np.ndarray:
    return rng(seed).standard_normal(size=shape, dtype=np.float32)


def varlen_lengths(seed: int, n: int = 256, total: int = 32768, median: float = 64.0,
                   sigma: float = 1.5, zero_frac: float = 0.10) -> np.ndarray:
    """Packed-batch sequence lengths.

    Log-normal draws (median ``median``, log-sd ``sigma``); round(zero_frac * n)
    slots, picked by a seeded permutation, are forced to 0; the rest are scaled
    to sum to ``total``, floored, clamped to at least 1, and the remainder goes
    to the largest fractional parts (taken back from the smallest fractional
    parts if the clamp overshot).
    """
    g = rng(seed)
    raw = g.lognormal(mean=math.log(median), sigma=sigma, size=n)
    n_zero = int(round(zero_frac * n))
    zero_idx = g.permutation(n)[:n_zero]
    keep = np.ones(n, bool)
    keep[zero_idx] = False
    lengths = np.zeros(n, np.int64)
    idx = np.nonzero(keep)[0]
    if len(idx) == 0:
        if total != 0:
            raise ValueError("no non-empty slot to hold the tokens")
        return lengths.astype(np.int32)
    scaled = raw[idx] * (total / raw[idx].sum())
    fl = np.maximum(np.floor(scaled).astype(np.int64), 1)
    frac = scaled - np.floor(scaled)
    rem = total - int(fl.sum())
    if rem > 0:
        order = np.argsort(-frac, kind="stable")
        fl[order[:rem]] += 1
    elif rem < 0:
        order = np.argsort(frac, kind="stable")
        for t in order:
            if rem == 0:
                break
            if fl[t] > 1:
                fl[t] -= 1
                rem += 1
    lengths[idx] = fl
    assert int(lengths.sum()) == total
    return lengths.astype(np.int32)


def cu_seqlens(lengths) -> np.ndarray:
    """int32 offsets [N+1] from 0 to the token count."""
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(len(lengths) + 1, np.int64)
    cu[1:] = np.cumsum(lengths)
    return cu.astype(np.int32)


# ----------------------------------------------------------------------------------------------
# The workloads.  Each is a dict of problem sizes; ``make`` draws its tensors.
# ----------------------------------------------------------------------------------------------

def workload(name: str, **over) -> dict:
    """Problem sizes of a named workload (keyword overrides allowed)."""
    w = dict(WORKLOADS[name])
    w.update(over)
    w.setdefault("name", name)
    return w


WORKLOADS = {
    # tiny forward+backward
    "tiny": dict(wid=1, B=1, s_q=128, s_kv=128, h_q=2, h_kv=2, d=64, causal=False,
                 window=(-1, -1), sinks=False, varlen=False),
    "tiny_causal": dict(wid=1, variant=1, B=1, s_q=128, s_kv=128, h_q=2, h_kv=2, d=64,
                        causal=True, window=(-1, -1), sinks=False, varlen=False),
    # dense sweep (fixed 16k tokens); the headline is s=8192 causal
    **{f"sweep_s{s}{'_causal' if c else ''}": dict(
        wid=2, variant=(2 * i + (1 if c else 0)), B=16384 // s, s_q=s, s_kv=s, h_q=16, h_kv=16,
        d=128, causal=c, window=(-1, -1), sinks=False, varlen=False)
       for i, s in enumerate((512, 1024, 2048, 4096, 8192, 16384)) for c in (False, True)},
    # grouped-query heads with sliding windows and sinks
    "gqa_window_causal": dict(wid=3, variant=0, B=2, s_q=4096, s_kv=4096, h_q=64, h_kv=8, d=64,
                              causal=True, window=(127, 0), sinks=True, varlen=False),
    "gqa_window_2sided": dict(wid=3, variant=1, B=2, s_q=4096, s_kv=4096, h_q=64, h_kv=8, d=64,
                              causal=False, window=(128, 128), sinks=True, varlen=False),
    # packed varlen
    "varlen": dict(wid=4, variant=0, B=256, T=32768, h_q=32, h_kv=32, d=128, causal=True,
                   window=(-1, -1), sinks=False, varlen=True),
    # head dim 256, forward and backward (16k tokens, 16 heads)
    "d256_s8192_causal": dict(wid=6, variant=0, B=2, s_q=8192, s_kv=8192, h_q=16, h_kv=16, d=256,
                              causal=True, window=(-1, -1), sinks=False, varlen=False),
    "d256_s4096": dict(wid=6, variant=1, B=4, s_q=4096, s_kv=4096, h_q=16, h_kv=16, d=256,
                       causal=False, window=(-1, -1), sinks=False, varlen=False),
    # head dim 192 (the padded size between 128 and 256), same token count
    "d192_s8192_causal": dict(wid=6, variant=2, B=2, s_q=8192, s_kv=8192, h_q=16, h_kv=16, d=192,
                              causal=True, window=(-1, -1), sinks=False, varlen=False),
    # decode / chunked prefill against a long cache
    **{f"decode_d{d}_sq{sq}": dict(wid=5, variant=(0 if d == 128 else 2) + (0 if sq == 1 else 1),
                                   B=64, s_q=sq, s_kv=32768, h_q=32, h_kv=8, d=d, causal=True,
                                   window=(-1, -1), sinks=False, varlen=False)
       for d in (128, 256) for sq in (1, 64)},
}


def make(w: dict) -> dict:
    """Draw the 16-bit bit patterns (uint16) and side inputs of workload ``w``.

    Returns q, k, v, dout (uint16, [B,S,H,D] or packed [T,H,D]), sinks (fp32 or
    None), cu_q / cu_k (int32 or None), and the sizes.  The N(0, 1) draws are rounded
    to bf16, or to fp16 when w["dtype"] == "f16" (the same fp32 draws either way).
    """
    wid, var = w["wid"], w.get("variant", 0)
    h_q, h_kv, d = w["h_q"], w["h_kv"], w["d"]
    out = dict(w)
    if w.get("varlen"):
        if "lengths" in w:
            lq = np.asarray(w["lengths"], np.int32)
            lk = np.asarray(w.get("lengths_k", lq), np.int32)
        else:
            lq = varlen_lengths(seed_of(wid, var, LENGTHS), n=w["B"], total=w["T"])
            lk = lq
        cu_q, cu_k = cu_seqlens(lq), cu_seqlens(lk)
        Tq, Tk = int(cu_q[-1]), int(cu_k[-1])
        qshape, kshape = (Tq, h_q, d), (Tk, h_kv, d)
        out.update(cu_q=cu_q, cu_k=cu_k, B=len(lq), s_q=Tq, s_kv=Tk)
    else:
        qshape = (w["B"], w["s_q"], h_q, d)
        kshape = (w["B"], w["s_kv"], h_kv, d)
        out.update(cu_q=None, cu_k=None)
    rnd = f16_bits if w.get("dtype") == "f16" else bf16_bits
    out["dtype"] = w.get("dtype", "bf16")
    out["q"] = rnd(normal_f32(seed_of(wid, var, Q), qshape))
    out["k"] = rnd(normal_f32(seed_of(wid, var, K), kshape))
    out["v"] = rnd(normal_f32(seed_of(wid, var, V), kshape))
    out["dout"] = rnd(normal_f32(seed_of(wid, var, DO), qshape))
    out["sinks"] = normal_f32(seed_of(wid, var, SINKS), (h_q,)) if w.get("sinks") else None
    out.setdefault("scale", 1.0 / math.sqrt(d))
    return out


def normal_bf16_torch(seed: int, shape, device):
    """i.i.d. N(0, 1) bf16 tensor drawn on `device` by torch's seeded Philox generator.

    For inputs too large to draw on the host in reasonable time (the long key/value
    caches); slices are copied back to the host for the oracle.
    """
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def normal_f16_torch(seed: int, shape, device):
    """The same draws as normal_bf16_torch, rounded to fp16 instead."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32).to(torch.float16)


def page_table(seed: int, B: int, max_blocks: int, num_pages: int) -> np.ndarray:
    """Block table of a paged key/value cache: int32 [B, max_blocks] page indices, a
    seeded draw of distinct pages (a permutation of the pool, cut to B * max_blocks)."""
    if num_pages < B * max_blocks:
        raise ValueError("the pool has fewer pages than the table needs")
    perm = rng(seed).permutation(num_pages)[: B * max_blocks]
    return perm.reshape(B, max_blocks).astype(np.int32)


def used_lengths(seed: int, B: int, s_kv: int) -> np.ndarray:
    """Filled lengths of B cache slots of s_kv keys: int32 [B], uniform on [0, s_kv], with
    the first slot full and (for B > 2) the second empty, so both ends are always covered."""
    n = rng(seed).integers(0, s_kv + 1, size=B).astype(np.int32)
    if B > 0:
        n[0] = s_kv
    if B > 2:
        n[1] = 0
    return n


# ----------------------------------------------------------------------------------------------
# e4m3 (fp8) inputs: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; largest finite
# value 448, subnormal spacing 2^-9, no infinities (0x7F / 0xFF are NaN)
# ----------------------------------------------------------------------------------------------

def e4m3_bits(x) -> np.ndarray:
    """Round to the nearest e4m3 value (ties to even), saturating at +-448; uint8 bit patterns."""
    x = np.asarray(x, np.float64)
    a = np.minimum(np.abs(x), 448.0)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.clip(ex - 1, -6, 8)                 # binade of a (subnormals share the -6 spacing)
    quantum = np.ldexp(1.0, e - 3)
    m = np.minimum(np.round(a / quantum) * quantum, 448.0)   # np.round: ties to even
    _, em = np.frexp(np.where(m > 0, m, 1.0))
    em = em - 1
    normal = m >= 2.0 ** -6
    field = np.where(normal, em + 7, 0).astype(np.int64)
    mant = np.where(normal, np.round((m / np.ldexp(1.0, em) - 1.0) * 8.0), np.round(m / 2.0 ** -9)).astype(np.int64)
    bits = (field << 3) | mant
    bits = np.where(m == 0, 0, bits)
    sign = np.signbit(x)  # kept on values that round to zero (-0), as the hardware conversion does
    return (bits | (sign.astype(np.int64) << 7)).astype(np.uint8)


def e4m3_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, np.uint8).astype(np.int64)
    s = np.where(b & 0x80, -1.0, 1.0)
    field = (b >> 3) & 0xF
    mant = b & 0x7
    val = np.where(field == 0, mant * 2.0 ** -9, (1.0 + mant / 8.0) * np.ldexp(1.0, field - 7))
    val = np.where((b & 0x7F) == 0x7F, np.nan, val)
    return s * val


def normal_e4m3(seed: int, shape, spread: float = 32.0) -> np.ndarray:
    """i.i.d. N(0, spread^2) draws rounded to e4m3 bit patterns (spread 32 keeps them well
    inside the format's range while using its full precision)."""
    return e4m3_bits(rng(seed).standard_normal(size=shape, dtype=np.float32).astype(np.float64) * spread)


def descales(seed: int, B: int, h_kv: int, spread: float = 32.0) -> np.ndarray:
    """Per-(batch, kv head) descale factors, fp32 [B * h_kv]: 1/spread times a seeded factor
    in [0.5, 2], so the true inputs have unit-order magnitudes that differ across heads."""
    f = np.exp2(rng(seed).uniform(-1.0, 1.0, size=B * h_kv))
    return (f / spread).astype(np.float32)
