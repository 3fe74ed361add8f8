"""Pins of the fp64 oracle against facts the pages and the mathematics fix.

Every check here is independent of the oracle's own code: invariants (rows of
P sum to one), closed forms (constant values, scale 0, a single allowed key),
library routines (scipy's logsumexp), worked examples printed on the pages
(tests/golden/), brute-force enumeration of the mask predicates stated on the
pages, equivalences (GQA vs repeated heads, packed vs unpacked) and central
finite differences for every gradient.
"""
import math
import os

import numpy as np
import pytest
from scipy.special import expit, logsumexp

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(seed, *shape, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _identity_v(B, s_kv, h_kv):
    """V whose head dim equals s_kv and whose row j is e_j, so that O = P."""
    v = np.zeros((B, s_kv, h_kv, s_kv))
    for j in range(s_kv):
        v[:, j, :, j] = 1.0
    return v


def _probs(q, k, *, scale=None, causal=False, window=(-1, -1), sinks=None):
    """P [B, h_q, s_q, s_kv] read out of the oracle's forward with V = I."""
    B, s_q, h_q, d = q.shape
    _, s_kv, h_kv, _ = k.shape
    # V = I needs the head dim of V equal to s_kv; the oracle takes one d for
    # q, k and v, so pad q and k with zero columns (the logits are unchanged).
    dd = max(d, s_kv)
    qp = np.zeros((B, s_q, h_q, dd))
    kp = np.zeros((B, s_kv, h_kv, dd))
    qp[..., :d] = q
    kp[..., :d] = k
    v = np.zeros((B, s_kv, h_kv, dd))
    v[..., :s_kv] = _identity_v(B, s_kv, h_kv)
    sc = (1.0 / math.sqrt(d)) if scale is None else scale
    o, lse, lse0 = oracle.fwd(qp, kp, v, scale=sc, causal=causal, window=window, sinks=sinks)
    return o[..., :s_kv].transpose(0, 2, 1, 3), lse, lse0


def _mask_bruteforce(s_q, s_kv, causal, left, right):
    """The keep-mask stated on the pages, enumerated index by index.

    vllm-project/flash-attention README, flash_attn_func docstring: query i
    attends to keys in [i + s_k - s_q - left, i + s_k - s_q + right], inclusive;
    -1 leaves a side open; causal keeps j <= i + s_k - s_q (bottom-right).
    """
    m = np.zeros((s_q, s_kv), bool)
    for i in range(s_q):
        for j in range(s_kv):
            keep = True
            if causal and j > i + s_kv - s_q:
                keep = False
            if left >= 0 and j < i + s_kv - s_q - left:
                keep = False
            if right >= 0 and j > i + s_kv - s_q + right:
                keep = False
            m[i, j] = keep
    return m


MASK_CASES = [
    (6, 6, False, (-1, -1)),
    (6, 6, True, (-1, -1)),
    (2, 5, True, (-1, -1)),
    (5, 2, True, (-1, -1)),
    (7, 7, False, (2, 1)),
    (7, 7, True, (2, 0)),
    (4, 9, False, (3, 3)),
    (9, 4, False, (1, 0)),
    (9, 4, True, (-1, 2)),
    (5, 8, False, (0, 0)),
    (8, 3, False, (-1, 0)),
]


# ----------------------------------------------------------------------------------------------
# probabilities, masks, LSE
# ----------------------------------------------------------------------------------------------

@pytest.mark.parametrize("s_q,s_kv,causal,window", MASK_CASES)
def test_mask_equals_bruteforce_predicate(s_q, s_kv, causal, window):
    q = _rand(1, 1, s_q, 2, 4)
    k = _rand(2, 1, s_kv, 1, 4)
    P, lse, _ = _probs(q, k, causal=causal, window=window)
    keep = _mask_bruteforce(s_q, s_kv, causal, *window)
    for h in range(2):
        assert np.array_equal(P[0, h] > 0, keep)
        # an empty row: zero output and LSE = -inf
        empty = ~keep.any(axis=1)
        assert np.all(np.isneginf(lse[0, h][empty]))
        assert np.all(np.isfinite(lse[0, h][~empty]))


def test_causal_golden_examples():
    """The 2x5 and 5x2 bottom-right causal masks printed on the pages."""
    lines = [l.split() for l in open(os.path.join(GOLDEN, "causal_bottom_right.txt"))
             if l.strip() and not l.startswith("#")]
    cases, cur = [], None
    for toks in lines:
        if toks[0].startswith("seqlen_q"):
            cur = (int(toks[0].split("=")[1]), int(toks[1].split("=")[1]), [])
            cases.append(cur)
        else:
            cur[2].append([int(t) for t in toks])
    assert len(cases) == 2
    for s_q, s_kv, rows in cases:
        expect = np.array(rows, bool)
        q = _rand(3, 1, s_q, 1, 3)
        k = _rand(4, 1, s_kv, 1, 3)
        P, lse, _ = _probs(q, k, causal=True)
        assert np.array_equal(P[0, 0] > 0, expect)
        # "If the row of the mask is all zero, the output will be zero."
        v = _rand(5, 1, s_kv, 1, 3)
        o, _, _ = oracle.fwd(q, k, v, causal=True)
        for i in range(s_q):
            if not expect[i].any():
                assert np.all(o[0, i, 0] == 0.0)


@pytest.mark.parametrize("s_q,s_kv,causal,window", MASK_CASES[:6])
@pytest.mark.parametrize("with_sinks", [False, True])
def test_rows_of_P_sum_to_one(s_q, s_kv, causal, window, with_sinks):
    q = _rand(10, 2, s_q, 4, 5, scale=2.0)
    k = _rand(11, 2, s_kv, 2, 5, scale=2.0)
    sinks = _rand(12, 4) if with_sinks else None
    P, lse, _ = _probs(q, k, causal=causal, window=window, sinks=sinks)
    rowsum = P.sum(axis=-1)
    keep = _mask_bruteforce(s_q, s_kv, causal, *window)
    nonempty = keep.any(axis=1)
    if with_sinks:
        # the sink's share completes every row, empty rows included
        share = np.exp(sinks[None, :, None] - lse)
        np.testing.assert_allclose(rowsum + share, 1.0, rtol=0, atol=1e-12)
    else:
        np.testing.assert_allclose(rowsum[..., nonempty], 1.0, rtol=0, atol=1e-12)
        assert np.all(rowsum[..., ~nonempty] == 0.0)
    assert np.all(P >= 0)


@pytest.mark.parametrize("causal,window", [(False, (-1, -1)), (True, (-1, -1)), (False, (3, 2))])
def test_lse_equals_library_logsumexp(causal, window):
    B, s_q, s_kv, h_q, h_kv, d = 2, 9, 11, 4, 2, 6
    q = _rand(20, B, s_q, h_q, d, scale=3.0)
    k = _rand(21, B, s_kv, h_kv, d, scale=3.0)
    v = _rand(22, B, s_kv, h_kv, d)
    sinks = _rand(23, h_q)
    scale = 0.37
    keep = _mask_bruteforce(s_q, s_kv, causal, *window)
    _, lse, lse0 = oracle.fwd(q, k, v, scale=scale, causal=causal, window=window, sinks=sinks)
    G = h_q // h_kv
    for b in range(B):
        for h in range(h_q):
            logits = scale * np.einsum("id,jd->ij", q[b, :, h], k[b, :, h // G])
            for i in range(s_q):
                x = logits[i][keep[i]]
                ref0 = logsumexp(x) if len(x) else -np.inf
                ref = logsumexp(np.append(x, sinks[h]))
                assert lse0[b, h, i] == pytest.approx(ref0, abs=1e-12) or (
                    np.isneginf(ref0) and np.isneginf(lse0[b, h, i]))
                assert lse[b, h, i] == pytest.approx(ref, abs=1e-12)


def test_lse_extreme_logits_mpmath():
    """Logits near the fp64 exp range: LSE from 60-digit arithmetic."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 60
    q = np.array([[[[30.0, -20.0]]], ])  # [1,1,1,2]
    k = np.array([[[[10.0, 1.0]], [[9.5, -3.0]], [[-8.0, 2.0]]]])  # [1,3,1,2]
    v = _rand(30, 1, 3, 1, 2)
    scale = 2.0
    _, lse, _ = oracle.fwd(q, k, v, scale=scale)
    logits = [scale * (30.0 * k[0, j, 0, 0] - 20.0 * k[0, j, 0, 1]) for j in range(3)]
    ref = mpmath.log(sum(mpmath.e ** mpmath.mpf(x) for x in logits))
    assert abs(lse[0, 0, 0] - float(ref)) <= 1e-12 * abs(float(ref))


# ----------------------------------------------------------------------------------------------
# closed forms of the output
# ----------------------------------------------------------------------------------------------

@pytest.mark.parametrize("causal,window", [(False, (-1, -1)), (True, (-1, -1)), (False, (2, 3)),
                                           (True, (4, 0))])
def test_constant_value_rows_give_the_constant(causal, window):
    B, s_q, s_kv, h_q, h_kv, d = 2, 7, 7, 4, 2, 5
    q = _rand(40, B, s_q, h_q, d)
    k = _rand(41, B, s_kv, h_kv, d)
    c = _rand(42, B, 1, h_kv, d)
    v = np.repeat(c, s_kv, axis=1)
    o, _, _ = oracle.fwd(q, k, v, causal=causal, window=window)
    keep = _mask_bruteforce(s_q, s_kv, causal, *window)
    G = h_q // h_kv
    for h in range(h_q):
        for i in range(s_q):
            if keep[i].any():
                np.testing.assert_allclose(o[:, i, h], c[:, 0, h // G], rtol=0, atol=1e-13)


def test_constant_values_with_sinks_scale_by_sigmoid():
    B, s, h_q, h_kv, d = 1, 6, 2, 1, 3
    q = _rand(50, B, s, h_q, d)
    k = _rand(51, B, s, h_kv, d)
    c = np.array([1.5, -2.0, 0.25])
    v = np.broadcast_to(c, (B, s, h_kv, d)).copy()
    sinks = np.array([0.3, -1.2])
    o, lse, lse0 = oracle.fwd(q, k, v, causal=True, sinks=sinks)
    for h in range(h_q):
        for i in range(s):
            share = expit(lse0[0, h, i] - sinks[h])
            np.testing.assert_allclose(o[0, i, h], c * share, rtol=1e-13, atol=1e-14)


def test_single_allowed_key_returns_its_value():
    # window (0, 0) with s_q == s_kv keeps exactly the diagonal key
    B, s, h, d = 2, 9, 3, 4
    q = _rand(60, B, s, h, d)
    k = _rand(61, B, s, h, d)
    v = _rand(62, B, s, h, d)
    o, _, _ = oracle.fwd(q, k, v, window=(0, 0))
    np.testing.assert_array_equal(o, v)
    # first causal row sees only key 0
    o, _, _ = oracle.fwd(q, k, v, causal=True)
    np.testing.assert_array_equal(o[:, 0], v[:, 0])


@pytest.mark.parametrize("s_q,s_kv,causal,window", MASK_CASES)
def test_scale_zero_gives_mean_over_allowed_keys(s_q, s_kv, causal, window):
    q = _rand(70, 1, s_q, 2, 3)
    k = _rand(71, 1, s_kv, 2, 3)
    v = _rand(72, 1, s_kv, 2, 3)
    o, lse, _ = oracle.fwd(q, k, v, scale=0.0, causal=causal, window=window)
    keep = _mask_bruteforce(s_q, s_kv, causal, *window)
    for h in range(2):
        for i in range(s_q):
            n = keep[i].sum()
            if n:
                np.testing.assert_allclose(o[0, i, h], v[0, keep[i], h].mean(axis=0), rtol=1e-13,
                                           atol=1e-14)
                assert lse[0, h, i] == pytest.approx(math.log(n), abs=1e-13)
            else:
                assert np.all(o[0, i, h] == 0)


def test_sink_identity_from_the_pages():
    """O_sink = O_nosink * sigmoid(lse - sink), with lse the sink-less LSE.

    dew-flash-attn PyPI page, the sinks paragraph.
    """
    B, s, h_q, h_kv, d = 2, 8, 4, 2, 6
    q = _rand(80, B, s, h_q, d)
    k = _rand(81, B, s, h_kv, d)
    v = _rand(82, B, s, h_kv, d)
    sinks = _rand(83, h_q) * 2
    for causal, window in [(False, (-1, -1)), (True, (3, 0)), (False, (2, 2))]:
        o0, l0, _ = oracle.fwd(q, k, v, causal=causal, window=window)
        o1, l1, l1_nosink = oracle.fwd(q, k, v, causal=causal, window=window, sinks=sinks)
        np.testing.assert_array_equal(l0, l1_nosink)
        share = expit(l0 - sinks[None, :, None])          # [B, h, s]
        np.testing.assert_allclose(o1, o0 * share.transpose(0, 2, 1)[..., None], rtol=1e-12,
                                   atol=1e-14)
        np.testing.assert_allclose(l1, np.logaddexp(l0, sinks[None, :, None]), rtol=0, atol=1e-12)


def test_empty_rows_with_sinks():
    # s_q > s_kv causal: the first rows see no key
    q = _rand(90, 1, 5, 2, 3)
    k = _rand(91, 1, 2, 1, 3)
    v = _rand(92, 1, 2, 1, 3)
    sinks = np.array([0.7, -0.4])
    o, lse, lse0 = oracle.fwd(q, k, v, causal=True, sinks=sinks)
    for i in range(3):
        assert np.all(o[0, i] == 0)
        np.testing.assert_array_equal(lse[0, :, i], sinks)
        assert np.all(np.isneginf(lse0[0, :, i]))
    dout = _rand(93, 1, 5, 2, 3)
    dq, dk, dv, ds = oracle.bwd(q, k, v, dout, causal=True, sinks=sinks)
    assert np.all(dq[0, :3] == 0)


# ----------------------------------------------------------------------------------------------
# grouped-query heads and packed batches
# ----------------------------------------------------------------------------------------------

def test_gqa_head_map_golden():
    lines = [l.split() for l in open(os.path.join(GOLDEN, "gqa_head_map.txt"))
             if l.strip() and not l.startswith("#")]
    h_q = int(lines[0][0].split("=")[1])
    h_kv = int(lines[0][1].split("=")[1])
    expect = [int(t) for t in lines[1]]
    # a key/value head whose values are all equal to its index reveals the map
    s, d = 4, 2
    q = _rand(100, 1, s, h_q, d)
    k = _rand(101, 1, s, h_kv, d)
    v = np.zeros((1, s, h_kv, d))
    for g in range(h_kv):
        v[:, :, g, :] = g
    o, _, _ = oracle.fwd(q, k, v)
    got = [int(round(o[0, 0, h, 0])) for h in range(h_q)]
    assert got == expect


@pytest.mark.parametrize("causal,window,with_sinks", [(False, (-1, -1), False), (True, (-1, -1), True),
                                                      (False, (2, 1), True)])
def test_gqa_equals_repeated_kv_heads(causal, window, with_sinks):
    B, s_q, s_kv, h_q, h_kv, d = 2, 6, 8, 6, 2, 4
    q = _rand(110, B, s_q, h_q, d)
    k = _rand(111, B, s_kv, h_kv, d)
    v = _rand(112, B, s_kv, h_kv, d)
    dout = _rand(113, B, s_q, h_q, d)
    sinks = _rand(114, h_q) if with_sinks else None
    G = h_q // h_kv
    kr = np.repeat(k, G, axis=2)
    vr = np.repeat(v, G, axis=2)
    kw = dict(causal=causal, window=window, sinks=sinks)
    o, l, _ = oracle.fwd(q, k, v, **kw)
    orr, lr, _ = oracle.fwd(q, kr, vr, **kw)
    np.testing.assert_array_equal(o, orr)
    np.testing.assert_array_equal(l, lr)
    dq, dk, dv, ds = oracle.bwd(q, k, v, dout, **kw)
    dqr, dkr, dvr, dsr = oracle.bwd(q, kr, vr, dout, **kw)
    np.testing.assert_allclose(dq, dqr, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dk, dkr.reshape(B, s_kv, h_kv, G, d).sum(3), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv, dvr.reshape(B, s_kv, h_kv, G, d).sum(3), rtol=1e-12, atol=1e-13)
    if with_sinks:
        np.testing.assert_allclose(ds, dsr, rtol=1e-12, atol=1e-14)


def _golden_cu():
    toks = [l.split() for l in open(os.path.join(GOLDEN, "varlen_offsets.txt"))
            if l.strip() and not l.startswith("#")]
    return np.array([int(t) for t in toks[0]], np.int32)


@pytest.mark.parametrize("cu_q,cu_k,causal,window", [
    (None, None, True, (-1, -1)),                    # the pages' [0, 17, 300, 428] packing
    ([0, 3, 3, 10, 11, 11], [0, 5, 9, 15, 15, 21], True, (-1, -1)),   # zero-length, cu_q != cu_k
    ([0, 4, 4, 12], [0, 1, 7, 7], False, (2, 1)),
    ([0, 0, 0], [0, 0, 4], False, (-1, -1)),         # all queries empty
])
def test_varlen_equals_unpacked_runs(cu_q, cu_k, causal, window):
    if cu_q is None:
        cu_q = cu_k = _golden_cu()
        h_q, h_kv, d = 2, 1, 3
    else:
        h_q, h_kv, d = 4, 2, 3
    cu_q = np.asarray(cu_q, np.int32)
    cu_k = np.asarray(cu_k, np.int32)
    Tq, Tk = int(cu_q[-1]), int(cu_k[-1])
    q = _rand(120, Tq, h_q, d)
    k = _rand(121, Tk, h_kv, d)
    v = _rand(122, Tk, h_kv, d)
    dout = _rand(123, Tq, h_q, d)
    sinks = _rand(124, h_q)
    kw = dict(causal=causal, window=window, sinks=sinks)
    o, lse, _ = oracle.fwd(q, k, v, cu_q=cu_q, cu_k=cu_k, **kw)
    dq, dk, dv, ds = oracle.bwd(q, k, v, dout, cu_q=cu_q, cu_k=cu_k, **kw)
    ds_sum = np.zeros(h_q)
    for b in range(len(cu_q) - 1):
        a, e = cu_q[b], cu_q[b + 1]
        ka, ke = cu_k[b], cu_k[b + 1]
        if e == a:
            continue
        ob, lb, _ = oracle.fwd(q[None, a:e], k[None, ka:ke], v[None, ka:ke], **kw)
        np.testing.assert_array_equal(o[a:e], ob[0])
        np.testing.assert_array_equal(lse[:, a:e], lb[0])
        dqb, dkb, dvb, dsb = oracle.bwd(q[None, a:e], k[None, ka:ke], v[None, ka:ke],
                                        dout[None, a:e], **kw)
        np.testing.assert_array_equal(dq[a:e], dqb[0])
        np.testing.assert_array_equal(dk[ka:ke], dkb[0])
        np.testing.assert_array_equal(dv[ka:ke], dvb[0])
        ds_sum += dsb
    np.testing.assert_allclose(ds, ds_sum, rtol=1e-13, atol=1e-15)
    # keys of a sequence with no queries get no gradient
    for b in range(len(cu_q) - 1):
        if cu_q[b + 1] == cu_q[b]:
            assert np.all(dk[cu_k[b]:cu_k[b + 1]] == 0)


# ----------------------------------------------------------------------------------------------
# backward: central finite differences of L = sum(O * dO)
# ----------------------------------------------------------------------------------------------

FD_CASES = [
    dict(s=5, causal=False, window=(-1, -1), sinks=False),
    dict(s=7, causal=True, window=(-1, -1), sinks=False),
    dict(s=7, causal=False, window=(2, 1), sinks=True),
    dict(s=5, causal=True, window=(1, 0), sinks=True),
    dict(s=7, causal=True, window=(-1, -1), sinks=True, s_kv=5),
]


@pytest.mark.parametrize("case", FD_CASES, ids=lambda c: str(c))
def test_backward_matches_finite_differences(case):
    B, h_q, h_kv, d = 1, 4, 2, 4
    s_q = case["s"]
    s_kv = case.get("s_kv", s_q)
    q = _rand(130, B, s_q, h_q, d)
    k = _rand(131, B, s_kv, h_kv, d)
    v = _rand(132, B, s_kv, h_kv, d)
    dout = _rand(133, B, s_q, h_q, d)
    sinks = _rand(134, h_q) if case["sinks"] else None
    scale = 0.6
    kw = dict(scale=scale, causal=case["causal"], window=case["window"])

    def loss(q_, k_, v_, s_):
        o, _, _ = oracle.fwd(q_, k_, v_, sinks=s_, **kw)
        return float(np.sum(o * dout))

    dq, dk, dv, ds = oracle.bwd(q, k, v, dout, sinks=sinks, **kw)
    eps = 1e-6

    def fd(arr, which):
        g = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            a1 = arr.copy()
            a1[idx] += eps
            a2 = arr.copy()
            a2[idx] -= eps
            args1 = dict(q_=q, k_=k, v_=v, s_=sinks)
            args2 = dict(args1)
            args1[which] = a1
            args2[which] = a2
            g[idx] = (loss(**args1) - loss(**args2)) / (2 * eps)
        return g

    for got, arr, which in [(dq, q, "q_"), (dk, k, "k_"), (dv, v, "v_")]:
        ref = fd(arr, which)
        err = np.abs(got - ref).max()
        assert err <= 1e-6 * max(1.0, np.abs(ref).max()), (which, err)
    if sinks is not None:
        ref = fd(sinks, "s_")
        assert np.abs(ds - ref).max() <= 1e-6 * max(1.0, np.abs(ref).max())


def test_backward_finite_differences_packed():
    cu = np.array([0, 3, 3, 7], np.int32)
    h_q, h_kv, d = 2, 1, 3
    q = _rand(140, 7, h_q, d)
    k = _rand(141, 7, h_kv, d)
    v = _rand(142, 7, h_kv, d)
    dout = _rand(143, 7, h_q, d)
    sinks = _rand(144, h_q)
    kw = dict(causal=True, window=(-1, -1), cu_q=cu, cu_k=cu, sinks=sinks)
    dq, dk, dv, ds = oracle.bwd(q, k, v, dout, **kw)
    eps = 1e-6
    for got, name in [(dq, "q"), (dk, "k"), (dv, "v")]:
        base = dict(q=q, k=k, v=v)
        arr = base[name]
        ref = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a1, a2 = arr.copy(), arr.copy()
            a1[idx] += eps
            a2[idx] -= eps
            b1, b2 = dict(base), dict(base)
            b1[name], b2[name] = a1, a2
            o1 = oracle.fwd(b1["q"], b1["k"], b1["v"], **kw)[0]
            o2 = oracle.fwd(b2["q"], b2["k"], b2["v"], **kw)[0]
            ref[idx] = (np.sum(o1 * dout) - np.sum(o2 * dout)) / (2 * eps)
        assert np.abs(got - ref).max() <= 1e-6 * max(1.0, np.abs(ref).max()), name


def test_softmax_of_printed_vector():
    """Tutorial section 2 applies softmax to [1, 2, 3]; the oracle's P matches scipy's softmax."""
    from scipy.special import softmax
    q = np.ones((1, 1, 1, 1))
    k = np.array([1.0, 2.0, 3.0]).reshape(1, 3, 1, 1)
    P, _, _ = _probs(q, k, scale=1.0)
    np.testing.assert_allclose(P[0, 0, 0], softmax([1.0, 2.0, 3.0]), rtol=1e-14, atol=0)
