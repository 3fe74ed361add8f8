"""GPU parity of the key/value-cache forms of the forward: partly filled cache slots
(seqused_k) and paged caches (block_table), against the fp64 oracle.

The oracle knows neither form; each case is restated for it as the attention problem the
form defines.  A slot filled to n keys is a sequence of n keys (fa4-jax, "Varlen
semantics": only the first seqused[b] tokens of slot b take part, bottom-right alignment
on that length), so a batch of B slots is a packed batch with query offsets b * s_q and
key offsets from the filled lengths.  A paged cache holds key j of sequence b in row
j % page_size of page block_table[b][j / page_size] (vllm-project/flash-attention README,
flash_attn_with_kvcache); the test gathers the pages into the dense cache they stand for.
Both restatements are plain indexing, done here on the host; the attention itself is the
oracle's.

The shapes reach every forward kernel: the CUDA-core decode kernel (few query rows per
key/value head), the split tensor-core forward (chunked prefill), the unsplit tensor-core
forward (d = 64 / 128), and the d = 256 forward, with ragged, full and empty slots.
"""
import numpy as np
import pytest

import oracle
from exact_attention_bwd_gb300 import inputs
from gpu_helpers import check, check_lse, to_dev, from_dev

pytestmark = pytest.mark.gpu

WID = 120
USED = 6   # tensor index of the filled lengths
TABLE = 7  # tensor index of the block table


def case(variant, *, B, s_q, s_kv, h_q, h_kv, d, causal=True, window=(-1, -1), sinks=False, used=True,
         page_size=None, spare_pages=3):
    """Seeded problem: q [B, s_q, h_q, d]; a dense cache [B, s_kv, h_kv, d] or a page pool
    [num_pages, page_size, h_kv, d] with its table; the filled lengths (or None)."""
    sd = lambda t: inputs.seed_of(WID, variant, t)  # noqa: E731
    c = dict(B=B, s_q=s_q, s_kv=s_kv, h_q=h_q, h_kv=h_kv, d=d, causal=causal, window=window,
             scale=1.0 / np.sqrt(d), page_size=page_size)
    c["q"] = inputs.normal_bf16(sd(inputs.Q), (B, s_q, h_q, d))
    if page_size is None:
        kshape = (B, s_kv, h_kv, d)
        c["table"] = None
    else:
        max_blocks = -(-s_kv // page_size)
        num_pages = B * max_blocks + spare_pages
        kshape = (num_pages, page_size, h_kv, d)
        c["table"] = inputs.page_table(sd(TABLE), B, max_blocks, num_pages)
    c["k"] = inputs.normal_bf16(sd(inputs.K), kshape)
    c["v"] = inputs.normal_bf16(sd(inputs.V), kshape)
    c["sinks"] = inputs.normal_f32(sd(inputs.SINKS), (h_q,)) if sinks else None
    c["used"] = inputs.used_lengths(sd(USED), B, s_kv) if used else None
    return c


def dense_cache(c, key):
    """The [B, s_kv, h_kv, d] cache a case's keys (or values) stand for."""
    x = c[key]
    if c["table"] is None:
        return x
    j = np.arange(c["s_kv"])
    ps = c["page_size"]
    return x[c["table"][:, j // ps], j % ps]


def oracle_of(c):
    """Oracle O [B, s_q, h_q, d] and LSE [B, h_q, s_q] of a case."""
    B, s_q, h_q, d = c["B"], c["s_q"], c["h_q"], c["d"]
    used = c["used"] if c["used"] is not None else np.full(B, c["s_kv"], np.int32)
    kd, vd = dense_cache(c, "k"), dense_cache(c, "v")
    k = np.concatenate([kd[b, :used[b]] for b in range(B)])
    v = np.concatenate([vd[b, :used[b]] for b in range(B)])
    cu_q = (np.arange(B + 1) * s_q).astype(np.int32)
    cu_k = inputs.cu_seqlens(used)
    q = inputs.bf16_to_f64(c["q"]).reshape(B * s_q, h_q, d)
    o, lse, _ = oracle.fwd(q, inputs.bf16_to_f64(k), inputs.bf16_to_f64(v), scale=c["scale"], causal=c["causal"],
                           window=c["window"], sinks=None if c["sinks"] is None else c["sinks"].astype(np.float64),
                           cu_q=cu_q, cu_k=cu_k)
    return o.reshape(B, s_q, h_q, d), lse.reshape(h_q, B, s_q).transpose(1, 0, 2)


def gpu_of(c, flags=0):
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    q, k, v = to_dev(c["q"]), to_dev(c["k"]), to_dev(c["v"])
    sinks = None if c["sinks"] is None else torch.from_numpy(c["sinks"]).cuda()
    used = None if c["used"] is None else torch.from_numpy(c["used"]).cuda()
    table = None if c["table"] is None else torch.from_numpy(c["table"]).cuda()
    o, lse, ws = fa.forward(q, k, v, causal=c["causal"], window=c["window"], softmax_scale=c["scale"], sinks=sinks,
                            seqused_k=used, block_table=table, s_kv=c["s_kv"] if table is not None else None,
                            flags=flags)
    torch.cuda.synchronize()
    assert fa.device_status(ws) == fa.FA_OK
    return from_dev(o), lse.cpu().numpy().astype(np.float64)


def compare(c, flags=0):
    o, lse = gpu_of(c, flags)
    ro, rl = oracle_of(c)
    check("O", o, ro)
    check_lse("LSE", lse, rl)
    return o, lse


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("s_q", [1, 2])
def test_seqused_decode(d, s_q):
    """Few query rows per key/value head: the CUDA-core decode kernel with split keys."""
    c = case(10 * d + s_q, B=5, s_q=s_q, s_kv=3000, h_q=8, h_kv=2, d=d)
    o, lse = compare(c)
    # the empty slot: zero output, -inf log-sum-exp
    assert np.all(o[1] == 0) and np.all(np.isneginf(lse[1]))


@pytest.mark.parametrize("d", [64, 128, 256])
def test_seqused_chunked_prefill(d):
    """64 queries against a long, partly filled cache: the split tensor-core forward; slots
    shorter than the chunk leave their first queries without keys (bottom-right)."""
    c = case(d, B=4, s_q=64, s_kv=2100, h_q=8, h_kv=2, d=d)
    c["used"][2] = 40
    compare(c)


@pytest.mark.parametrize("d", [64, 128])
def test_seqused_prefill_window_sinks(d):
    c = case(3 * d, B=3, s_q=300, s_kv=520, h_q=8, h_kv=2, d=d, causal=False, window=(100, 30), sinks=True)
    compare(c)


def test_seqused_packed_batch():
    """seqused_k on a packed batch: each sequence uses the first seqused_k[b] keys of its
    own key range."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    lq, lk = [5, 130, 0, 64, 200], [300, 140, 20, 64, 250]
    used = np.array([300, 17, 5, 0, 251], np.int32)   # the last one exceeds its range: clamped
    w = inputs.make(dict(wid=WID, variant=90, h_q=4, h_kv=2, d=128, causal=True, window=(-1, -1), sinks=False,
                         varlen=True, lengths=lq, lengths_k=lk))
    dev = lambda a: torch.from_numpy(a).cuda()  # noqa: E731
    o, lse, ws = fa.forward(to_dev(w["q"]), to_dev(w["k"]), to_dev(w["v"]), causal=True, softmax_scale=w["scale"],
                            cu_q=dev(w["cu_q"]), cu_k=dev(w["cu_k"]), seqused_k=dev(used))
    torch.cuda.synchronize()
    assert fa.device_status(ws) == fa.FA_OK
    eff = np.minimum(used, np.asarray(lk, np.int32))
    k = inputs.bf16_to_f64(w["k"])
    v = inputs.bf16_to_f64(w["v"])
    ks = np.concatenate([k[w["cu_k"][b]:w["cu_k"][b] + eff[b]] for b in range(len(lk))])
    vs = np.concatenate([v[w["cu_k"][b]:w["cu_k"][b] + eff[b]] for b in range(len(lk))])
    ro, rl, _ = oracle.fwd(inputs.bf16_to_f64(w["q"]), ks, vs, scale=w["scale"], causal=True, cu_q=w["cu_q"],
                           cu_k=inputs.cu_seqlens(eff))
    check("O", from_dev(o), ro)
    check_lse("LSE", lse.cpu().numpy().astype(np.float64), rl)


@pytest.mark.parametrize("d,s_q,page", [(128, 1, 256), (64, 2, 128), (256, 1, 256), (128, 64, 256),
                                        (256, 64, 128), (64, 200, 128), (128, 300, 256)])
def test_paged_cache(d, s_q, page):
    """Pages drawn as a seeded permutation of a pool with spare pages; the logical length is
    not a multiple of the page size."""
    c = case(500 + d + s_q + page, B=3, s_q=s_q, s_kv=1000, h_q=8, h_kv=2, d=d, page_size=page, used=False)
    compare(c)


@pytest.mark.parametrize("d,s_q", [(128, 1), (128, 64), (256, 2), (64, 130)])
def test_paged_cache_with_seqused(d, s_q):
    c = case(700 + d + s_q, B=4, s_q=s_q, s_kv=1300, h_q=8, h_kv=4, d=d, page_size=256, sinks=True)
    compare(c)


def test_paged_equals_dense():
    """The same cache, paged and dense, gives the same bits (same kernels, same order)."""
    c = case(800, B=3, s_q=64, s_kv=1000, h_q=8, h_kv=2, d=128, page_size=256)
    o_p, lse_p = gpu_of(c)
    dense = dict(c, k=dense_cache(c, "k"), v=dense_cache(c, "v"), table=None, page_size=None)
    o_d, lse_d = gpu_of(dense)
    assert np.array_equal(o_p, o_d)
    assert np.array_equal(lse_p, lse_d)


@pytest.mark.parametrize("d", [128, 256])
def test_paged_decode_full_size(d):
    """The decode workload's size (B=64, s_kv=32768, h_q=32, h_kv=8, s_q=1) as a paged cache of
    256-key pages in seeded random order with partly filled slots: sampled sequences (the
    first, the last and two more, all heads) against the oracle on their gathered pages."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    B, s_kv, h_q, h_kv, ps = 64, 32768, 32, 8, 256
    dev = torch.device("cuda", 0)
    sd = lambda t: inputs.seed_of(WID, 900 + d, t)  # noqa: E731
    mb = s_kv // ps
    table = inputs.page_table(sd(TABLE), B, mb, B * mb)
    used = inputs.used_lengths(sd(USED), B, s_kv)
    q = inputs.normal_bf16_torch(sd(inputs.Q), (B, 1, h_q, d), dev)
    k = inputs.normal_bf16_torch(sd(inputs.K), (B * mb, ps, h_kv, d), dev)
    v = inputs.normal_bf16_torch(sd(inputs.V), (B * mb, ps, h_kv, d), dev)
    o, lse, ws = fa.forward(q, k, v, causal=True, softmax_scale=d ** -0.5, seqused_k=torch.from_numpy(used).to(dev),
                            block_table=torch.from_numpy(table).to(dev), s_kv=s_kv)
    torch.cuda.synchronize()
    assert fa.device_status(ws) == fa.FA_OK
    for b in (0, 1, 37, B - 1):
        n = int(used[b])
        pages = torch.from_numpy(table[b, : -(-n // ps)].astype(np.int64)).to(dev)
        kb = k.index_select(0, pages).reshape(-1, h_kv, d)[:n]
        vb = v.index_select(0, pages).reshape(-1, h_kv, d)[:n]
        tof64 = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
        ro, rl, _ = oracle.fwd(tof64(q[b:b + 1]), tof64(kb)[None], tof64(vb)[None], scale=d ** -0.5, causal=True)
        check(f"O[{b}]", from_dev(o[b:b + 1]), ro)
        check_lse(f"LSE[{b}]", lse[b:b + 1].cpu().numpy().astype(np.float64), rl)


def _packed_oracle(w, used_q, used_k, bwd):
    """Oracle of a dense batch restricted to its first used_q[b] queries and used_k[b] keys:
    the packed batch of those rows (P2 "Varlen semantics"); returns per-batch lists."""
    B = w["B"]
    cat = lambda x, n: np.concatenate([x[b, :n[b]] for b in range(B)])  # noqa: E731
    q, k, v, do = (inputs.bf16_to_f64(w[t]) for t in ("q", "k", "v", "dout"))
    cu_q, cu_k = inputs.cu_seqlens(used_q), inputs.cu_seqlens(used_k)
    kw = dict(scale=w["scale"], causal=w["causal"], window=w["window"], cu_q=cu_q, cu_k=cu_k,
              sinks=None if w["sinks"] is None else w["sinks"].astype(np.float64))
    args = (cat(q, used_q), cat(k, used_k), cat(v, used_k))
    o, lse, _ = oracle.fwd(*args, **kw)
    out = dict(o=o, lse=lse, cu_q=cu_q, cu_k=cu_k)
    if bwd:
        out["dq"], out["dk"], out["dv"], out["ds"] = oracle.bwd(*args, cat(do, used_q), **kw)
    return out


@pytest.mark.parametrize("d,causal,window,sinks", [(64, True, (-1, -1), False), (128, True, (-1, -1), True),
                                                   (128, False, (90, 40), True), (64, False, (-1, -1), False)])
def test_seqused_q_and_k_forward_backward(d, causal, window, sinks):
    """Partly filled query and key slots, forward and backward: used rows of O, LSE, dQ and
    used keys of dK, dV against the oracle on the packed batch of the used rows."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    B, s_q, s_kv = 4, 300, 450
    w = inputs.make(dict(wid=WID, variant=40 + d + int(causal) + 2 * int(sinks), B=B, s_q=s_q, s_kv=s_kv, h_q=8,
                         h_kv=2, d=d, causal=causal, window=window, sinks=sinks, varlen=False))
    used_q = inputs.used_lengths(inputs.seed_of(WID, 60 + d, USED), B, s_q)
    used_k = inputs.used_lengths(inputs.seed_of(WID, 61 + d, USED), B, s_kv)
    used_q[2], used_k[2] = 0, 17   # an empty query slot, and
    used_q[3], used_k[3] = 250, 0  # queries against an empty key slot
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    tq, tk, tv, tdo = (to_dev(w[t]) for t in ("q", "k", "v", "dout"))
    sk = None if w["sinks"] is None else dev(w["sinks"])
    kw = dict(causal=causal, window=window, softmax_scale=w["scale"], sinks=sk, seqused_q=dev(used_q),
              seqused_k=dev(used_k))
    o, lse, ws = fa.forward(tq, tk, tv, **kw)
    dq, dk, dv, ds, ws2 = fa.backward(tq, tk, tv, o, lse, tdo, **kw)
    torch.cuda.synchronize()
    assert fa.device_status(ws) == fa.FA_OK and fa.device_status(ws2) == fa.FA_OK
    ref = _packed_oracle(w, used_q, used_k, bwd=True)
    o, lse, dq, dk, dv = from_dev(o), lse.cpu().numpy().astype(np.float64), from_dev(dq), from_dev(dk), from_dev(dv)
    for b in range(B):
        q0, q1 = ref["cu_q"][b], ref["cu_q"][b + 1]
        k0, k1 = ref["cu_k"][b], ref["cu_k"][b + 1]
        check(f"O[{b}]", o[b, :used_q[b]], ref["o"][q0:q1])
        check_lse(f"LSE[{b}]", lse[b, :, :used_q[b]], ref["lse"][:, q0:q1])
        check(f"dQ[{b}]", dq[b, :used_q[b]], ref["dq"][q0:q1])
        check(f"dK[{b}]", dk[b, :used_k[b]], ref["dk"][k0:k1])
        check(f"dV[{b}]", dv[b, :used_k[b]], ref["dv"][k0:k1])
    if sinks:
        err = float(np.abs(ds.cpu().numpy() - ref["ds"]).max())
        assert err <= 2e-2 * max(1.0, float(np.abs(ref["ds"]).max()))


def test_seqused_q_decode():
    """Few query rows per key/value head (the CUDA-core decode kernel) with partly filled
    query slots: the bottom-right alignment follows the used query count."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    B, s_q, s_kv = 4, 2, 2000
    w = inputs.make(dict(wid=WID, variant=77, B=B, s_q=s_q, s_kv=s_kv, h_q=8, h_kv=2, d=128, causal=True,
                         window=(-1, -1), sinks=False, varlen=False))
    used_q = np.array([2, 1, 0, 2], np.int32)
    used_k = np.array([2000, 1500, 900, 0], np.int32)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    o, lse, ws = fa.forward(to_dev(w["q"]), to_dev(w["k"]), to_dev(w["v"]), causal=True, softmax_scale=w["scale"],
                            seqused_q=dev(used_q), seqused_k=dev(used_k))
    torch.cuda.synchronize()
    assert fa.device_status(ws) == fa.FA_OK
    ref = _packed_oracle(w, used_q, used_k, bwd=False)
    o, lse = from_dev(o), lse.cpu().numpy().astype(np.float64)
    for b in range(B):
        q0, q1 = ref["cu_q"][b], ref["cu_q"][b + 1]
        check(f"O[{b}]", o[b, :used_q[b]], ref["o"][q0:q1])
        check_lse(f"LSE[{b}]", lse[b, :, :used_q[b]], ref["lse"][:, q0:q1])


@pytest.mark.parametrize("d,causal,window,sinks", [(64, True, (-1, -1), True), (128, False, (40, 10), False)])
def test_seqused_packed_token_tiles(d, causal, window, sinks):
    """A packed batch whose queries and keys share one offsets array (token tiles) with
    partly used slots: each slot uses its first seqused_q[b] queries and seqused_k[b] keys,
    forward and backward, against the oracle on the packed batch of the used rows."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    slots = [40, 3, 0, 200, 17, 90, 1, 130]
    rng = np.random.default_rng(inputs.seed_of(WID, 70 + d, USED))
    used_q = np.array([rng.integers(0, n + 1) for n in slots], np.int32)
    used_k = np.array([rng.integers(0, n + 1) for n in slots], np.int32)
    used_q[3], used_k[3] = 200, 120
    w = inputs.make(dict(wid=WID, variant=80 + d, B=len(slots), s_q=0, s_kv=0, h_q=4, h_kv=2, d=d, causal=causal,
                         window=window, sinks=sinks, varlen=True, lengths=slots))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    cu = dev(w["cu_q"])
    tq, tk, tv, tdo = (to_dev(w[t]) for t in ("q", "k", "v", "dout"))
    kw = dict(causal=causal, window=window, softmax_scale=w["scale"], sinks=None if w["sinks"] is None else dev(w["sinks"]),
              cu_q=cu, cu_k=cu, seqused_q=dev(used_q), seqused_k=dev(used_k))
    o, lse, ws = fa.forward(tq, tk, tv, **kw)
    dq, dk, dv, ds, ws2 = fa.backward(tq, tk, tv, o, lse, tdo, **kw)
    torch.cuda.synchronize()
    assert fa.device_status(ws) == fa.FA_OK and fa.device_status(ws2) == fa.FA_OK
    # the oracle's problem: the used rows of every slot, packed
    cu_h = w["cu_q"]
    cat = lambda x, n: np.concatenate([x[cu_h[b]:cu_h[b] + n[b]] for b in range(len(slots))])  # noqa: E731
    q, k, v, do = (inputs.bf16_to_f64(w[t]) for t in ("q", "k", "v", "dout"))
    rcq, rck = inputs.cu_seqlens(used_q), inputs.cu_seqlens(used_k)
    okw = dict(scale=w["scale"], causal=causal, window=window, cu_q=rcq, cu_k=rck,
               sinks=None if w["sinks"] is None else w["sinks"].astype(np.float64))
    args = (cat(q, used_q), cat(k, used_k), cat(v, used_k))
    ro, rl, _ = oracle.fwd(*args, **okw)
    rdq, rdk, rdv, rds = oracle.bwd(*args, cat(do, used_q), **okw)
    o, lse, dq, dk, dv = from_dev(o), lse.cpu().numpy().astype(np.float64), from_dev(dq), from_dev(dk), from_dev(dv)
    check("O", cat(o, used_q), ro)
    check_lse("LSE", np.concatenate([lse[:, cu_h[b]:cu_h[b] + used_q[b]] for b in range(len(slots))], axis=1), rl)
    check("dQ", cat(dq, used_q), rdq)
    check("dK", cat(dk, used_k), rdk)
    check("dV", cat(dv, used_k), rdv)
    if sinks:
        err = float(np.abs(ds.cpu().numpy() - rds).max())
        assert err <= 2e-2 * max(1.0, float(np.abs(rds).max()))
