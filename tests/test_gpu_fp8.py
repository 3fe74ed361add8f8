"""GPU parity of the e4m3 (fp8) forward against the fp64 oracle.

The oracle receives the true inputs (the e4m3 values times their per-(batch, key/value
head) descale factors, exact in fp64).  O is judged by the pages' test rule
(vllm-project/flash-attention README, "Tests"): its maximum and mean errors against fp64
are at most twice those of a CPU run that rounds P to e4m3 the same way
(tests/fp8_emulation.py), plus a small floor; in absolute terms that stays far below
what one e4m3 rounding of P (relative 2^-4) could cause.  The LSE is exact up to fp32
summation and is held to the bf16 path's 1e-3.  The shapes reach the unsplit and the
split-key kernel (decode and chunked-prefill shapes), masks, sinks, grouped heads,
s_q != s_kv, partly filled caches, and the benchmark's size (sampled rows).
"""
import numpy as np
import pytest

import fp8_emulation
import oracle
from exact_attention_bwd_gb300 import inputs
from gpu_helpers import check_lse, from_dev

pytestmark = pytest.mark.gpu

WID = 140


def case(variant, *, B=2, s_q=300, s_kv=None, h_q=8, h_kv=2, causal=False, window=(-1, -1), sinks=False,
         used=False, unit_descale=False):
    s_kv = s_q if s_kv is None else s_kv
    sd = lambda t: inputs.seed_of(WID, variant, t)  # noqa: E731
    spread = 1.0 if unit_descale else 32.0
    c = dict(B=B, s_q=s_q, s_kv=s_kv, h_q=h_q, h_kv=h_kv, d=128, causal=causal, window=window,
             scale=1.0 / np.sqrt(128.0))
    c["q"] = inputs.normal_e4m3(sd(inputs.Q), (B, s_q, h_q, 128), spread)
    c["k"] = inputs.normal_e4m3(sd(inputs.K), (B, s_kv, h_kv, 128), spread)
    c["v"] = inputs.normal_e4m3(sd(inputs.V), (B, s_kv, h_kv, 128), spread)
    if unit_descale:
        c["descale"] = None
    else:
        c["descale"] = tuple(inputs.descales(sd(10 + t), B, h_kv) for t in range(3))
    c["sinks"] = inputs.normal_f32(sd(inputs.SINKS), (h_q,)) if sinks else None
    c["used"] = inputs.used_lengths(sd(6), B, s_kv) if used else None
    return c


def true_inputs(c):
    """fp64 true values: stored e4m3 value x its (batch, kv head) descale."""
    B, G = c["B"], c["h_q"] // c["h_kv"]
    out = []
    for t, key in enumerate(("q", "k", "v")):
        x = inputs.e4m3_to_f64(c[key])
        if c["descale"] is not None:
            ds = c["descale"][t].astype(np.float64).reshape(B, c["h_kv"])
            if key == "q":
                ds = np.repeat(ds, G, axis=1)
            x = x * ds[:, None, :, None]
        out.append(x)
    return out


def run_gpu(c):
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    q, k, v = dev(c["q"]), dev(c["k"]), dev(c["v"])
    descale = None if c["descale"] is None else tuple(dev(x) for x in c["descale"])
    sinks = None if c["sinks"] is None else dev(c["sinks"])
    used = None if c["used"] is None else dev(c["used"])
    o, lse, ws = fa.forward(q, k, v, causal=c["causal"], window=c["window"], softmax_scale=c["scale"], sinks=sinks,
                            seqused_k=used, descale=descale)
    torch.cuda.synchronize()
    assert fa.device_status(ws) == fa.FA_OK
    return from_dev(o), lse.cpu().numpy().astype(np.float64)


def reference(c):
    q, k, v = true_inputs(c)
    B, s_q, h_q = c["B"], c["s_q"], c["h_q"]
    sinks = None if c["sinks"] is None else c["sinks"].astype(np.float64)
    if c["used"] is None:
        ro, rl, _ = oracle.fwd(q, k, v, scale=c["scale"], causal=c["causal"], window=c["window"], sinks=sinks)
    else:  # partly filled slots: a packed batch of the used keys (see test_gpu_kvcache)
        used = c["used"]
        ks = np.concatenate([k[b, :used[b]] for b in range(B)])
        vs = np.concatenate([v[b, :used[b]] for b in range(B)])
        cu_q = (np.arange(B + 1) * s_q).astype(np.int32)
        ro, rl, _ = oracle.fwd(q.reshape(B * s_q, h_q, 128), ks, vs, scale=c["scale"], causal=c["causal"],
                               window=c["window"], sinks=sinks, cu_q=cu_q, cu_k=inputs.cu_seqlens(used))
        ro = ro.reshape(B, s_q, h_q, 128)
        rl = rl.reshape(h_q, B, s_q).transpose(1, 0, 2)
    f32 = lambda x: x.astype(np.float32)  # noqa: E731
    emu = fp8_emulation.fwd(f32(q), f32(k), f32(v), scale=c["scale"], causal=c["causal"], window=c["window"],
                            sinks=None if sinks is None else f32(sinks), kv_len=c["used"])
    return ro, rl, emu


def judge(o, ro, emu):
    assert np.all(np.isfinite(o))
    e_gpu, e_emu = np.abs(o - ro), np.abs(emu - ro)
    at = np.unravel_index(int(np.argmax(e_gpu)), e_gpu.shape)
    assert e_gpu.max() <= 2.0 * e_emu.max() + 2e-3, (
        f"max error {e_gpu.max():.3e} at {at} (emulation there {e_emu[at]:.3e}) > 2 x emulation {e_emu.max():.3e}; "
        f"elements above: {int((e_gpu > 2.0 * e_emu.max() + 2e-3).sum())}")
    assert e_gpu.mean() <= 2.0 * e_emu.mean() + 2e-4, f"mean error {e_gpu.mean():.3e} > 2 x {e_emu.mean():.3e}"


CASES = [
    dict(),
    dict(causal=True),
    dict(causal=False, window=(100, 30), sinks=True),
    dict(causal=True, window=(127, 0), h_q=16, h_kv=2, sinks=True),
    dict(s_q=200, s_kv=333, causal=True),
    dict(s_q=333, s_kv=200, causal=True),
    dict(h_q=6, h_kv=2, causal=True),
    dict(unit_descale=True, causal=True),
    dict(B=2, s_q=1, s_kv=3000, causal=True),       # decode shape: split keys
    dict(B=1, s_q=64, s_kv=2100, causal=True),      # chunked prefill: split keys
    dict(B=3, s_q=64, s_kv=1000, causal=True, used=True),
    dict(B=2, s_q=1, s_kv=3000, causal=True, sinks=True, h_q=16, h_kv=2),  # split keys, sinks in the combine
    dict(B=1, s_q=64, s_kv=2100, causal=False, window=(500, 0), sinks=True),
]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_fp8_forward(i):
    c = case(i, **CASES[i])
    o, lse = run_gpu(c)
    ro, rl, emu = reference(c)
    judge(o, ro, emu)
    check_lse("LSE", lse, rl)


def test_fp8_full_size_sampled():
    """The benchmark's shape (B=2, s=8192, h=16, d=128, causal) in e4m3: the last 64 query
    rows of each batch entry and every head against the oracle run on just those rows
    (bottom-right alignment keeps them exact), by the same rule."""
    c = case(50, B=2, s_q=8192, h_q=16, h_kv=16, causal=True)
    o, lse = run_gpu(c)
    q, k, v = true_inputs(c)
    rows = 64
    for b in range(2):
        sub = dict(c, B=1, s_q=rows, q=c["q"][b:b + 1, -rows:], k=c["k"][b:b + 1], v=c["v"][b:b + 1],
                   descale=None if c["descale"] is None else tuple(x.reshape(2, 16)[b:b + 1].ravel()
                                                                    for x in c["descale"]))
        ro, rl, emu = reference(sub)
        judge(o[b:b + 1, -rows:], ro, emu)
        check_lse("LSE", lse[b:b + 1, :, -rows:], rl)


def test_fp8_cache_shape_sampled():
    """The chunked-prefill cache shape in e4m3 (s_q=64 against s_kv=32768, h_q=32, h_kv=8,
    causal; split keys with the LSE combine), batch entries 0 and 7 of 8 against the oracle."""
    c = case(51, B=8, s_q=64, s_kv=32768, h_q=32, h_kv=8, causal=True)
    o, lse = run_gpu(c)
    for b in (0, 7):
        sub = dict(c, B=1, q=c["q"][b:b + 1], k=c["k"][b:b + 1], v=c["v"][b:b + 1],
                   descale=tuple(x.reshape(8, 8)[b:b + 1].ravel() for x in c["descale"]))
        ro, rl, emu = reference(sub)
        judge(o[b:b + 1], ro, emu)
        check_lse("LSE", lse[b:b + 1], rl)


PACKED = [
    dict(lq=[300, 0, 129, 1, 1000, 64], causal=True, sinks=True),
    dict(lq=[100, 250, 17], lk=[300, 250, 40], causal=True, window=(64, 0)),
    dict(lq=[2000, 3, 700], causal=False, window=(100, 30), h_q=16, h_kv=2),
]


@pytest.mark.parametrize("i", range(len(PACKED)))
def test_fp8_packed_batch(i):
    """Packed batches (cu_seqlens; empty and one-token sequences, s_q != s_kv per sequence):
    each sequence against the oracle and the emulation run on it alone, judged together."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    kw = dict(PACKED[i])
    lq = np.asarray(kw.pop("lq"))
    lk = np.asarray(kw.pop("lk", lq))
    B = len(lq)
    c = case(60 + i, B=B, s_q=int(lq.max()), s_kv=int(lk.max()), **kw)
    cu_q, cu_k = inputs.cu_seqlens(lq), inputs.cu_seqlens(lk)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    pack = lambda x, n: np.concatenate([x[b, :n[b]] for b in range(B)])  # noqa: E731
    q, k, v = dev(pack(c["q"], lq)), dev(pack(c["k"], lk)), dev(pack(c["v"], lk))
    tcq = dev(cu_q)
    tck = tcq if np.array_equal(cu_q, cu_k) else dev(cu_k)
    o, lse, ws = fa.forward(q, k, v, causal=c["causal"], window=c["window"], softmax_scale=c["scale"],
                            sinks=None if c["sinks"] is None else dev(c["sinks"]), cu_q=tcq, cu_k=tck,
                            descale=tuple(dev(x) for x in c["descale"]))
    torch.cuda.synchronize()
    assert fa.device_status(ws) == fa.FA_OK
    o, lse = from_dev(o), lse.cpu().numpy().astype(np.float64)
    got, ref, emu = [], [], []
    for b in range(B):
        if lq[b] == 0:
            continue
        sub = dict(c, B=1, s_q=int(lq[b]), s_kv=int(lk[b]), q=c["q"][b:b + 1, :lq[b]], k=c["k"][b:b + 1, :lk[b]],
                   v=c["v"][b:b + 1, :lk[b]], descale=tuple(x.reshape(B, -1)[b:b + 1].ravel() for x in c["descale"]))
        ro, rl, em = reference(sub)
        got.append(o[cu_q[b]:cu_q[b + 1]])
        ref.append(ro[0])
        emu.append(em[0])
        check_lse(f"LSE sequence {b}", lse[None, :, cu_q[b]:cu_q[b + 1]], rl)
    judge(np.concatenate(got), np.concatenate(ref), np.concatenate(emu))


@pytest.mark.parametrize("s_q,used", [(1, False), (64, True)])
def test_fp8_paged_cache(s_q, used):
    """A paged e4m3 cache (256-key pages in a seeded order, spare pages in the pool, a
    logical length that is not a multiple of the page size): the same bits as the dense
    cache (same kernel, same tile order), and the oracle by the same rule."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    B, s_kv, ps = 3, 1000, 256
    c = case(70 + s_q, B=B, s_q=s_q, s_kv=s_kv, h_q=8, h_kv=2, causal=True, used=used)
    mb = -(-s_kv // ps)
    n_pages = B * mb + 3
    table = inputs.page_table(inputs.seed_of(WID, 70 + s_q, 20), B, mb, n_pages)

    def pool_of(x):
        pool = np.zeros((n_pages, ps, c["h_kv"], 128), np.uint8)
        for b in range(B):
            for blk in range(mb):
                seg = x[b, blk * ps:(blk + 1) * ps]
                pool[table[b, blk], :seg.shape[0]] = seg
        return pool
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    kw = dict(causal=True, window=c["window"], softmax_scale=c["scale"], descale=tuple(dev(x) for x in c["descale"]),
              seqused_k=None if c["used"] is None else dev(c["used"]))
    q = dev(c["q"])
    o_p, lse_p, ws = fa.forward(q, dev(pool_of(c["k"])), dev(pool_of(c["v"])), block_table=dev(table), s_kv=s_kv,
                                **kw)
    o_d, lse_d, ws2 = fa.forward(q, dev(c["k"]), dev(c["v"]), **kw)
    torch.cuda.synchronize()
    assert fa.device_status(ws) == fa.FA_OK and fa.device_status(ws2) == fa.FA_OK
    assert torch.equal(o_p.view(torch.int16), o_d.view(torch.int16))
    assert torch.equal(lse_p.view(torch.int32), lse_d.view(torch.int32))
    ro, rl, emu = reference(c)
    judge(from_dev(o_p), ro, emu)
    check_lse("LSE", lse_p.cpu().numpy().astype(np.float64), rl)


def test_fp8_seqused_q_and_k():
    """Partly filled query and key slots (seqused_q, seqused_k; a slot with no queries): the
    used rows of each batch entry against the oracle and the emulation on the used part
    alone (bottom-right alignment follows the used counts)."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    B = 3
    c = case(80, B=B, s_q=64, s_kv=1000, h_q=8, h_kv=2, causal=True)
    used_q = np.array([64, 10, 0], np.int32)
    used_k = np.array([1000, 500, 300], np.int32)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    o, lse, ws = fa.forward(dev(c["q"]), dev(c["k"]), dev(c["v"]), causal=True, softmax_scale=c["scale"],
                            descale=tuple(dev(x) for x in c["descale"]), seqused_q=dev(used_q), seqused_k=dev(used_k))
    torch.cuda.synchronize()
    assert fa.device_status(ws) == fa.FA_OK
    o, lse = from_dev(o), lse.cpu().numpy().astype(np.float64)
    got, ref, emu = [], [], []
    for b in range(B):
        if used_q[b] == 0:
            continue
        sub = dict(c, B=1, s_q=int(used_q[b]), s_kv=int(used_k[b]), q=c["q"][b:b + 1, :used_q[b]],
                   k=c["k"][b:b + 1, :used_k[b]], v=c["v"][b:b + 1, :used_k[b]],
                   descale=tuple(x.reshape(B, -1)[b:b + 1].ravel() for x in c["descale"]))
        ro, rl, em = reference(sub)
        got.append(o[b, :used_q[b]])
        ref.append(ro[0])
        emu.append(em[0])
        check_lse(f"LSE[{b}]", lse[b:b + 1, :, :used_q[b]], rl)
    judge(np.concatenate(got), np.concatenate(ref), np.concatenate(emu))


def test_fp8_tail_split():
    """B=40 (batch, kv head) units of s_q=64 rows against s_kv=2048 keys: 320 items over the
    GB300's 152 SMs leave a last round of 16, whose units the planner cuts into key ranges
    merged by the combine (the tail split).  Units on both sides of the boundary, and the
    first and last, against the oracle by the same rule."""
    c = case(90, B=40, s_q=64, s_kv=2048, h_q=32, h_kv=8, causal=True, sinks=True)
    o, lse = run_gpu(c)
    got, ref, emu = [], [], []
    for unit in (0, 303, 304, 319):
        b, g = divmod(unit, 8)
        hs = slice(4 * g, 4 * g + 4)
        sub = dict(c, B=1, h_q=4, h_kv=1, q=c["q"][b:b + 1, :, hs], k=c["k"][b:b + 1, :, g:g + 1],
                   v=c["v"][b:b + 1, :, g:g + 1], sinks=c["sinks"][hs],
                   descale=tuple(x.reshape(40, 8)[b:b + 1, g:g + 1].ravel() for x in c["descale"]))
        ro, rl, em = reference(sub)
        got.append(o[b:b + 1, :, hs])
        ref.append(ro)
        emu.append(em)
        check_lse(f"LSE unit {unit}", lse[b:b + 1, hs], rl)
    judge(np.concatenate(got), np.concatenate(ref), np.concatenate(emu))
