"""GPU parity at the workloads' full sizes, in the launch configuration the benchmark uses.

The whole problem runs on the GPU; the fp64 oracle recomputes seeded samples that it can
compute exactly on its own:
  * a block of query rows [i0, i1) of a causal problem equals the problem with those
    rows against keys [0, i1) (bottom-right alignment puts the offset back), and of a
    non-causal one against all keys, so O, LSE and dQ of sampled rows are exact;
  * dK and dV of a key are sums over the rows that see it: the last key block of a causal
    problem is seen only by the last query rows, and a whole head is the sum of row-chunk
    problems (run in parallel worker processes);
  * packed batches and decode caches are independent per sequence / per (batch, head).
"""
import multiprocessing as mp
import os

import numpy as np
import pytest

import oracle
from exact_attention_bwd_gb300 import inputs
from gpu_helpers import check, check_lse, dev_inputs, from_dev

pytestmark = pytest.mark.gpu

_POOL = None


def pool():
    """A spawn-started pool of single-threaded oracle workers (created before any fork)."""
    global _POOL
    if _POOL is None:
        ctx = mp.get_context("spawn")
        n = max(1, min(16, os.cpu_count() or 1))
        _POOL = ctx.Pool(n, initializer=_worker_init)
    return _POOL


def _worker_init():
    os.environ["OMP_NUM_THREADS"] = "1"


def _chunk_bwd(args):
    q, k, v, do, kw = args
    import oracle as o
    return o.bwd(q, k, v, do, **kw)


def oracle_head_bwd(q, k, v, do, causal, scale, chunk=512):
    """Exact dQ, dK, dV of one dense head ([1, s, 1, d] arrays) as a sum of row chunks."""
    s_q, s_kv = q.shape[1], k.shape[1]
    jobs = []
    for i0 in range(0, s_q, chunk):
        i1 = min(s_q, i0 + chunk)
        kend = (i1 + s_kv - s_q) if causal else s_kv
        jobs.append((q[:, i0:i1], k[:, :kend], v[:, :kend], do[:, i0:i1],
                     dict(scale=scale, causal=causal)))
    res = pool().map(_chunk_bwd, jobs)
    dq = np.concatenate([r[0] for r in res], axis=1)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for (qq, kk, vv, dd, _), r in zip(jobs, res):
        dk[:, :kk.shape[1]] += r[1]
        dv[:, :kk.shape[1]] += r[2]
    return dq, dk, dv


def run_full(w, bwd=True):
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    d = dev_inputs(w)
    kw = dict(causal=w["causal"], window=w["window"], softmax_scale=w["scale"], sinks=d["sinks"],
              cu_q=d["cu_q"], cu_k=d["cu_k"])
    o, lse, ws = fa.forward(d["q"], d["k"], d["v"], **kw)
    res = dict(o=o, lse=lse)
    if bwd:
        dq, dk, dv, ds, ws2 = fa.backward(d["q"], d["k"], d["v"], o, lse, d["dout"], **kw)
        res.update(dq=dq, dk=dk, dv=dv, dsinks=ds)
        torch.cuda.synchronize()
        assert fa.device_status(ws2) == 0
    torch.cuda.synchronize()
    assert fa.device_status(ws) == 0
    return res


SWEEP = [(s, c) for s in (512, 1024, 2048, 4096, 8192, 16384) for c in (True, False)]


@pytest.mark.parametrize("s,causal", SWEEP, ids=[f"s{s}-{'causal' if c else 'full'}" for s, c in SWEEP])
def test_dense_sweep(s, causal):
    w = inputs.make(inputs.workload(f"sweep_s{s}{'_causal' if causal else ''}"))
    got = run_full(w)
    f = inputs.bf16_to_f64
    scale = w["scale"]
    B = w["B"]
    for b, h in [(0, 0), (B - 1, 15)]:
        q, k, v, do = (f(w[x][b:b + 1, :, h:h + 1]) for x in ("q", "k", "v", "dout"))
        # sampled query-row blocks: O, LSE, dQ
        for i0 in (0, (s // 2) - 64, s - 128):
            i1 = i0 + 128
            kend = i1 if causal else s
            ro, rl, _ = oracle.fwd(q[:, i0:i1], k[:, :kend], v[:, :kend], scale=scale, causal=causal)
            rdq, _, _, _ = oracle.bwd(q[:, i0:i1], k[:, :kend], v[:, :kend], do[:, i0:i1], scale=scale, causal=causal)
            check(f"O b{b} h{h} rows {i0}", from_dev(got["o"][b:b + 1, i0:i1, h:h + 1]), ro)
            check_lse(f"LSE b{b} h{h} rows {i0}", got["lse"][b, h, i0:i1].cpu().numpy(), rl[0, 0])
            check(f"dQ b{b} h{h} rows {i0}", from_dev(got["dq"][b:b + 1, i0:i1, h:h + 1]), rdq)
        if causal:
            # the last key block is seen only by the last query rows
            j0 = s - 128
            _, rdk, rdv, _ = oracle.bwd(q[:, j0:], k, v, do[:, j0:], scale=scale, causal=True)
            check(f"dK b{b} h{h} last block", from_dev(got["dk"][b:b + 1, j0:, h:h + 1]), rdk[:, j0:])
            check(f"dV b{b} h{h} last block", from_dev(got["dv"][b:b + 1, j0:, h:h + 1]), rdv[:, j0:])
    # one whole head exactly (all of dK, dV)
    if s <= 8192 or causal:
        b, h = 0, 3
        q, k, v, do = (f(w[x][b:b + 1, :, h:h + 1]) for x in ("q", "k", "v", "dout"))
        rdq, rdk, rdv = oracle_head_bwd(q, k, v, do, causal, scale)
        check(f"dK head b{b} h{h}", from_dev(got["dk"][b:b + 1, :, h:h + 1]), rdk)
        check(f"dV head b{b} h{h}", from_dev(got["dv"][b:b + 1, :, h:h + 1]), rdv)
        check(f"dQ head b{b} h{h}", from_dev(got["dq"][b:b + 1, :, h:h + 1]), rdq)


@pytest.mark.parametrize("name", ["gqa_window_causal", "gqa_window_2sided"])
def test_gqa_window_sinks_full(name):
    """B=2, s=4096, h_q=64, h_kv=8, d=64, sinks: every output against the full oracle."""
    w = inputs.make(inputs.workload(name))
    got = run_full(w)
    f = inputs.bf16_to_f64
    kw = dict(scale=w["scale"], causal=w["causal"], window=w["window"], sinks=w["sinks"].astype(np.float64))
    q, k, v, do = (f(w[x]) for x in ("q", "k", "v", "dout"))
    ro, rl, _ = oracle.fwd(q, k, v, **kw)
    check("O", from_dev(got["o"]), ro)
    check_lse("LSE", got["lse"].cpu().numpy(), rl)
    rdq, rdk, rdv, rds = oracle.bwd(q, k, v, do, **kw)
    check("dQ", from_dev(got["dq"]), rdq)
    check("dK", from_dev(got["dk"]), rdk)
    check("dV", from_dev(got["dv"]), rdv)
    ds = got["dsinks"].cpu().numpy().astype(np.float64)
    assert np.abs(ds - rds).max() <= 2e-2 * max(1.0, np.abs(rds).max()), (ds[:4], rds[:4])


def test_varlen_full():
    """T=32768 packed causal, h=32, d=128: sampled sequences against the oracle."""
    w = inputs.make(inputs.workload("varlen"))
    got = run_full(w)
    cu = w["cu_q"]
    lengths = np.diff(cu)
    order = np.argsort(lengths)
    pick = sorted(set([int(order[-1]), int(order[-2]), int(np.nonzero(lengths == 1)[0][0]) if (lengths == 1).any()
                       else int(order[0]), int(np.nonzero(lengths == 0)[0][0])] +
                      list(np.random.default_rng(0).choice(len(lengths), 4, replace=False))))
    f = inputs.bf16_to_f64
    rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in pick])
    sub_cu = inputs.cu_seqlens(lengths[pick])
    q, k, v, do = (f(w[x][rows]) for x in ("q", "k", "v", "dout"))
    kw = dict(scale=w["scale"], causal=True, cu_q=sub_cu, cu_k=sub_cu)
    ro, rl, _ = oracle.fwd(q, k, v, **kw)
    rdq, rdk, rdv, _ = oracle.bwd(q, k, v, do, **kw)
    idx = torch_index(rows)
    check("O", from_dev(got["o"][idx]), ro)
    check_lse("LSE", got["lse"][:, idx].cpu().numpy(), rl)
    check("dQ", from_dev(got["dq"][idx]), rdq)
    check("dK", from_dev(got["dk"][idx]), rdk)
    check("dV", from_dev(got["dv"][idx]), rdv)


def torch_index(rows):
    import torch
    return torch.from_numpy(rows.astype(np.int64)).cuda()


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("s_q", [1, 64])
def test_decode_full(d, s_q):
    """B=64, h_q=32, h_kv=8, s_kv=32768 causal cache: sampled (batch, kv-head) units."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    w = inputs.workload(f"decode_d{d}_sq{s_q}")
    B, h_q, h_kv, s_kv = w["B"], w["h_q"], w["h_kv"], w["s_kv"]
    G = h_q // h_kv
    seed = lambda t: inputs.seed_of(w["wid"], w["variant"], t)  # noqa: E731
    q = inputs.normal_bf16_torch(seed(inputs.Q), (B, s_q, h_q, d), "cuda")
    k = inputs.normal_bf16_torch(seed(inputs.K), (B, s_kv, h_kv, d), "cuda")
    v = inputs.normal_bf16_torch(seed(inputs.V), (B, s_kv, h_kv, d), "cuda")
    scale = 1.0 / np.sqrt(d)
    o, lse, ws = fa.forward(q, k, v, causal=True, softmax_scale=scale)
    torch.cuda.synchronize()
    assert fa.device_status(ws) == 0
    for b, g in [(0, 0), (B - 1, h_kv - 1), (17, 3)]:
        hs = slice(g * G, (g + 1) * G)
        qq = from_dev(q[b:b + 1, :, hs])
        kk = from_dev(k[b:b + 1, :, g:g + 1])
        vv = from_dev(v[b:b + 1, :, g:g + 1])
        ro, rl, _ = oracle.fwd(qq, kk, vv, scale=scale, causal=True)
        check(f"O b{b} g{g}", from_dev(o[b:b + 1, :, hs]), ro)
        check_lse(f"LSE b{b} g{g}", lse[b, hs].cpu().numpy(), rl[0])
    del k, v
    torch.cuda.empty_cache()


@pytest.mark.parametrize("d,sinks", [(256, False), (256, True), (192, False), (128, True), (64, False)])
def test_tail_split(d, sinks):
    """B=40, h_q=32, h_kv=8, s_q=64, s_kv=4096 causal cache: at d = 192 / 256, 640 one-CTA
    items over the GB300's 152 SMs leave a last wave of 32; at d = 64 / 128 (the persistent
    kernel, one item per unit), 320 items leave a last round of 16.  The planner then cuts
    the last 16 (batch, kv head) units' items into key ranges merged by the combine (the
    tail split).  Whole units on both sides of that boundary, and the first and last,
    against the oracle."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    B, s_q, s_kv, h_q, h_kv = 40, 64, 4096, 32, 8
    G = h_q // h_kv
    w = inputs.make(dict(wid=32, variant=d + int(sinks), B=B, s_q=s_q, s_kv=s_kv, h_q=h_q, h_kv=h_kv, d=d,
                         causal=True, window=(-1, -1), sinks=sinks, varlen=False))
    dv = dev_inputs(w)
    o, lse, ws = fa.forward(dv["q"], dv["k"], dv["v"], causal=True, softmax_scale=w["scale"], sinks=dv["sinks"])
    torch.cuda.synchronize()
    assert fa.device_status(ws) == 0
    for unit in (0, 303, 304, 319):
        b, g = divmod(unit, h_kv)
        hs = slice(g * G, (g + 1) * G)
        qq = inputs.bf16_to_f64(w["q"][b:b + 1, :, hs])
        kk = inputs.bf16_to_f64(w["k"][b:b + 1, :, g:g + 1])
        vv = inputs.bf16_to_f64(w["v"][b:b + 1, :, g:g + 1])
        sk = None if w["sinks"] is None else w["sinks"][hs].astype(np.float64)
        ro, rl, _ = oracle.fwd(qq, kk, vv, scale=w["scale"], causal=True, sinks=sk)
        check(f"O unit {unit}", from_dev(o[b:b + 1, :, hs]), ro)
        check_lse(f"LSE unit {unit}", lse[b, hs].cpu().numpy(), rl[0])


@pytest.mark.parametrize("packed", [False, True], ids=["dense", "packed"])
def test_offsets_beyond_int32_elements(packed):
    """Q, O, dO and dQ of more than 2^31 elements (s=140000 tokens, h_q=128, h_kv=32, d=128:
    2.29e9 each, 4.6 GB in bf16; the fp32 dQ accumulator 9.2 GB), with a causal (127, 0)
    window so the whole call stays short (groups of 4 query heads: with 16, the dK and dV
    of the first keys, which sum 16 heads' rows of nearly one-hot P, exceed the absolute
    bound already in an exact bf16-operand emulation).  Every address the kernels form past
    element 2^31 must be 64-bit.  Dense: one batch of 140000 positions; packed: the same
    tokens as sequences of 60000, 0 and 80000 (one offsets array for queries and keys, so
    the token-tile path).  A query row sees its 128 nearest keys of its sequence and a key
    is seen by the 128 rows after it, so a block of rows together with the up to 127 keys
    before it is an exact sub-problem (bottom-right alignment keeps the diagonal) for O,
    LSE and dQ of its rows and for dK, dV of its own keys; blocks at the start, across
    element 2^31 and at the end are checked (packed: also at the third sequence's start)."""
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    s, h_q, h_kv, d = 140000, 128, 32, 128
    G = h_q // h_kv
    assert s * h_q * d > 2 ** 31
    window = (127, 0)
    seed = lambda t: inputs.seed_of(34, 0, t)  # noqa: E731
    q = inputs.normal_bf16_torch(seed(inputs.Q), (1, s, h_q, d), "cuda")
    k = inputs.normal_bf16_torch(seed(inputs.K), (1, s, h_kv, d), "cuda")
    v = inputs.normal_bf16_torch(seed(inputs.V), (1, s, h_kv, d), "cuda")
    do = inputs.normal_bf16_torch(seed(inputs.DO), (1, s, h_q, d), "cuda")
    scale = 1.0 / np.sqrt(d)
    kw = dict(causal=True, window=window, softmax_scale=scale)
    starts = [0]
    if packed:
        cu = torch.tensor([0, 60000, 60000, s], dtype=torch.int32, device="cuda")
        kw.update(cu_q=cu, cu_k=cu)
        starts = [0, 60000]
        q, k, v, do = (t[0] for t in (q, k, v, do))
    o, lse, ws = fa.forward(q, k, v, **kw)
    torch.cuda.synchronize()
    assert fa.device_status(ws) == 0
    del ws
    dq, dk, dv, _, ws2 = fa.backward(q, k, v, o, lse, do, **kw)
    torch.cuda.synchronize()
    assert fa.device_status(ws2) == 0
    del ws2
    torch.cuda.empty_cache()
    if packed:  # back to the dense [1, s, h, d] / [1, h, s] views for the checks
        q, k, v, do, o, dq, dk, dv = (t.unsqueeze(0) for t in (q, k, v, do, o, dq, dk, dv))
        lse = lse.unsqueeze(0)
    edge = 2 ** 31 // (h_q * d)  # the position whose first element is element 2^31
    blocks = [(0, 0), (edge - 100, 3), (s - 200, h_kv - 1)] + ([(60000, 17)] if packed else [])
    for i0, g in blocks:
        i1 = i0 + 200
        start = max(x for x in starts if x <= i0)
        j0 = max(start, i0 - 127)
        hs = slice(g * G, (g + 1) * G)
        qq, dd = (from_dev(t[:, i0:i1, hs]) for t in (q, do))
        kk, vv = (from_dev(t[:, j0:i1, g:g + 1]) for t in (k, v))
        okw = dict(scale=scale, causal=True, window=window)
        ro, rl, _ = oracle.fwd(qq, kk, vv, **okw)
        rdq, rdk, rdv, _ = oracle.bwd(qq, kk, vv, dd, **okw)
        check(f"O rows {i0}", from_dev(o[:, i0:i1, hs]), ro)
        check_lse(f"LSE rows {i0}", lse[0, hs, i0:i1].cpu().numpy(), rl[0])
        check(f"dQ rows {i0}", from_dev(dq[:, i0:i1, hs]), rdq)
        # keys of the block that no row after i1 sees
        kb = i0 - j0
        check(f"dK keys {i0}", from_dev(dk[:, i0:i1 - 127, g:g + 1]), rdk[:, kb:kb + 200 - 127])
        check(f"dV keys {i0}", from_dev(dv[:, i0:i1 - 127, g:g + 1]), rdv[:, kb:kb + 200 - 127])
        if i1 == s:  # the last block's keys are all seen only by the block's rows
            check("dK last keys", from_dev(dk[:, i0:, g:g + 1]), rdk[:, kb:])
            check("dV last keys", from_dev(dv[:, i0:, g:g + 1]), rdv[:, kb:])
    del q, k, v, do, o, lse, dq, dk, dv
    torch.cuda.empty_cache()
