"""GPU parity: the CUDA library against the fp64 oracle, element by element.

Sizes are small enough for the oracle to finish in seconds yet span several 128-row
tiles with a ragged tail, and cover the masks, grouped-query heads (including a group
size that does not divide 128), sinks, packed batches with empty sequences, s_q != s_kv
in both directions, and decode shapes.
"""
import numpy as np
import pytest

import oracle
from exact_attention_bwd_gb300 import inputs
from gpu_helpers import check, check_lse, f64, oracle_args, run_gpu

pytestmark = pytest.mark.gpu


def make_case(wid, variant, *, B=1, s_q=128, s_kv=None, h_q=2, h_kv=None, d=64, causal=False, window=(-1, -1),
              sinks=False, lengths=None, lengths_k=None):
    w = dict(wid=wid, variant=variant, B=B, s_q=s_q, s_kv=s_kv if s_kv is not None else s_q, h_q=h_q,
             h_kv=h_kv or h_q, d=d, causal=causal, window=window, sinks=sinks, varlen=lengths is not None)
    if lengths is not None:
        w["lengths"] = lengths
        if lengths_k is not None:
            w["lengths_k"] = lengths_k
        w["B"] = len(lengths)
    return inputs.make(w)


def compare(w, bwd=True, flags=0, fa_rule=(), share_cu=True):
    """Element-wise parity with the oracle.  Outputs named in `fa_rule` are judged by the
    pages' secondary rule instead: max error at most twice that of the bf16-operand
    emulation (tests/bf16_emulation.py) — for shapes where bf16 rounding of the GEMM
    operands alone exceeds the absolute bound."""
    got = run_gpu(w, bwd=bwd, flags=flags, share_cu=share_cu)
    q, k, v, do = f64(w, "q"), f64(w, "k"), f64(w, "v"), f64(w, "dout")
    kw = oracle_args(w)
    o, lse, _ = oracle.fwd(q, k, v, **kw)
    emul = None
    if fa_rule:
        import bf16_emulation
        f32 = lambda x: x.astype(np.float32)  # noqa: E731
        emul = bf16_emulation.fwd_bwd(f32(q), f32(k), f32(v), f32(do), scale=w["scale"], causal=w["causal"],
                                      window=w["window"], sinks=kw["sinks"])

    def judge(name, key, ref):
        if key in fa_rule:
            e_gpu = float(np.abs(got[key] - ref).max())
            e_emu = float(np.abs(emul[key] - ref).max())
            assert e_gpu <= 2.0 * e_emu + 1e-4, f"{name}: max error {e_gpu:.3e} > 2 x bf16 emulation {e_emu:.3e}"
            m_gpu = float(np.abs(got[key] - ref).mean())
            m_emu = float(np.abs(emul[key] - ref).mean())
            assert m_gpu <= max(2e-3, 2.0 * m_emu), f"{name}: mean error {m_gpu:.3e} > 2 x emulation {m_emu:.3e}"
        else:
            check(name, got[key], ref)

    judge("O", "o", o)
    check_lse("LSE", got["lse"], lse)
    if bwd:
        dq, dk, dv, ds = oracle.bwd(q, k, v, do, **kw)
        judge("dQ", "dq", dq)
        judge("dK", "dk", dk)
        judge("dV", "dv", dv)
        if ds is not None:
            scale = max(1.0, float(np.abs(ds).max()))
            err = float(np.abs(got["dsinks"] - ds).max())
            assert err <= 2e-2 * scale, f"dsink max-abs {err:.3e} (scale {scale:.2f})"


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_workload(causal):
    """B=1, s=128, h=2, d=64, scale 1/8 — the tiny forward+backward workload."""
    compare(inputs.make(inputs.workload("tiny_causal" if causal else "tiny")))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_multi_tile(d, causal):
    compare(make_case(100, 10 * d + causal, B=2, s_q=300, h_q=4, d=d, causal=causal))


@pytest.mark.parametrize("s_q,s_kv", [(200, 333), (333, 200), (1, 300), (257, 1)])
def test_bottom_right_alignment(s_q, s_kv):
    compare(make_case(101, s_q % 97, B=2, s_q=s_q, s_kv=s_kv, h_q=2, d=64, causal=True))


@pytest.mark.parametrize("window,causal", [((127, 0), True), ((128, 128), False), ((5, 40), False),
                                           ((0, 0), False), ((-1, 3), False), ((300, -1), False)])
def test_gqa_windows_sinks(window, causal):
    # window (0, 0): one key per row, so dK is a short sum of large, cancelling dS q terms
    # and the bf16 rounding of dS alone reaches the absolute bound; judged by the FA rule
    fa_rule = ("dk", "dq", "dv") if window == (0, 0) else ()
    compare(make_case(102, window[0] % 50 + 3, B=1, s_q=700, h_q=16, h_kv=2, d=64, causal=causal, window=window,
                      sinks=True), fa_rule=fa_rule)


@pytest.mark.parametrize("h_q,h_kv,d", [(6, 2, 64), (6, 2, 128), (8, 1, 128), (5, 5, 64)])
def test_group_sizes(h_q, h_kv, d):
    compare(make_case(103, h_q + 10 * h_kv, B=2, s_q=250, h_q=h_q, h_kv=h_kv, d=d, causal=True, sinks=True))


@pytest.mark.parametrize("share_cu", [True, False])
@pytest.mark.parametrize("d", [64, 128])
def test_packed_batch(d, share_cu):
    """The pages' offsets [0, 17, 300, 428] plus empty and one-token sequences; one offsets
    array for queries and keys (token tiles) and two equal ones (tiles per sequence)."""
    lengths = [17, 283, 128, 0, 1, 0, 300, 129]
    compare(make_case(104, d, h_q=4, h_kv=2, d=d, causal=True, lengths=lengths), share_cu=share_cu)


def _short_lengths(seed, n, long_len):
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in rng.integers(0, 40, size=n)]
    lengths[n // 3] = long_len  # one long sequence among many short ones and some empty
    return lengths


@pytest.mark.parametrize("d,causal,window,sinks,h_q,h_kv", [
    (64, True, (-1, -1), False, 4, 2), (128, True, (-1, -1), True, 2, 2), (64, False, (-1, -1), True, 8, 2),
    (128, False, (30, 10), True, 4, 1), (64, True, (20, 0), False, 16, 2)])
def test_packed_many_short_sequences(d, causal, window, sinks, h_q, h_kv):
    """Token tiles: 128-row query tiles that hold the ends and middles of many short
    sequences (lengths 0 to 39, one of 600), each row masked to its own sequence."""
    lengths = _short_lengths(d + h_q + int(causal), 60, 600)
    compare(make_case(113, d + 7 * h_q + int(causal) + 3 * int(sinks), h_q=h_q, h_kv=h_kv, d=d, causal=causal,
                      window=window, sinks=sinks, lengths=lengths))


def test_packed_batch_different_q_k_packing():
    compare(make_case(105, 0, h_q=4, h_kv=4, d=64, causal=True, lengths=[1, 5, 0, 130, 64, 3],
                      lengths_k=[300, 5, 17, 200, 0, 1], sinks=True))


def test_packed_batch_window():
    compare(make_case(105, 1, h_q=8, h_kv=2, d=128, causal=False, window=(50, 20),
                      lengths=[400, 3, 0, 250], sinks=True))


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("s_q", [1, 2, 4])
def test_decode_shapes(d, s_q):
    """Few query rows per key/value head against a long cache: 4 or 8 rows per key/value
    head take the CUDA-core split path, 16 rows the tensor-core path."""
    compare(make_case(106, d + s_q, B=2, s_q=s_q, s_kv=3000, h_q=8, h_kv=2, d=d, causal=True), bwd=False)


@pytest.mark.parametrize("d", [64, 128])
def test_decode_window_and_sinks(d):
    compare(make_case(106, 7 * d, B=3, s_q=2, s_kv=1500, h_q=8, h_kv=4, d=d, causal=False, window=(300, 0),
                      sinks=True), bwd=False)


@pytest.mark.parametrize("d", [64, 128])
def test_chunked_prefill_split(d):
    """s_q = 64 against a long cache: the tensor-core path with the key range split."""
    compare(make_case(107, d, B=1, s_q=64, s_kv=4100, h_q=8, h_kv=2, d=d, causal=True), bwd=False)


def test_no_split_flag_matches():
    from exact_attention_bwd_gb300 import binding as fa
    w = make_case(107, 3, B=1, s_q=64, s_kv=2100, h_q=8, h_kv=2, d=128, causal=True)
    a = run_gpu(w, bwd=False)
    b = run_gpu(w, bwd=False, flags=fa.FA_FLAG_NO_SPLIT)
    check("O split vs unsplit", a["o"], b["o"], max_abs=1e-2, mean_abs=1e-3)


def test_empty_key_sequences_give_zero_and_neg_inf():
    w = make_case(108, 0, h_q=2, d=64, causal=False, lengths=[5, 3], lengths_k=[0, 4])
    got = run_gpu(w, bwd=True)
    assert np.all(got["o"][:5] == 0)
    assert np.all(np.isneginf(got["lse"][:, :5]))
    assert np.all(got["dq"][:5] == 0)


@pytest.mark.parametrize("causal,window,sinks", [(True, (-1, -1), False), (False, (-1, -1), True),
                                                 (False, (70, 9), True)])
def test_d256_forward(causal, window, sinks):
    """d = 256: one query tile per CTA, 64-key tiles, 256-column accumulator."""
    compare(make_case(110, int(causal) + 3 * int(sinks), B=2, s_q=300, s_kv=333, h_q=8, h_kv=2, d=256,
                      causal=causal, window=window, sinks=sinks), bwd=False)


def test_d256_chunked_prefill_split():
    compare(make_case(110, 9, B=1, s_q=64, s_kv=4100, h_q=8, h_kv=2, d=256, causal=True), bwd=False)


def test_d256_packed_forward():
    compare(make_case(110, 10, h_q=4, h_kv=4, d=256, causal=True, lengths=[17, 283, 0, 1, 129]), bwd=False)


@pytest.mark.parametrize("h_q,h_kv,d,causal", [(128, 1, 64, True), (128, 2, 128, False), (32, 2, 128, True),
                                               (24, 8, 64, False)])
def test_large_groups(h_q, h_kv, d, causal):
    """Group sizes up to the largest supported (128 query heads per key/value head: one
    query position per 128-row tile) and ones that do not divide 128."""
    compare(make_case(111, h_q + h_kv + d, B=1, s_q=70, s_kv=200, h_q=h_q, h_kv=h_kv, d=d, causal=causal,
                      sinks=True))


@pytest.mark.parametrize("d", [64, 128, 256])
def test_decode_long_cache(d):
    """One query row per head against a quarter-million-key cache (the split count caps at
    64 splits, each spanning many key tiles; the combine then spreads more splits than it
    has lanes per row over each lane)."""
    compare(make_case(112, d, B=1, s_q=1, s_kv=262144, h_q=8, h_kv=2, d=d, causal=True), bwd=False)
