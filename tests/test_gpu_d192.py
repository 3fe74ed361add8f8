"""GPU parity at head dimension 192 against the fp64 oracle, forward and backward.

d = 192 is one of the head sizes the pages pad to (dew-flash-attn PyPI page, the FA3
head-dim padding to 64 / 128 / 192 / 256; fa4-jax PyPI page, Restrictions: d a multiple
of 8 and at most 256).  The forward runs the wide-head kernel with three 64-column chunks
(one 128-row query tile per CTA, 64-key tiles, O in 192 tensor-memory columns); the
backward runs the wide-head layout (64 keys per CTA, query rows or halves of d on the
lanes) with K = 192 for S and dP and a zero fourth chunk under the second d-half GEMMs;
decode shapes take the CUDA-core kernel with six head-dim elements per lane, and long
key ranges are split and merged by the combine kernel.  The cases span several 64-key
blocks and query tiles with ragged tails, causal and two-sided windows with sinks,
grouped-query heads (one query head per key/value head included), s_q != s_kv both ways,
packed batches with empty sequences, and fp16 inputs.  Tolerances are the bf16 ones of the
other parity tests.
"""
import numpy as np
import pytest

import oracle
from exact_attention_bwd_gb300 import inputs
from gpu_helpers import check, check_lse, f64, oracle_args, run_gpu

pytestmark = pytest.mark.gpu

WID = 160


def case(variant, **kw):
    w = dict(wid=WID, variant=variant, B=2, s_q=300, s_kv=300, h_q=4, h_kv=2, d=192, causal=True,
             window=(-1, -1), sinks=False, varlen=False)
    w.update(kw)
    if "lengths" in w:
        w["varlen"] = True
        w["B"] = len(w["lengths"])
    return inputs.make(w)


def compare(w, bwd=True):
    got = run_gpu(w, bwd=bwd)
    q, k, v, do = f64(w, "q"), f64(w, "k"), f64(w, "v"), f64(w, "dout")
    kw = oracle_args(w)
    o, lse, _ = oracle.fwd(q, k, v, **kw)
    check("O", got["o"], o)
    check_lse("LSE", got["lse"], lse)
    if not bwd:
        return
    dq, dk, dv, ds = oracle.bwd(q, k, v, do, **kw)
    check("dQ", got["dq"], dq)
    check("dK", got["dk"], dk)
    check("dV", got["dv"], dv)
    if ds is not None:
        err = float(np.abs(got["dsinks"] - ds).max())
        assert err <= 2e-2 * max(1.0, float(np.abs(ds).max())), f"dsink max-abs {err:.3e}"


CASES = [
    dict(),
    dict(causal=False),
    dict(causal=False, window=(130, 40), h_q=8, h_kv=2, sinks=True),
    dict(window=(70, 0), h_q=4, h_kv=4, sinks=True),
    dict(s_q=200, s_kv=650, h_q=6, h_kv=2),
    dict(s_q=650, s_kv=200, h_q=4, h_kv=4),
    dict(B=1, s_q=1024, s_kv=1024, h_q=8, h_kv=8),
    dict(lengths=[17, 283, 128, 0, 1, 0, 300, 129], h_q=4, h_kv=2),
    dict(lengths=[400, 3, 0, 250], h_q=8, h_kv=2, causal=False, window=(50, 20), sinks=True),
    dict(dtype="f16", h_q=8, h_kv=2, sinks=True),
]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_forward_backward_d192(i):
    compare(case(i, **CASES[i]))


@pytest.mark.parametrize("s_q", [1, 2, 64])
def test_decode_and_chunked_prefill_d192(s_q):
    """A long cache: 4 and 8 rows per key/value head (the CUDA-core kernel for 4, the
    tensor-core kernel for 8) and s_q = 64 (the tensor-core kernel with split keys)."""
    compare(case(20 + s_q, B=2, s_q=s_q, s_kv=4100, h_q=8, h_kv=2), bwd=False)


def test_decode_d192_sinks_window():
    compare(case(30, B=3, s_q=1, s_kv=1500, h_q=8, h_kv=2, causal=False, window=(300, 0), sinks=True), bwd=False)
