"""GPU parity of the d = 256 backward against the fp64 oracle.

At d = 256 each CTA owns 64 keys and the GEMMs put the query rows (S, dP) or a half of d
(dV^T, dK^T, dQ^T) on the tensor-memory lanes, with P and dS passed through shared memory.
The cases span several 64-key blocks and 128-row query tiles with ragged tails, causal and
two-sided windows with sinks, grouped-query heads (including one query head per key/value
head, P = 128 positions per tile), s_q != s_kv both ways, packed batches with empty
sequences, and fp16 inputs.  Tolerances are the bf16 ones of the other parity tests.
"""
import numpy as np
import pytest

import oracle
from exact_attention_bwd_gb300 import inputs
from gpu_helpers import check, check_lse, f64, oracle_args, run_gpu

pytestmark = pytest.mark.gpu

WID = 150


def case(variant, **kw):
    w = dict(wid=WID, variant=variant, B=2, s_q=300, s_kv=300, h_q=4, h_kv=2, d=256, causal=True,
             window=(-1, -1), sinks=False, varlen=False)
    w.update(kw)
    if "lengths" in w:
        w["varlen"] = True
        w["B"] = len(w["lengths"])
    return inputs.make(w)


def compare(w):
    got = run_gpu(w, bwd=True)
    q, k, v, do = f64(w, "q"), f64(w, "k"), f64(w, "v"), f64(w, "dout")
    kw = oracle_args(w)
    o, lse, _ = oracle.fwd(q, k, v, **kw)
    check("O", got["o"], o)
    check_lse("LSE", got["lse"], lse)
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
def test_backward_d256(i):
    compare(case(i, **CASES[i]))
