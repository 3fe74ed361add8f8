"""fa_fwd_noalloc: the forward for callers that cannot allocate device memory.

Such a caller (a host framework that owns every allocation, or a loop that must not
enter the CUDA allocator) cannot pass fa_fwd a workspace, so fa_fwd_noalloc runs the same
kernels on a scratch array compiled into the library.  These tests call it through the
C ABI on shapes that do use scratch (split-KV partial results: the decode kernel and the
split tensor-core forward) and compare it with fa_fwd on a workspace allocated here, on
two calls in a row with different problems, so the second call also shows that what the
first one left in the shared array does not leak into its results.

This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

from exact_attention_bwd_gb300 import inputs
from gpu_helpers import check, check_lse, dev_inputs, from_dev

pytestmark = pytest.mark.gpu


def _problem(wid, variant, *, B, s_q, s_kv, h_q, h_kv, d):
    return inputs.make(dict(wid=wid, variant=variant, B=B, s_q=s_q, s_kv=s_kv, h_q=h_q, h_kv=h_kv, d=d,
                            causal=True, window=(-1, -1), sinks=False, varlen=False))


def _run_both(w):
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    d = dev_inputs(w)
    kw = dict(causal=True, softmax_scale=w["scale"])
    o_ref, lse_ref, ws = fa.forward(d["q"], d["k"], d["v"], **kw)
    p = fa.make_params(d["q"], d["k"], **kw)
    assert fa.fa_fwd_workspace_size(p) > 256, "the case must use scratch beyond the status word"
    o = torch.full_like(d["q"], float("nan"))
    lse = torch.full_like(lse_ref, float("nan"))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = fa.fa_fwd_noalloc(p, ctypes.c_void_p(d["q"].data_ptr()), ctypes.c_void_p(d["k"].data_ptr()),
                           ctypes.c_void_p(d["v"].data_ptr()), ctypes.c_void_p(o.data_ptr()),
                           ctypes.c_void_p(lse.data_ptr()), stream)
    assert rc == fa.FA_OK, fa.fa_status_string(rc)
    torch.cuda.synchronize()
    return from_dev(o), lse.cpu().numpy().astype(np.float64), from_dev(o_ref), lse_ref.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("first,second", [
    # decode kernel (CUDA cores, split-KV partials) then the split tensor-core forward
    (dict(B=2, s_q=1, s_kv=3000, h_q=8, h_kv=2, d=128), dict(B=1, s_q=64, s_kv=4100, h_q=8, h_kv=2, d=128)),
    # two decode calls of different shapes
    (dict(B=3, s_q=4, s_kv=2500, h_q=8, h_kv=2, d=64), dict(B=2, s_q=1, s_kv=5000, h_q=16, h_kv=4, d=256)),
])
def test_noalloc_matches_workspace_forward_twice(first, second):
    for n, shape in enumerate((first, second)):
        w = _problem(109, 10 * n + shape["d"] % 7, **shape)
        o, lse, o_ref, lse_ref = _run_both(w)
        check(f"O call {n + 1}", o, o_ref)
        check_lse(f"LSE call {n + 1}", lse, lse_ref)


def test_noalloc_rejects_problems_beyond_its_scratch():
    from exact_attention_bwd_gb300 import binding as fa
    p = fa.FaParams()
    # a decode-shaped problem (8 query rows per key/value head) whose split partials alone
    # need 4096 * 32 * 2 rows * 128 floats = 128 MiB
    p.B, p.s_q, p.s_kv, p.h_q, p.h_kv, p.d = 4096, 2, 1024, 32, 8, 128
    p.causal, p.window_left, p.window_right = 1, -1, -1
    assert fa.fa_fwd_workspace_size(p) > fa.FA_NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x100000)
    rc = fa.fa_fwd_noalloc(p, fake, fake, fake, fake, None, None)
    assert rc == fa.FA_ERR_WORKSPACE
