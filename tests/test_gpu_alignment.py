"""Output and workspace pointers that are 16-byte but not 32-byte aligned (the least the
C ABI accepts).  The forward writes its output rows and split partials, and the backward
its dK and dV rows, with 32-byte stores where the base pointer allows and with 16-byte
stores otherwise; both forms must give the same bits (dQ, summed by fp32 atomic adds in
no fixed order, to within one bf16 rounding), and the offset run must write nothing
outside its buffers (guard bytes before and after stay as filled).  The aligned runs
themselves are checked against the fp64 oracle by the parity tests of the same shapes."""
from __future__ import annotations

import numpy as np
import pytest

from exact_attention_bwd_gb300 import inputs

from gpu_helpers import dev_inputs

pytestmark = pytest.mark.gpu

GUARD = 256
FILL = 0xA5


def offset_view(nbytes, offset, dtype, shape):
    """A tensor of `shape` that starts `offset` bytes into a filled byte buffer, and the buffer."""
    import torch
    buf = torch.full((GUARD + offset + nbytes + GUARD,), FILL, dtype=torch.uint8, device="cuda")
    t = buf[GUARD + offset:GUARD + offset + nbytes].view(dtype).view(shape)
    return t, buf


def guards_intact(buf, offset, nbytes):
    b = buf.cpu().numpy()
    return bool(np.all(b[:GUARD + offset] == FILL) and np.all(b[GUARD + offset + nbytes:] == FILL))


@pytest.mark.parametrize("case", [
    # d = 64 under a window: 64-key tiles, two CTAs per SM
    dict(B=2, s_q=300, s_kv=300, h_q=16, h_kv=2, d=64, causal=True, window=(127, 0), sinks=True),
    # d = 128 causal: 128-key tiles
    dict(B=2, s_q=333, s_kv=333, h_q=4, h_kv=2, d=128, causal=True, window=(-1, -1), sinks=False),
    # few rows against many keys: key splits, partials in the workspace, then the combine
    dict(B=1, s_q=128, s_kv=8192, h_q=2, h_kv=2, d=128, causal=False, window=(-1, -1), sinks=False),
    # the wide-head forward
    dict(B=1, s_q=200, s_kv=200, h_q=4, h_kv=2, d=256, causal=True, window=(-1, -1), sinks=True),
])
def test_forward_sixteen_byte_aligned_outputs(case):
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    w = inputs.make(dict(wid=30, variant=case["d"] + case["s_kv"] % 7, varlen=False, **case))
    d = dev_inputs(w)
    kw = dict(causal=w["causal"], window=w["window"], softmax_scale=w["scale"], sinks=d["sinks"])
    o_ref, lse_ref, ws = fa.forward(d["q"], d["k"], d["v"], **kw)
    torch.cuda.synchronize()
    o_bytes = o_ref.numel() * 2
    l_bytes = lse_ref.numel() * 4
    w_bytes = ws.numel()
    for off in (16, 48):
        o, obuf = offset_view(o_bytes, off, torch.bfloat16, o_ref.shape)
        lse, lbuf = offset_view(l_bytes, off, torch.float32, lse_ref.shape)
        wsv, wbuf = offset_view(w_bytes, off, torch.uint8, (w_bytes,))
        assert o.data_ptr() % 32 == 16 and wsv.data_ptr() % 32 == 16
        fa.forward(d["q"], d["k"], d["v"], **kw, out=o, lse=lse, workspace=wsv)
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16)), f"O differs at offset {off}"
        assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32)), f"LSE differs at offset {off}"
        assert guards_intact(obuf, off, o_bytes), "write outside O"
        assert guards_intact(lbuf, off, l_bytes), "write outside LSE"
        assert guards_intact(wbuf, off, w_bytes), "write outside the workspace"


@pytest.mark.parametrize("case", [
    dict(B=2, s_q=300, s_kv=300, h_q=16, h_kv=2, d=64, causal=True, window=(127, 0), sinks=False),
    dict(B=2, s_q=333, s_kv=333, h_q=4, h_kv=2, d=128, causal=True, window=(-1, -1), sinks=False),
])
def test_backward_sixteen_byte_aligned_grads(case):
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    w = inputs.make(dict(wid=31, variant=case["d"], varlen=False, **case))
    d = dev_inputs(w)
    kw = dict(causal=w["causal"], window=w["window"], softmax_scale=w["scale"])
    o, lse, _ = fa.forward(d["q"], d["k"], d["v"], **kw)
    dq_ref, dk_ref, dv_ref, _, ws = fa.backward(d["q"], d["k"], d["v"], o, lse, d["dout"], **kw)
    torch.cuda.synchronize()
    off = 16
    views = []
    for ref in (dq_ref, dk_ref, dv_ref):
        views.append(offset_view(ref.numel() * 2, off, torch.bfloat16, ref.shape))
    wsv, wbuf = offset_view(ws.numel(), off, torch.uint8, (ws.numel(),))
    (dq, qbuf), (dk, kbuf), (dv, vbuf) = views
    assert dk.data_ptr() % 32 == 16 and dv.data_ptr() % 32 == 16
    fa.backward(d["q"], d["k"], d["v"], o, lse, d["dout"], **kw, workspace=wsv, grads=(dq, dk, dv, None))
    torch.cuda.synchronize()
    assert torch.equal(dk.view(torch.int16), dk_ref.view(torch.int16)), "dK differs"
    assert torch.equal(dv.view(torch.int16), dv_ref.view(torch.int16)), "dV differs"
    assert torch.allclose(dq.float(), dq_ref.float(), atol=1e-2, rtol=1e-2), "dQ differs"
    for t, buf in ((dq, qbuf), (dk, kbuf), (dv, vbuf)):
        assert guards_intact(buf, off, t.numel() * 2), "write outside a gradient"
    assert guards_intact(wbuf, off, ws.numel()), "write outside the workspace"
