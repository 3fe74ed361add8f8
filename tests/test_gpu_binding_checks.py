"""The binding's argument checks on CUDA tensors: every tensor it hands to the C ABI is on
q's device, contiguous, of the stated type and of a shape consistent with q (so no kernel
reads or writes past a buffer).  Each call below fails in the binding, before any launch."""
import pytest

pytestmark = pytest.mark.gpu


def _inputs(B=2, s=64, h_q=4, h_kv=2, d=64):
    import torch
    g = torch.Generator(device="cuda").manual_seed(5)
    q = torch.randn(B, s, h_q, d, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, s, h_kv, d, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, s, h_kv, d, generator=g, device="cuda").to(torch.bfloat16)
    return q, k, v


def test_forward_argument_checks():
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    q, k, v = _inputs()
    with pytest.raises(ValueError, match="contiguous"):
        fa.forward(q, k.transpose(1, 2).contiguous().transpose(1, 2), v)
    with pytest.raises(ValueError, match="shape"):
        fa.forward(q, k[:1].contiguous(), v[:1].contiguous())      # k's batch is not q's
    with pytest.raises(ValueError, match="shape"):
        fa.forward(q, k, v[:, :32].contiguous())                   # v is not k's shape
    with pytest.raises(ValueError, match="device"):
        fa.forward(q, k.cpu(), v)
    with pytest.raises(ValueError, match="shape"):
        fa.forward(q, k, v, out=torch.empty(2, 64, 4, 32, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(TypeError):
        fa.forward(q, k, v, lse=torch.empty(2, 4, 64, dtype=torch.float16, device="cuda"))
    with pytest.raises(ValueError, match="elements"):
        fa.forward(q, k, v, sinks=torch.zeros(3, dtype=torch.float32, device="cuda"))
    with pytest.raises(TypeError):
        fa.forward(q, k, v, sinks=torch.zeros(4, dtype=torch.bfloat16, device="cuda"))
    qp, kp, vp = (t.reshape(-1, t.shape[2], t.shape[3]) for t in (q, k, v))
    with pytest.raises(TypeError):
        cu = torch.tensor([0, 64, 128], dtype=torch.int64, device="cuda")
        fa.forward(qp, kp, vp, cu_q=cu, cu_k=cu)
    # the same calls with valid arguments run
    o, lse, ws = fa.forward(q, k, v, sinks=torch.zeros(4, dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert fa.device_status(ws) == 0


def test_backward_argument_checks():
    import torch
    from exact_attention_bwd_gb300 import binding as fa
    q, k, v = _inputs()
    o, lse, _ = fa.forward(q, k, v, causal=True)
    do = torch.randn_like(q)
    with pytest.raises(ValueError, match="lse"):
        fa.backward(q, k, v, o, None, do, causal=True)
    with pytest.raises(ValueError, match="shape"):
        fa.backward(q, k, v, o, lse[:, :2].contiguous(), do, causal=True)
    with pytest.raises(ValueError, match="shape"):
        fa.backward(q, k, v, o[:, :32].contiguous(), lse, do, causal=True)
    with pytest.raises(ValueError, match="contiguous"):
        fa.backward(q, k, v, o, lse, do.transpose(1, 2).contiguous().transpose(1, 2), causal=True)
    with pytest.raises(ValueError, match="shape"):
        fa.backward(q, k, v, o, lse, do, causal=True,
                    grads=(torch.empty_like(q), torch.empty_like(q), torch.empty_like(k), None))
    dq, dk, dv, _, ws = fa.backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert fa.device_status(ws) == 0
