"""ctypes binding of libfa_gb300.so (include/fa.h): argument marshalling only.

The functions named like the C entry points (``fa_fwd``, ``fa_bwd``, ...) pass raw
device pointers straight through.  ``forward`` / ``backward`` are conveniences that
take torch CUDA tensors, allocate the outputs and the workspace with torch and call
the same entry points on torch's current stream.  Every step of the computation runs
in the library's kernels; there is no CPU path.  Loading fails loudly when the
library is missing or cannot be built.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_WORKSPACE = 3
FA_ERR_CUDA = 4
FA_ERR_TIMEOUT = 5
FA_ERR_DEVICE_CHECK = 6

FA_FLAG_VALIDATE_CU = 1
FA_FLAG_NO_SPLIT = 2
FA_FLAG_DETERMINISTIC = 4
FA_DTYPE_BF16 = 0
FA_DTYPE_E4M3 = 1
FA_DTYPE_F16 = 2

EXPORTS = ("fa_fwd", "fa_bwd", "fa_fwd_workspace_size", "fa_bwd_workspace_size", "fa_read_device_status",
           "fa_status_string", "fa_profile_enable", "fa_profile_read", "fa_version", "fa_fwd_noalloc")

FA_NOALLOC_SCRATCH_BYTES = 64 << 20


class FaParams(ctypes.Structure):
    """Mirror of ``fa_params``."""
    _fields_ = [
        ("B", ctypes.c_int), ("s_q", ctypes.c_int), ("s_kv", ctypes.c_int),
        ("h_q", ctypes.c_int), ("h_kv", ctypes.c_int), ("d", ctypes.c_int),
        ("softmax_scale", ctypes.c_float), ("causal", ctypes.c_int),
        ("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
        ("sinks", ctypes.c_void_p), ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
        ("max_seqlen_q", ctypes.c_int), ("max_seqlen_k", ctypes.c_int), ("flags", ctypes.c_uint),
        ("seqused_k", ctypes.c_void_p), ("block_table", ctypes.c_void_p), ("page_size", ctypes.c_int),
        ("max_blocks_per_seq", ctypes.c_int), ("num_pages", ctypes.c_int),
        ("dtype", ctypes.c_int), ("q_descale", ctypes.c_void_p), ("k_descale", ctypes.c_void_p),
        ("v_descale", ctypes.c_void_p), ("seqused_q", ctypes.c_void_p),
        ("wait_limit_ns", ctypes.c_ulonglong),
    ]


class FaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {fa_status_string(code)} (status {code})")


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Loads (building first if stale) the CUDA library; raises if that is impossible.

    With FA_TRACE=1 in the environment the trace build (libfa_gb300_trace.so, whose
    kernels record per-role event traces into the workspace; see trace.py) is loaded
    instead of the product library."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        trace = os.environ.get("FA_TRACE", "") == "1"
        path = _build.TRACE_LIB if trace else _build.LIB
        if build_if_missing:
            _build.build(trace=trace)
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is missing; run exact_attention_bwd_gb300/build.py")
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(FaParams)
        vp, sz = ctypes.c_void_p, ctypes.c_size_t
        lib.fa_fwd.argtypes = [P, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.fa_fwd.restype = ctypes.c_int
        lib.fa_bwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.fa_bwd.restype = ctypes.c_int
        lib.fa_fwd_workspace_size.argtypes = [P]
        lib.fa_fwd_workspace_size.restype = sz
        lib.fa_bwd_workspace_size.argtypes = [P]
        lib.fa_bwd_workspace_size.restype = sz
        lib.fa_read_device_status.argtypes = [vp, vp]
        lib.fa_read_device_status.restype = ctypes.c_int
        lib.fa_status_string.argtypes = [ctypes.c_int]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_profile_enable.argtypes = [ctypes.c_int]
        lib.fa_profile_enable.restype = ctypes.c_int
        lib.fa_profile_read.argtypes = [ctypes.c_char_p, ctypes.POINTER(ctypes.c_float)]
        lib.fa_profile_read.restype = ctypes.c_int
        lib.fa_fwd_noalloc.argtypes = [P, vp, vp, vp, vp, vp, vp]
        lib.fa_fwd_noalloc.restype = ctypes.c_int
        lib.fa_version.argtypes = []
        lib.fa_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


# ----------------------------------------------------------------------------------------------
# raw entry points (same names as the C ABI)
# ----------------------------------------------------------------------------------------------

def fa_fwd(params: FaParams, q, k, v, o, lse, workspace, workspace_bytes, stream) -> int:
    return load().fa_fwd(ctypes.byref(params), q, k, v, o, lse, workspace, workspace_bytes, stream)


def fa_fwd_noalloc(params: FaParams, q, k, v, o, lse, stream) -> int:
    """fa_fwd on the library's built-in scratch array: for callers that cannot allocate."""
    return load().fa_fwd_noalloc(ctypes.byref(params), q, k, v, o, lse, stream)


def fa_bwd(params: FaParams, q, k, v, o, lse, dout, dq, dk, dv, dsinks, workspace, workspace_bytes,
           stream) -> int:
    return load().fa_bwd(ctypes.byref(params), q, k, v, o, lse, dout, dq, dk, dv, dsinks, workspace,
                         workspace_bytes, stream)


def fa_fwd_workspace_size(params: FaParams) -> int:
    return int(load().fa_fwd_workspace_size(ctypes.byref(params)))


def fa_bwd_workspace_size(params: FaParams) -> int:
    return int(load().fa_bwd_workspace_size(ctypes.byref(params)))


def fa_read_device_status(workspace, stream) -> int:
    return load().fa_read_device_status(workspace, stream)


def fa_status_string(code: int) -> str:
    return load().fa_status_string(code).decode()


def fa_profile_enable(on: bool) -> int:
    return load().fa_profile_enable(1 if on else 0)


def fa_profile_read(kernel: str):
    ms = ctypes.c_float(0.0)
    rc = load().fa_profile_read(kernel.encode(), ctypes.byref(ms))
    return rc, float(ms.value)


def fa_version() -> str:
    return load().fa_version().decode()


# ----------------------------------------------------------------------------------------------
# torch conveniences: allocation and stream plumbing only
# ----------------------------------------------------------------------------------------------

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def make_params(q, k, *, causal=False, window=(-1, -1), softmax_scale=None, sinks=None, cu_q=None,
                cu_k=None, flags=0, seqused_k=None, block_table=None, s_kv=None, dtype=None, q_descale=None,
                k_descale=None, v_descale=None, seqused_q=None, wait_limit_ns=0) -> FaParams:
    """fa_params from tensor shapes: [B,S,H,D] dense or [T,H,D] packed (with cu_q / cu_k).

    With a block_table ([B, max_blocks_per_seq] int32), k is a page pool
    [num_pages, page_size, h_kv, d] and s_kv (the logical cache length) must be given.
    seqused_q / seqused_k: int32 [B] queries / keys used per sequence, or None."""
    if block_table is not None:
        B, s_q, h_q, d = q.shape
        num_pages, page_size, h_kv, _ = k.shape
        if s_kv is None:
            raise ValueError("a paged cache needs the logical cache length s_kv")
    elif cu_q is None:
        B, s_q, h_q, d = q.shape
        _, s_kv, h_kv, _ = k.shape
    else:
        T_q, h_q, d = q.shape
        T_k, h_kv, _ = k.shape
        B, s_q, s_kv = cu_q.numel() - 1, T_q, T_k
    p = FaParams()
    p.B, p.s_q, p.s_kv, p.h_q, p.h_kv, p.d = B, s_q, s_kv, h_q, h_kv, d
    p.softmax_scale = float(softmax_scale) if softmax_scale else 0.0
    p.causal = 1 if causal else 0
    p.window_left, p.window_right = int(window[0]), int(window[1])
    p.sinks = None if sinks is None else sinks.data_ptr()
    p.cu_seqlens_q = None if cu_q is None else cu_q.data_ptr()
    p.cu_seqlens_k = None if cu_k is None else cu_k.data_ptr()
    p.max_seqlen_q = p.max_seqlen_k = 0
    p.flags = flags
    p.seqused_k = None if seqused_k is None else seqused_k.data_ptr()
    p.seqused_q = None if seqused_q is None else seqused_q.data_ptr()
    p.dtype = FA_DTYPE_BF16 if dtype is None else int(dtype)
    p.q_descale = None if q_descale is None else q_descale.data_ptr()
    p.k_descale = None if k_descale is None else k_descale.data_ptr()
    p.v_descale = None if v_descale is None else v_descale.data_ptr()
    p.wait_limit_ns = int(wait_limit_ns)
    if block_table is not None:
        p.block_table = block_table.data_ptr()
        p.page_size, p.num_pages = int(page_size), int(num_pages)
        p.max_blocks_per_seq = int(block_table.shape[1])
    return p


def _type_code(t):
    """FA_DTYPE_* code of a torch dtype, or None when the library does not take it."""
    import torch
    return {torch.bfloat16: FA_DTYPE_BF16, torch.float16: FA_DTYPE_F16, torch.uint8: FA_DTYPE_E4M3}.get(t)


def _stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check_tensors(q, named):
    """Every tensor handed to the library: on q's CUDA device (the C ABI takes plain device
    pointers; a host pointer there would be dereferenced by the kernels), contiguous (the
    layouts are dense [B, S, H, D], [T, H, D] or the stated vectors), with the given element
    type and element count or shape.  named: (name, tensor or None, dtype, shape or count)."""
    import torch
    if q.device.type != "cuda":
        raise ValueError(f"q must be a CUDA tensor; it is on {q.device}")
    if not q.is_contiguous():
        raise ValueError("q must be contiguous")
    for name, t, dtype, want in named:
        if t is None:
            continue
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch tensor")
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}; every tensor must be on q's device {q.device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if dtype is not None and t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}; it is {t.dtype}")
        if isinstance(want, int):
            if t.numel() != want:
                raise ValueError(f"{name} must have {want} elements; it has {t.numel()}")
        elif want is not None and tuple(t.shape) != tuple(want):
            raise ValueError(f"{name} must have shape {tuple(want)}; it has {tuple(t.shape)}")


def _vector_args(p, sinks, cu_q, cu_k, seqused_q, seqused_k):
    """The optional per-head / per-sequence vectors of a call, for _check_tensors."""
    import torch
    i32, f32 = torch.int32, torch.float32
    return [("sinks", sinks, f32, p.h_q), ("cu_q", cu_q, i32, p.B + 1), ("cu_k", cu_k, i32, p.B + 1),
            ("seqused_q", seqused_q, i32, p.B), ("seqused_k", seqused_k, i32, p.B)]


def _kv_shape(p, k, cu_q, block_table):
    """The shape k must have: [B, s_kv, h_kv, d] dense, [T_k, h_kv, d] packed, or a page pool
    [num_pages, page_size, h_kv, d]; B and d are q's (so no kernel reads past k's end)."""
    if block_table is not None:
        return (p.num_pages, p.page_size, p.h_kv, p.d)
    if cu_q is not None:
        return (p.s_kv, p.h_kv, p.d)
    return (p.B, p.s_kv, p.h_kv, p.d)


def forward(q, k, v, *, causal=False, window=(-1, -1), softmax_scale=None, sinks=None, cu_q=None, cu_k=None,
            flags=0, out=None, lse=None, workspace=None, seqused_k=None, block_table=None, s_kv=None,
            descale=None, seqused_q=None, wait_limit_ns=0):
    """Runs fa_fwd on torch CUDA tensors; returns (o, lse, workspace).

    q, k, v are all bfloat16, all float16, or all uint8 = e4m3 bytes (FA_DTYPE_E4M3);
    descale = (q, k, v) fp32 [B * h_kv] factors or None (all 1).  The output has the
    inputs' type (bf16 for e4m3 inputs)."""
    import torch
    fp8 = q.dtype == torch.uint8
    if _type_code(q.dtype) is None or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must all be bfloat16, all float16 or all uint8 (e4m3 bytes); "
                        f"got {q.dtype}, {k.dtype}, {v.dtype}")
    if descale is not None and not fp8:
        raise TypeError("descale factors apply to e4m3 (uint8) inputs only")
    dq_, dk_, dv_ = descale if descale is not None else (None, None, None)
    p = make_params(q, k, causal=causal, window=window, softmax_scale=softmax_scale, sinks=sinks, cu_q=cu_q,
                    cu_k=cu_k, flags=flags, seqused_k=seqused_k, block_table=block_table, s_kv=s_kv,
                    dtype=_type_code(q.dtype), q_descale=dq_, k_descale=dk_, v_descale=dv_,
                    seqused_q=seqused_q, wait_limit_ns=wait_limit_ns)
    lse_shape = (p.B, p.h_q, p.s_q) if cu_q is None else (p.h_q, p.s_q)
    _check_tensors(q, [("k", k, None, _kv_shape(p, k, cu_q, block_table)), ("v", v, None, k.shape),
                       ("out", out, torch.bfloat16 if fp8 else q.dtype, q.shape), ("lse", lse, torch.float32, lse_shape),
                       ("workspace", workspace, torch.uint8, None),
                       ("block_table", block_table, torch.int32, None if block_table is None else
                        (p.B, p.max_blocks_per_seq)),
                       ("q_descale", dq_, torch.float32, p.B * p.h_kv), ("k_descale", dk_, torch.float32, p.B * p.h_kv),
                       ("v_descale", dv_, torch.float32, p.B * p.h_kv)]
                   + _vector_args(p, sinks, cu_q, cu_k, seqused_q, seqused_k))
    nbytes = fa_fwd_workspace_size(p)
    if nbytes == 0:
        raise FaError(FA_ERR_UNSUPPORTED, "fa_fwd_workspace_size")
    if workspace is None or workspace.numel() < nbytes:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16 if fp8 else q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=q.device)
    rc = fa_fwd(p, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _stream())
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd")
    return out, lse, workspace


def backward(q, k, v, o, lse, dout, *, causal=False, window=(-1, -1), softmax_scale=None, sinks=None,
             cu_q=None, cu_k=None, flags=0, workspace=None, grads=None, seqused_q=None, seqused_k=None,
             wait_limit_ns=0):
    """Runs fa_bwd on torch CUDA tensors; returns (dq, dk, dv, dsinks, workspace).

    q, k, v, o, dout (and dq, dk, dv when given) are all bfloat16 or all float16."""
    import torch
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(f"the backward takes bfloat16 or float16 tensors; q is {q.dtype}")
    named = [("k", k), ("v", v), ("o", o), ("dout", dout)]
    if grads is not None:
        named += [("dq", grads[0]), ("dk", grads[1]), ("dv", grads[2])]
    for name, t in named:
        if t.dtype != q.dtype:
            raise TypeError(f"the backward's tensors must share q's type {q.dtype}; {name} is {t.dtype}")
    p = make_params(q, k, causal=causal, window=window, softmax_scale=softmax_scale, sinks=sinks, cu_q=cu_q,
                    cu_k=cu_k, flags=flags, seqused_q=seqused_q, seqused_k=seqused_k, dtype=_type_code(q.dtype),
                    wait_limit_ns=wait_limit_ns)
    lse_shape = (p.B, p.h_q, p.s_q) if cu_q is None else (p.h_q, p.s_q)
    g = (None, None, None, None) if grads is None else tuple(grads)
    _check_tensors(q, [("k", k, None, _kv_shape(p, k, cu_q, None)), ("v", v, None, k.shape), ("o", o, None, q.shape),
                       ("lse", lse, torch.float32, lse_shape), ("dout", dout, None, q.shape),
                       ("dq", g[0], None, q.shape), ("dk", g[1], None, k.shape), ("dv", g[2], None, k.shape),
                       ("dsinks", g[3], torch.float32, p.h_q), ("workspace", workspace, torch.uint8, None)]
                   + _vector_args(p, sinks, cu_q, cu_k, seqused_q, seqused_k))
    if lse is None:
        raise ValueError("the backward needs the forward's lse")
    nbytes = fa_bwd_workspace_size(p)
    if nbytes == 0:
        raise FaError(FA_ERR_UNSUPPORTED, "fa_bwd_workspace_size")
    if workspace is None or workspace.numel() < nbytes:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if grads is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        dsinks = None if sinks is None else torch.empty_like(sinks)
    else:
        dq, dk, dv, dsinks = grads
    rc = fa_bwd(p, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                _ptr(dsinks), _ptr(workspace), workspace.numel(), _stream())
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd")
    return dq, dk, dv, dsinks, workspace


def device_status(workspace) -> int:
    return fa_read_device_status(_ptr(workspace), _stream())
