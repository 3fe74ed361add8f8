"""The C ABI on a host without a GPU: exports, argument checks and workspace sizing.

Every call here fails its host-side checks before anything is launched (the pointers
are never dereferenced), or only asks for a workspace size.
"""
import ctypes
import os
import re
import subprocess

import pytest

from exact_attention_bwd_gb300 import binding as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", src)))


def test_library_exports_every_declared_function():
    lib = fa.load()
    names = declared_functions()
    assert "fa_fwd" in names and "fa_bwd" in names
    for n in names:
        assert hasattr(lib, n), f"{n} is declared in include/fa.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", fa.library_path()], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (fa_\w+)", out))
    assert set(names) <= exported
    assert set(names) == set(fa.EXPORTS)


def test_status_strings():
    for code in range(7):
        assert fa.fa_status_string(code) and fa.fa_status_string(code) != "unknown status"
    assert fa.fa_status_string(99) == "unknown status"


def params(**kw):
    p = fa.FaParams()
    base = dict(B=1, s_q=256, s_kv=256, h_q=4, h_kv=2, d=128, softmax_scale=0.0, causal=0, window_left=-1,
                window_right=-1, sinks=None, cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=0, max_seqlen_k=0,
                flags=0)
    base.update(kw)
    for k, v in base.items():
        setattr(p, k, v)
    return p


FAKE = ctypes.c_void_p(0x100000)     # 16-byte aligned, never dereferenced
MISAL = ctypes.c_void_p(0x100008)


def call_fwd(p, q=FAKE, k=FAKE, v=FAKE, o=FAKE, ws=FAKE, ws_bytes=1 << 30):
    return fa.fa_fwd(p, q, k, v, o, None, ws, ws_bytes, None)


def call_bwd(p, dsinks=FAKE, ws=FAKE, ws_bytes=1 << 30, q=FAKE):
    return fa.fa_bwd(p, q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, dsinks, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(h_q=6, h_kv=4), fa.FA_ERR_INVALID_ARG),          # h_kv must divide h_q
    (dict(B=-1), fa.FA_ERR_INVALID_ARG),
    (dict(h_q=0), fa.FA_ERR_INVALID_ARG),
    (dict(window_left=-2), fa.FA_ERR_INVALID_ARG),
    (dict(cu_seqlens_q=0x2000), fa.FA_ERR_INVALID_ARG),     # cu_q without cu_k
    (dict(d=100), fa.FA_ERR_UNSUPPORTED),                    # not a multiple of 8
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=512), fa.FA_ERR_UNSUPPORTED),
    (dict(h_q=256, h_kv=1, s_q=1), fa.FA_ERR_UNSUPPORTED),   # group of 256 heads
])
def test_forward_rejects(kw, code):
    assert call_fwd(params(**kw)) == code


def test_d256_forward_is_planned():
    # d = 256 forward is supported: it passes the problem checks and stops at the
    # (deliberately too small) workspace, before anything is launched
    assert fa.fa_fwd_workspace_size(params(d=256)) == 256
    assert call_fwd(params(d=256), ws_bytes=16) == fa.FA_ERR_WORKSPACE


def test_forward_pointer_checks():
    p = params()
    assert call_fwd(p, q=None) == fa.FA_ERR_INVALID_ARG
    assert call_fwd(p, o=MISAL) == fa.FA_ERR_INVALID_ARG
    assert call_fwd(p, ws=None) == fa.FA_ERR_INVALID_ARG
    assert call_fwd(p, ws=MISAL) == fa.FA_ERR_INVALID_ARG


def test_workspace_too_small():
    p = params(s_q=1, s_kv=4096, h_q=8, h_kv=2, causal=1)   # decode shape: needs split partials
    need = fa.fa_fwd_workspace_size(p)
    assert need > 256
    assert call_fwd(p, ws_bytes=need - 1) == fa.FA_ERR_WORKSPACE
    pb = params()
    needb = fa.fa_bwd_workspace_size(pb)
    assert call_bwd(pb, ws_bytes=needb - 1) == fa.FA_ERR_WORKSPACE


def test_backward_rejects():
    assert call_bwd(params(sinks=0x3000), dsinks=None) == fa.FA_ERR_INVALID_ARG
    assert call_bwd(params(d=160)) == fa.FA_ERR_UNSUPPORTED
    assert call_bwd(params(h_q=3, h_kv=2)) == fa.FA_ERR_INVALID_ARG
    assert call_bwd(params(), q=MISAL) == fa.FA_ERR_INVALID_ARG


def test_workspace_sizes():
    # dense prefill forward needs only the status word
    assert fa.fa_fwd_workspace_size(params()) == 256
    # backward: status + tiled D and LSE (h_kv x tiles x 128 fp32 each) + dQ accumulator
    p = params(B=2, s_q=300, s_kv=300, h_q=4, h_kv=2, d=64)
    G, P = 2, 64
    tiles = 2 * -(-300 // P)
    stat = 2 * tiles * 128 * 4
    align = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert fa.fa_bwd_workspace_size(p) == 256 + 2 * align(stat) + align(2 * tiles * 128 * 64 * 4)
    # invalid parameters report 0
    assert fa.fa_fwd_workspace_size(params(h_q=5, h_kv=2)) == 0
    assert fa.fa_bwd_workspace_size(params(d=96)) == 0


def test_empty_problem_needs_no_launch_until_status():
    # B = 0: only the status-word reset would run; sizes still defined
    assert fa.fa_fwd_workspace_size(params(B=0)) == 256
    assert fa.fa_bwd_workspace_size(params(B=0)) == 256


def test_profile_read_unknown_kernel():
    rc, _ = fa.fa_profile_read("nope")
    assert rc == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,code", [
    (dict(page_size=100, max_blocks_per_seq=4, num_pages=8), fa.FA_ERR_INVALID_ARG),   # not a multiple of 128
    (dict(page_size=0, max_blocks_per_seq=4, num_pages=8), fa.FA_ERR_INVALID_ARG),
    (dict(page_size=128, max_blocks_per_seq=1, num_pages=8), fa.FA_ERR_INVALID_ARG),   # 128 < s_kv = 256
    (dict(page_size=128, max_blocks_per_seq=2, num_pages=0), fa.FA_ERR_INVALID_ARG),
    (dict(page_size=128, max_blocks_per_seq=2, num_pages=4, cu_seqlens_q=0x2000, cu_seqlens_k=0x2000),
     fa.FA_ERR_UNSUPPORTED),                                                             # paged: dense q only
])
def test_paged_cache_rejects(kw, code):
    assert call_fwd(params(block_table=0x4000, **kw)) == code


def test_paged_cache_is_planned():
    p = params(block_table=0x4000, page_size=128, max_blocks_per_seq=2, num_pages=4)
    assert fa.fa_fwd_workspace_size(p) == 256
    assert call_fwd(p, ws_bytes=16) == fa.FA_ERR_WORKSPACE


def test_backward_cache_forms():
    # partly filled slots are supported by the backward, paged caches are not
    assert fa.fa_bwd_workspace_size(params(seqused_k=0x4000, seqused_q=0x5000)) > 256
    assert call_bwd(params(seqused_k=0x4000), ws_bytes=16) == fa.FA_ERR_WORKSPACE
    assert call_bwd(params(block_table=0x4000, page_size=128, max_blocks_per_seq=2, num_pages=4)) == \
        fa.FA_ERR_UNSUPPORTED
    assert fa.fa_bwd_workspace_size(params(block_table=0x4000, page_size=128, max_blocks_per_seq=2,
                                           num_pages=4)) == 0


def test_deterministic_workspace():
    # the deterministic backward adds one int32 counter per (key/value head, query tile)
    p = params(B=2, s_q=300, s_kv=300, h_q=4, h_kv=2, d=64)
    base = fa.fa_bwd_workspace_size(p)
    tiles = 2 * -(-300 // 64)
    pd = params(B=2, s_q=300, s_kv=300, h_q=4, h_kv=2, d=64, flags=fa.FA_FLAG_DETERMINISTIC)
    assert fa.fa_bwd_workspace_size(pd) == base + (2 * tiles * 4 + 255) // 256 * 256
    # the forward ignores the flag
    assert fa.fa_fwd_workspace_size(pd) == fa.fa_fwd_workspace_size(p)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=fa.FA_DTYPE_E4M3, d=64), fa.FA_ERR_UNSUPPORTED),        # e4m3: d = 128 only
    (dict(dtype=fa.FA_DTYPE_E4M3, d=256), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=7), fa.FA_ERR_INVALID_ARG),
])
def test_e4m3_forward_rejects(kw, code):
    assert call_fwd(params(**kw)) == code


def test_e4m3_packed_and_paged_are_planned():
    # packed e4m3 batches are planned like bf16 ones, without token tiles; paged caches too
    p = params(dtype=fa.FA_DTYPE_E4M3, B=3, s_q=700, s_kv=700, cu_seqlens_q=0x2000, cu_seqlens_k=0x2000)
    assert fa.fa_fwd_workspace_size(p) > 0
    assert call_bwd(p) == fa.FA_ERR_UNSUPPORTED
    kw = dict(B=2, s_q=64, s_kv=1000, block_table=0x4000, page_size=256, max_blocks_per_seq=4, num_pages=8)
    assert fa.fa_fwd_workspace_size(params(dtype=fa.FA_DTYPE_E4M3, **kw)) == fa.fa_fwd_workspace_size(params(**kw))
    bad = dict(kw, page_size=64)
    assert fa.fa_fwd_workspace_size(params(dtype=fa.FA_DTYPE_E4M3, **bad)) == 0


def test_e4m3_workspace_and_backward():
    # V is transposed tile by tile inside the kernel: the workspace is the bf16 forward's
    # (the status word alone without key splits, plus the partials with them)
    for kw in (dict(B=2, s_q=300, s_kv=300, h_q=4, h_kv=2, d=128), dict(B=1, s_q=64, s_kv=32768, h_q=4, h_kv=1, d=128)):
        assert fa.fa_fwd_workspace_size(params(dtype=fa.FA_DTYPE_E4M3, **kw)) == fa.fa_fwd_workspace_size(params(**kw))
    p = params(dtype=fa.FA_DTYPE_E4M3, B=2, s_q=300, s_kv=300, h_q=4, h_kv=2, d=128)
    assert fa.fa_fwd_workspace_size(p) == 256
    assert call_fwd(p, ws_bytes=100) == fa.FA_ERR_WORKSPACE
    assert call_bwd(p) == fa.FA_ERR_UNSUPPORTED


def test_binding_checks_dtypes():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 8, 2, 128, dtype=torch.bfloat16)
    k8 = torch.zeros(1, 8, 2, 128, dtype=torch.uint8)
    with pytest.raises(TypeError):
        fa.forward(q, k8, k8)              # mixed bf16 / e4m3
    with pytest.raises(TypeError):
        fa.forward(q, q, q, descale=(None, None, None))
    with pytest.raises(TypeError):
        fa.backward(k8, k8, k8, q, None, q)


def test_f16_is_planned_like_bf16():
    # fp16 inputs take the same paths and the same workspace as bf16 ones, forward and backward
    for kw in (dict(), dict(B=2, s_q=300, s_kv=300, h_q=4, h_kv=2, d=64), dict(d=256), dict(s_q=1, s_kv=4096),
               dict(cu_seqlens_q=0x2000, cu_seqlens_k=0x2000)):
        assert fa.fa_fwd_workspace_size(params(dtype=fa.FA_DTYPE_F16, **kw)) == fa.fa_fwd_workspace_size(params(**kw))
    for kw in (dict(), dict(d=64, flags=fa.FA_FLAG_DETERMINISTIC), dict(cu_seqlens_q=0x2000, cu_seqlens_k=0x2000)):
        assert fa.fa_bwd_workspace_size(params(dtype=fa.FA_DTYPE_F16, **kw)) == fa.fa_bwd_workspace_size(params(**kw))
    assert call_fwd(params(dtype=fa.FA_DTYPE_F16), ws_bytes=16) == fa.FA_ERR_WORKSPACE
    assert call_bwd(params(dtype=fa.FA_DTYPE_F16), ws_bytes=16) == fa.FA_ERR_WORKSPACE
    assert call_bwd(params(dtype=fa.FA_DTYPE_F16, d=256), ws_bytes=16) == fa.FA_ERR_WORKSPACE


def test_binding_checks_f16_types():
    torch = pytest.importorskip("torch")
    b = torch.zeros(1, 8, 2, 128, dtype=torch.bfloat16)
    h = torch.zeros(1, 8, 2, 128, dtype=torch.float16)
    f = torch.zeros(1, 8, 2, 128, dtype=torch.float32)
    with pytest.raises(TypeError):
        fa.forward(h, b, b)                # mixed fp16 / bf16
    with pytest.raises(TypeError):
        fa.forward(f, f, f)                # fp32 is not an input type
    with pytest.raises(TypeError):
        fa.forward(h, h, h, descale=(None, None, None))
    with pytest.raises(TypeError):
        fa.backward(h, h, h, b, None, h)   # o of another type
    with pytest.raises(TypeError):
        fa.backward(h, h, h, h, None, h, grads=(b, h, h, None))


def test_params_layout_and_constants_match_the_header(tmp_path):
    """The ctypes mirror of fa_params has the C struct's size and field offsets, and the
    binding's constants equal the header's (a plain C compile of include/fa.h)."""
    import shutil
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = [f[0] for f in fa.FaParams._fields_]
    consts = [n for n in dir(fa) if re.fullmatch(r"FA_(OK|ERR_\w+|FLAG_\w+|DTYPE_\w+)", n)]
    src = ["#include <stdio.h>", "#include <stddef.h>", '#include "fa.h"', "int main(void) {",
           '  printf("size %zu\\n", sizeof(fa_params));']
    src += [f'  printf("off {f} %zu\\n", offsetof(fa_params, {f}));' for f in fields]
    src += [f'  printf("const {n} %lld\\n", (long long)({n}));' for n in consts]
    src += ["  return 0;", "}"]
    c = tmp_path / "layout.c"
    c.write_text("\n".join(src) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), str(c), "-o", str(exe)],
                   check=True)
    got = {}
    for line in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines():
        kind, *rest = line.split()
        got[(kind, rest[0]) if kind != "size" else ("size", "")] = int(rest[-1])
    assert got[("size", "")] == ctypes.sizeof(fa.FaParams)
    for f in fields:
        assert got[("off", f)] == getattr(fa.FaParams, f).offset, f
    assert len(consts) == 13  # 7 status codes, 3 flags, 3 element types
    for n in consts:
        assert got[("const", n)] == getattr(fa, n), n


def test_d192_is_planned():
    """d = 192 runs forward (dense, packed, decode and split shapes) and backward."""
    for kw in (dict(d=192), dict(d=192, s_q=1, s_kv=4096), dict(d=192, s_q=64, s_kv=8192, causal=1)):
        assert fa.fa_fwd_workspace_size(params(**kw)) >= 256, kw
    p = params(B=2, s_q=300, s_kv=300, h_q=4, h_kv=2, d=192)
    tiles = 2 * -(-300 // 64)
    stat = 2 * tiles * 128 * 4
    align = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert fa.fa_bwd_workspace_size(p) == 256 + 2 * align(stat) + align(2 * tiles * 128 * 192 * 4)


def test_d256_backward_workspace():
    """d = 256: 64-key blocks; the workspace holds the same per-row statistics and a dQ
    accumulator of 128 rows x 256 fp32 columns per (query tile, key/value head)."""
    p = params(B=2, s_q=300, s_kv=300, h_q=4, h_kv=2, d=256)
    tiles = 2 * -(-300 // 64)   # P = 64 positions per 128-row tile (G = 2)
    stat = 2 * tiles * 128 * 4
    align = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert fa.fa_bwd_workspace_size(p) == 256 + 2 * align(stat) + align(2 * tiles * 128 * 256 * 4)
    assert call_bwd(p, ws_bytes=16) == fa.FA_ERR_WORKSPACE


@pytest.mark.parametrize("d", [64, 128, 192, 256])
def test_deterministic_workspace_adds_tile_counters(d):
    """FA_FLAG_DETERMINISTIC (every head dimension) adds one int32 turn counter per (key/value
    head, query tile) to the backward's workspace."""
    def align(x):
        return (x + 255) // 256 * 256
    p0 = params(B=2, s_q=300, s_kv=300, h_q=4, h_kv=2, d=d)
    p1 = params(B=2, s_q=300, s_kv=300, h_q=4, h_kv=2, d=d, flags=fa.FA_FLAG_DETERMINISTIC)
    tiles = 2 * ((300 + 63) // 64)  # P = 64 positions per tile (G = 2)
    assert fa.fa_bwd_workspace_size(p1) == fa.fa_bwd_workspace_size(p0) + align(2 * tiles * 4)


def test_binding_rejects_host_tensors():
    """The library takes device pointers only: host tensors never reach it (no CPU path)."""
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 8, 2, 128, dtype=torch.bfloat16)
    lse = torch.zeros(1, 2, 8, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA"):
        fa.forward(q, q, q)
    with pytest.raises(ValueError, match="CUDA"):
        fa.backward(q, q, q, q, lse, q)


def test_tail_split_plans():
    """The forward planner's tail split, by its workspace (status word + fp32 partials of
    the tail rows).  Without a device the planner counts 152 SMs, the GB300's count.  The
    d = 128 chunked-prefill shape (512 items of one unit each, a last round of 56) cuts the
    last 56 units into 8 key ranges instead of splitting every unit in two; d = 256 (1024
    items, two per unit, a last wave of 112) cuts the last 56 units into 4; with 8 batch
    entries (64 items, under one round) every unit's keys stay split (7 ways)."""
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731

    def ws(d, k, rows):
        return 256 + al(rows * k * d * 4) + al(rows * k * 4)
    kw = dict(s_q=64, s_kv=32768, h_q=32, h_kv=8, causal=1)
    assert fa.fa_fwd_workspace_size(params(B=64, d=128, **kw)) == ws(128, 8, 56 * 4 * 64)
    assert fa.fa_fwd_workspace_size(params(B=64, d=256, **kw)) == ws(256, 4, 56 * 4 * 64)
    assert fa.fa_fwd_workspace_size(params(B=8, d=128, **kw)) == ws(128, 7, 8 * 32 * 64)
    # no key split planned (B=40 against 4096 keys: 320 items, a last round of 16): the last
    # 16 units are cut 8 ways (2 + 1/8 rounds instead of 3), at d = 64 and 128
    kw40 = dict(B=40, s_q=64, s_kv=4096, h_q=32, h_kv=8, causal=1)
    for d in (64, 128):
        assert fa.fa_fwd_workspace_size(params(d=d, **kw40)) == ws(d, 8, 16 * 4 * 64)
    # the headline shape (no split, no tail): the status word alone
    assert fa.fa_fwd_workspace_size(params(B=2, s_q=8192, s_kv=8192, h_q=16, h_kv=16, d=128, causal=1)) == 256
    # e4m3 takes the same plans as bf16
    assert fa.fa_fwd_workspace_size(params(B=64, d=128, dtype=fa.FA_DTYPE_E4M3, **kw)) == ws(128, 8, 56 * 4 * 64)
