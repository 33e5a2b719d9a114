"""C-ABI checks that need no GPU: the library builds, loads, exports every symbol
include/fa.h declares, and rejects bad arguments with the documented codes
before touching a device.  No compute call is made here: the pointers are fake,
never-allocated addresses, so a call whose arguments all pass validation (it would
go on to launch work) is made only where no CUDA device exists, and there it must
fail with FA_ERR_DEVICE.
"""
import ctypes
import os
import re

import pytest

from tiled_attention_11_gb300 import _lib
from tiled_attention_11_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def L():
    build()
    return _lib.lib()


def _device_present() -> bool:
    import torch
    return torch.cuda.is_available() or os.path.exists("/dev/nvidiactl")


DEVICE_PRESENT = _device_present()


def reaches_device(call):
    """Make a call that passes every host check only where no device can run it."""
    if DEVICE_PRESENT:
        return
    assert call() == _lib.FA_ERR_DEVICE


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_strerror"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in fa.h but not exported"
    assert set(declared_functions()) == set(_lib.EXPORTED)


def test_strerror_strings(L):
    for code in range(0, 9):
        assert len(_lib.strerror(code)) > 3
    assert "unknown" in _lib.strerror(99)


# fake, never-dereferenced device addresses (16-byte aligned, far apart)
A = 0x10000000
GAP = 0x10000000


def ptrs(n, base=A):
    return [base + i * GAP for i in range(n)]


def fwd_call(L, q, k, v, o, lse, B=2, H=3, Nq=100, Nk=77, D=64, scale=0.125, causal=1):
    vp = ctypes.c_void_p
    return L.fa_fwd(vp(q), vp(k), vp(v), vp(o), vp(lse), B, H, Nq, Nk, D, scale, causal, None)


def bwd_call(L, p, B=2, H=3, Nq=100, Nk=77, D=64, scale=0.125, causal=1, ws=None, ws_bytes=None):
    vp = ctypes.c_void_p
    need = L.fa_bwd_workspace_size(B, H, Nq, Nk, D)
    ws = p[9] if ws is None else ws
    ws_bytes = need if ws_bytes is None else ws_bytes
    return L.fa_bwd(*[vp(x) for x in p[:9]], B, H, Nq, Nk, D, scale, causal, vp(ws), ws_bytes, None)


def test_fwd_validation_codes(L):
    q, k, v, o, lse = ptrs(5)
    assert fwd_call(L, 0, k, v, o, lse) == _lib.FA_ERR_INVALID_ARG
    assert fwd_call(L, q, k, v, o, 0) == _lib.FA_ERR_INVALID_ARG
    assert fwd_call(L, q, k, v, o, lse, D=48) == _lib.FA_ERR_UNSUPPORTED_D
    assert fwd_call(L, q, k, v, o, lse, D=256) == _lib.FA_ERR_UNSUPPORTED_D
    assert fwd_call(L, q, k, v, o, lse, Nq=0) == _lib.FA_ERR_INVALID_ARG
    assert fwd_call(L, q, k, v, o, lse, Nk=-1) == _lib.FA_ERR_INVALID_ARG
    assert fwd_call(L, q, k, v, o, lse, B=0) == _lib.FA_ERR_INVALID_ARG
    assert fwd_call(L, q, k, v, o, lse, scale=float("nan")) == _lib.FA_ERR_INVALID_ARG
    assert fwd_call(L, q, k, v, o, lse, scale=float("inf")) == _lib.FA_ERR_INVALID_ARG
    assert fwd_call(L, q, k, v, o, lse, scale=-0.1) == _lib.FA_ERR_INVALID_ARG
    assert fwd_call(L, q, k, v, o, lse, B=256, H=256) == _lib.FA_ERR_INVALID_ARG  # B*H > 65535
    assert fwd_call(L, q + 8, k, v, o, lse) == _lib.FA_ERR_MISALIGNED
    assert fwd_call(L, q, k, v, o + 2, lse) == _lib.FA_ERR_MISALIGNED
    assert fwd_call(L, q, k, v, o, lse + 2) == _lib.FA_ERR_MISALIGNED
    # output overlapping an input
    assert fwd_call(L, q, k, v, q + 1024, lse) == _lib.FA_ERR_INVALID_ARG
    assert fwd_call(L, q, k, v, o, o + 16) == _lib.FA_ERR_INVALID_ARG
    # every argument valid: the only failure left is the missing sm_103 device
    reaches_device(lambda: fwd_call(L, q, k, v, o, lse))


def test_bwd_validation_codes(L):
    p = ptrs(10)
    assert bwd_call(L, [0] + p[1:]) == _lib.FA_ERR_INVALID_ARG
    assert bwd_call(L, p, D=8) == _lib.FA_ERR_UNSUPPORTED_D
    assert bwd_call(L, p[:6] + [p[6] + 4] + p[7:]) == _lib.FA_ERR_MISALIGNED
    need = L.fa_bwd_workspace_size(2, 3, 100, 77, 64)
    assert bwd_call(L, p, ws_bytes=need - 1) == _lib.FA_ERR_WORKSPACE
    assert bwd_call(L, p, ws=0) == _lib.FA_ERR_WORKSPACE
    assert bwd_call(L, p, ws=p[9] + 128) == _lib.FA_ERR_WORKSPACE
    # workspace overlapping dq
    assert bwd_call(L, p[:9] + [p[6] + 256]) == _lib.FA_ERR_INVALID_ARG
    # dk overlapping an input
    assert bwd_call(L, p[:7] + [p[0] + 64] + p[8:]) == _lib.FA_ERR_INVALID_ARG
    reaches_device(lambda: bwd_call(L, p))


def test_workspace_size_formula(L):
    def rnd(x):
        return (x + 255) // 256 * 256
    for (B, H, Nq, Nk, D) in [(2, 3, 100, 77, 64), (1, 1, 1, 1, 16), (4, 32, 4096, 4096, 128), (1, 8, 65537, 65537, 128)]:
        nq_pad = (Nq + 63) // 64 * 64
        rows = B * H * nq_pad
        assert L.fa_bwd_workspace_size(B, H, Nq, Nk, D) == rnd(rows * D * 4) + 2 * rnd(rows * 4)
    assert L.fa_bwd_workspace_size(1, 1, 16, 16, 24) == 0
    assert L.fa_bwd_workspace_size(0, 1, 16, 16, 64) == 0


def test_binding_rejects_missing_gpu():
    """The Python path has no CPU fallback: without a GPU the call raises."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    q = torch.zeros(1, 1, 8, 16, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        _lib.forward(q, q, q, causal=False)


def test_wait_probe_needs_device(L):
    reaches_device(lambda: L.fa_wait_probe(1000, None))


def test_noalloc_size_limit_checked_on_host(L):
    vp = ctypes.c_void_p
    p = [vp(x) for x in ptrs(9)]
    assert L.fa_bwd_noalloc(*p, 4, 32, 4096, 4096, 128, 0.088, 1, None) == _lib.FA_ERR_SCRATCH_LIMIT
    reaches_device(lambda: L.fa_bwd_noalloc(*p, 2, 3, 100, 77, 64, 0.125, 1, None))


def test_varlen_validation_codes(L):
    vp = ctypes.c_void_p
    q, k, v, o, lse, cq, ck = (vp(x) for x in ptrs(7))
    call = lambda **kw: L.fa_fwd_varlen(q, k, v, o, lse, kw.get("cq", cq), ck, kw.get("B", 3), 2, 100, 90,  # noqa: E731
                                        kw.get("mq", 60), 50, kw.get("D", 64), 0.125, 1, None)
    assert call(cq=vp(0)) == _lib.FA_ERR_INVALID_ARG
    assert call(B=0) == _lib.FA_ERR_INVALID_ARG
    assert call(mq=0) == _lib.FA_ERR_INVALID_ARG
    assert call(D=80) == _lib.FA_ERR_UNSUPPORTED_D
    assert call(cq=vp(ptrs(1)[0] + 2)) == _lib.FA_ERR_MISALIGNED
    reaches_device(lambda: call())
    rows = 64 * ((100 + 63) // 64 + 3)
    def rnd(x):
        return (x + 255) // 256 * 256
    assert L.fa_bwd_varlen_workspace_size(3, 2, 100, 60, 64) == rnd(2 * rows * 64 * 4) + 2 * rnd(2 * rows * 4)


def test_window_validation_codes(L):
    vp = ctypes.c_void_p
    q, k, v, o, lse = (vp(x) for x in ptrs(5))
    call = lambda **kw: L.fa_fwd_window(kw.get("q", q), k, v, o, lse, 2, 3, 100, 77, kw.get("D", 64), 0.125, 1,  # noqa: E731
                                        kw.get("wl", 16), -1, kw.get("g", 4), None, 0, None)
    assert call(q=vp(0)) == _lib.FA_ERR_INVALID_ARG
    assert call(D=48) == _lib.FA_ERR_UNSUPPORTED_D
    assert call(q=vp(ptrs(1)[0] + 8)) == _lib.FA_ERR_MISALIGNED
    # any window / global-token values are valid (negative: unbounded, large: clipped)
    for wl, g in ((-1, 0), (0, 0), (1 << 30, 1 << 30), (-5, -3)):
        reaches_device(lambda: call(wl=wl, g=g))
    p = [vp(x) for x in ptrs(10)]
    need = L.fa_bwd_workspace_size(2, 3, 100, 77, 64)
    assert L.fa_bwd_window(*p[:9], 2, 3, 100, 77, 64, 0.125, 1, 16, -1, 4, p[9], need - 1, None) == _lib.FA_ERR_WORKSPACE
    reaches_device(lambda: L.fa_bwd_window(*p[:9], 2, 3, 100, 77, 64, 0.125, 1, 16, -1, 4, p[9], need, None))


def test_fp8_validation_codes(L):
    vp = ctypes.c_void_p
    q, k, vt, qd, kd, vd, o, lse = (vp(x) for x in ptrs(8))
    call = lambda **kw: L.fa_fwd_fp8(q, k, vt, kw.get("ldv", 96), qd, kd, vd, kw.get("o", o), lse, 2, 3, 100,  # noqa: E731
                                     kw.get("Nk", 90), kw.get("D", 128), 0.125, 1, None)
    assert call(D=32) == _lib.FA_ERR_UNSUPPORTED_D
    assert call(ldv=88) == _lib.FA_ERR_INVALID_ARG      # < Nk
    assert call(ldv=100) == _lib.FA_ERR_INVALID_ARG     # not a multiple of 16
    assert call(o=vp(0)) == _lib.FA_ERR_INVALID_ARG
    assert call(o=vp(ptrs(1)[0] + 8)) == _lib.FA_ERR_MISALIGNED
    reaches_device(lambda: call())
    x, c, a, d = (vp(v) for v in ptrs(4))
    assert L.fa_quantize_e4m3(x, 0, c, a, d, None) == _lib.FA_ERR_INVALID_ARG
    assert L.fa_quantize_e4m3(vp(ptrs(1)[0] + 2), 100, c, a, d, None) == _lib.FA_ERR_MISALIGNED
    assert L.fa_quantize_e4m3(x, 100, x, a, d, None) == _lib.FA_ERR_INVALID_ARG  # codes overlap x
    reaches_device(lambda: L.fa_quantize_e4m3(x, 100, c, a, d, None))
    assert L.fa_quantize_e4m3_transposed(x, 1, 2, 100, 64, 100, c, a, d, None) == _lib.FA_ERR_INVALID_ARG
    assert L.fa_quantize_e4m3_transposed(x, 1, 2, 100, 48, 112, c, a, d, None) == _lib.FA_ERR_UNSUPPORTED_D
    reaches_device(lambda: L.fa_quantize_e4m3_transposed(x, 1, 2, 100, 64, 112, c, a, d, None))
    q, k, v, q8, k8, vt8, am, de = (vp(x) for x in ptrs(8))
    qkv = lambda **kw: L.fa_quantize_qkv_e4m3(kw.get("q", q), k, v, 2, 3, 100, kw.get("Nk", 90),  # noqa: E731
                                             kw.get("D", 128), kw.get("q8", q8), k8, vt8, kw.get("ldv", 96),
                                             kw.get("am", am), kw.get("de", de), None)
    assert qkv(D=32) == _lib.FA_ERR_UNSUPPORTED_D
    assert qkv(ldv=80) == _lib.FA_ERR_INVALID_ARG       # < Nk
    assert qkv(ldv=100) == _lib.FA_ERR_INVALID_ARG      # not a multiple of 16
    assert qkv(Nk=0) == _lib.FA_ERR_INVALID_ARG
    assert qkv(q8=vp(0)) == _lib.FA_ERR_INVALID_ARG
    assert qkv(q8=q) == _lib.FA_ERR_INVALID_ARG         # codes overlap their input
    assert qkv(de=vp(ptrs(8)[6] + 8)) == _lib.FA_ERR_INVALID_ARG  # descale[3] overlaps amax[3]
    assert qkv(q=vp(ptrs(1)[0] + 8)) == _lib.FA_ERR_MISALIGNED
    assert qkv(am=vp(ptrs(8)[6] + 2)) == _lib.FA_ERR_MISALIGNED
    reaches_device(lambda: qkv())


def test_step_host_validation_codes(L):
    vp = ctypes.c_void_p
    p = [vp(x) for x in ptrs(10)]
    need = L.fa_step_host_device_bytes(2, 3, 100, 77, 64)
    assert need > 0 and need % 256 == 0
    assert L.fa_step_host_device_bytes(2, 3, 100, 77, 48) == 0
    call = lambda dev=p[9], nbytes=need, D=64: L.fa_step_host(*p[:9], dev, nbytes, 2, 3, 100, 77, D, 0.125, 1, None)  # noqa: E731
    assert call(dev=vp(0)) == _lib.FA_ERR_INVALID_ARG
    assert call(D=48) == _lib.FA_ERR_UNSUPPORTED_D
    assert call(nbytes=need - 1) == _lib.FA_ERR_WORKSPACE
    assert call(dev=vp(ptrs(1)[0] + 16)) == _lib.FA_ERR_WORKSPACE
    reaches_device(lambda: call())


def test_window_split_workspace(L):
    vp = ctypes.c_void_p
    # causal or short key ranges need no split; non-causal long ones with global tokens do
    assert L.fa_fwd_window_workspace_size(1, 2, 8192, 8192, 64, 1, 256, -1, 64) == 0
    assert L.fa_fwd_window_workspace_size(1, 2, 4000, 4000, 64, 0, 256, 256, 64) == 0   # 32 key tiles
    need = L.fa_fwd_window_workspace_size(1, 2, 5000, 5000, 64, 0, 100, 100, 40)
    # 1 global pair x 256 rows x 3 chunks of 16 key tiles: O (64 fp32) and 4 floats per record
    recs = 2 * 256 * 3
    assert need == (recs * 64 * 4 + 255) // 256 * 256 + (recs * 16 + 255) // 256 * 256
    assert L.fa_fwd_window_workspace_size(1, 2, 5000, 5000, 64, 0, 100, 100, 0) == 0   # no global tokens
    q, k, v, o, lse, ws = (vp(x) for x in ptrs(6))
    args = (q, k, v, o, lse, 1, 2, 5000, 5000, 64, 0.125, 0, 100, 100, 40)
    assert L.fa_fwd_window(*args, None, 0, None) == _lib.FA_ERR_WORKSPACE
    assert L.fa_fwd_window(*args, ws, need - 1, None) == _lib.FA_ERR_WORKSPACE
    assert L.fa_fwd_window(*args, vp(ptrs(6)[5] + 16), need, None) == _lib.FA_ERR_WORKSPACE  # misaligned
    reaches_device(lambda: L.fa_fwd_window(*args, ws, need, None))


def test_window_bwd_split_workspace(L):
    base = L.fa_bwd_workspace_size(1, 2, 5000, 5000, 64)
    assert L.fa_bwd_window_workspace_size(1, 2, 5000, 5000, 64, 100, 100, 0) == base     # no global tokens
    assert L.fa_bwd_window_workspace_size(1, 2, 4000, 4000, 64, 100, 100, 40) == \
        L.fa_bwd_workspace_size(1, 2, 4000, 4000, 64)                                      # 63 query steps
    # 5000 queries = 79 steps > 64: one global key tile, dK and dV rows of 64 fp32
    assert L.fa_bwd_window_workspace_size(1, 2, 5000, 5000, 64, 100, 100, 40) == base + (2 * 128 * 2 * 64 * 4)
    need = base + 2 * 128 * 2 * 64 * 4
    vp = ctypes.c_void_p
    p = [vp(x) for x in ptrs(10)]
    args = (*p[:9], 1, 2, 5000, 5000, 64, 0.125, 0, 100, 100, 40, p[9])
    assert L.fa_bwd_window(*args, base, None) == _lib.FA_ERR_WORKSPACE      # split area missing
    assert L.fa_bwd_window(*args, need - 1, None) == _lib.FA_ERR_WORKSPACE
    reaches_device(lambda: L.fa_bwd_window(*args, need, None))


def test_noalloc_scratch_boundary(L):
    """fa_bwd_noalloc's limit is fa_bwd_workspace_size <= 32 MiB, checked before launching:
    at D = 128 and 64 queries per head, 1008 heads fit and 1009 do not."""
    vp = ctypes.c_void_p
    p = [vp(x) for x in ptrs(9)]
    limit = 32 << 20
    assert L.fa_bwd_workspace_size(1, 1008, 64, 64, 128) <= limit < L.fa_bwd_workspace_size(1, 1009, 64, 64, 128)
    assert L.fa_bwd_noalloc(*p, 1, 1009, 64, 64, 128, 0.088, 1, None) == _lib.FA_ERR_SCRATCH_LIMIT
    # short heads count as 64 padded rows each
    assert L.fa_bwd_noalloc(*p, 1, 1009, 1, 1, 128, 0.088, 1, None) == _lib.FA_ERR_SCRATCH_LIMIT
    reaches_device(lambda: L.fa_bwd_noalloc(*p, 1, 1008, 64, 64, 128, 0.088, 1, None))


def test_length_limit(L):
    """Sequence lengths (and packed totals) above 2^29 are rejected on the host: rows and
    tiles are indexed with 32-bit ints, and an unbounded window side must reach past
    every row."""
    vp = ctypes.c_void_p
    far = [vp((i + 1) << 40) for i in range(10)]  # 1 TiB apart: no overlap at these sizes
    M = 1 << 29
    bad = _lib.FA_ERR_INVALID_ARG
    assert L.fa_bwd_workspace_size(1, 1, M, M, 16) > 0
    assert L.fa_bwd_workspace_size(1, 1, M + 1, 16, 16) == 0
    assert L.fa_bwd_workspace_size(1, 1, 16, M + 1, 16) == 0
    assert L.fa_bwd_varlen_workspace_size(1, 1, M + 1, 16, 16) == 0
    fwd = lambda nq, nk: L.fa_fwd(*far[:5], 1, 1, nq, nk, 16, 0.25, 1, None)  # noqa: E731
    assert fwd(M + 1, 16) == bad
    assert fwd(16, M + 1) == bad
    assert fwd((1 << 31) - 1, 16) == bad
    reaches_device(lambda: fwd(M, M))
    assert L.fa_fwd_window(*far[:5], 1, 1, M + 1, 16, 16, 0.25, 0, -1, -1, 0, None, 0, None) == bad
    assert L.fa_bwd(*far[:9], 1, 1, 16, M + 1, 16, 0.25, 1, far[9], 1 << 20, None) == bad
    varlen = lambda tq, tk, mq, mk: L.fa_fwd_varlen(*far[:7], 1, 1, tq, tk, mq, mk, 16, 0.25, 1, None)  # noqa: E731
    assert varlen(M + 1, 16, 16, 16) == bad
    assert varlen(16, M + 1, 16, 16) == bad
    assert varlen(16, 16, M + 1, 16) == bad
    assert varlen(16, 16, 16, M + 1) == bad
    reaches_device(lambda: varlen(M, M, M, M))
    fp8 = lambda nq, nk, ldv: L.fa_fwd_fp8(*far[:3], ldv, *far[3:8], 1, 1, nq, nk, 64, 0.125, 1, None)  # noqa: E731
    assert fp8(M + 1, 16, 16) == bad
    assert fp8(16, M + 16, M + 16) == bad
    assert L.fa_quantize_e4m3_transposed(far[0], 1, 1, M + 1, 64, M + 16, *far[1:4], None) == bad
    assert L.fa_quantize_qkv_e4m3(*far[:3], 1, 1, M + 1, 16, 64, *far[3:6], 16, *far[6:8], None) == bad
    assert L.fa_quantize_qkv_e4m3(*far[:3], 1, 1, 16, M + 1, 64, *far[3:6], M + 16, *far[6:8], None) == bad
