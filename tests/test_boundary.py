"""The C ABI on the host: the library builds for sm_103a, loads, exports every
function include/fa.h declares, and rejects invalid arguments with the documented
status before any CUDA work.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")

OK, INVALID, UNSUPPORTED, MISALIGNED = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    from exact_io_aware_22_gb300 import build
    import exact_io_aware_22_gb300 as fa
    path = build.build()
    return fa.load_library(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_status_string",
              "fa_device_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in fa.h but not exported"


def test_status_strings(lib):
    for code in range(6):
        s = lib.fa_status_string(code)
        assert s and s.startswith(b"FA_")


A16 = 0x10000  # fake, 16-byte aligned device addresses (never dereferenced on rejection)


def fwd(lib, **kw):
    a = dict(Q=A16, K=2 * A16, V=3 * A16, O=4 * A16, L=5 * A16, B=1, H=1, N=128, d=64,
             causal=0, scale=0.125, dtype=0)
    a.update(kw)
    return lib.fa_fwd(*(ctypes.c_void_p(a[k]) for k in ("Q", "K", "V", "O", "L")), a["B"],
                      a["H"], a["N"], a["d"], a["causal"], a["scale"], a["dtype"], None)


def bwd(lib, **kw):
    a = dict(Q=A16, K=2 * A16, V=3 * A16, O=4 * A16, dO=5 * A16, L=6 * A16, dQ=7 * A16,
             dK=8 * A16, dV=9 * A16, ws=10 * A16, ws_bytes=1 << 20, B=1, H=1, N=128, d=64,
             causal=1, scale=0.125, dtype=1)
    a.update(kw)
    ptrs = [ctypes.c_void_p(a[k]) for k in ("Q", "K", "V", "O", "dO", "L", "dQ", "dK", "dV", "ws")]
    return lib.fa_bwd(*ptrs, a["ws_bytes"], a["B"], a["H"], a["N"], a["d"], a["causal"],
                      a["scale"], a["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=48), UNSUPPORTED), (dict(d=256), UNSUPPORTED), (dict(d=16), UNSUPPORTED),
    (dict(dtype=2), UNSUPPORTED), (dict(dtype=-1), UNSUPPORTED),
    (dict(B=0), INVALID), (dict(H=0), INVALID), (dict(N=0), INVALID), (dict(N=-5), INVALID),
    (dict(scale=0.0), INVALID), (dict(scale=-0.1), INVALID), (dict(scale=float("nan")), INVALID),
    (dict(scale=float("inf")), INVALID), (dict(causal=2), INVALID),
    (dict(Q=0), INVALID), (dict(O=0), INVALID), (dict(L=0), INVALID),
    (dict(Q=A16 + 8), MISALIGNED), (dict(V=3 * A16 + 2), MISALIGNED), (dict(O=4 * A16 + 4), MISALIGNED),
    (dict(L=5 * A16 + 2), MISALIGNED),
    (dict(O=A16 + 64), INVALID),                      # output overlaps Q
    (dict(L=2 * A16 + 4), INVALID),                   # L inside K
])
def test_fwd_rejects(lib, kw, code):
    assert fwd(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), UNSUPPORTED), (dict(dtype=7), UNSUPPORTED),
    (dict(N=0), INVALID), (dict(scale=-1.0), INVALID),
    (dict(dQ=0), INVALID), (dict(L=0), INVALID), (dict(dO=0), INVALID),
    (dict(dK=8 * A16 + 8), MISALIGNED), (dict(ws=10 * A16 + 4), MISALIGNED),
    (dict(ws_bytes=16), INVALID),                     # workspace too small
    (dict(dK=7 * A16 + 16), INVALID),                 # dK overlaps dQ
    (dict(dV=A16), INVALID),                          # dV aliases Q
])
def test_bwd_rejects(lib, kw, code):
    assert bwd(lib, **kw) == code


M1 = 0x100000   # fake buffers 1 MiB apart: the 8-head tensors here are 128 KiB


def fwd_gqa(lib, Hkv, **kw):
    a = dict(Q=M1, K=2 * M1, V=3 * M1, O=4 * M1, L=5 * M1, B=1, H=8, N=128, d=64,
             causal=1, scale=0.125, dtype=1)
    a.update(kw)
    return lib.fa_fwd_gqa(*(ctypes.c_void_p(a[k]) for k in ("Q", "K", "V", "O", "L")), a["B"],
                          a["H"], Hkv, a["N"], a["d"], a["causal"], a["scale"], a["dtype"], None)


def bwd_gqa(lib, Hkv, **kw):
    a = dict(Q=M1, K=2 * M1, V=3 * M1, O=4 * M1, dO=5 * M1, L=6 * M1, dQ=7 * M1,
             dK=8 * M1, dV=9 * M1, ws=10 * M1, ws_bytes=1 << 20, B=1, H=8, N=128, d=64,
             causal=1, scale=0.125, dtype=1)
    a.update(kw)
    ptrs = [ctypes.c_void_p(a[k]) for k in ("Q", "K", "V", "O", "dO", "L", "dQ", "dK", "dV", "ws")]
    return lib.fa_bwd_gqa(*ptrs, a["ws_bytes"], a["B"], a["H"], Hkv, a["N"], a["d"], a["causal"],
                          a["scale"], a["dtype"], None)


@pytest.mark.parametrize("Hkv", [0, -1, 9, 3, 5])
def test_gqa_rejects_head_counts(lib, Hkv):
    # K/V heads must divide the 8 query heads
    assert fwd_gqa(lib, Hkv) == INVALID
    assert bwd_gqa(lib, Hkv) == INVALID


def test_gqa_rejects_like_mha(lib):
    assert fwd_gqa(lib, 2, d=48) == UNSUPPORTED
    assert fwd_gqa(lib, 2, K=2 * M1 + 8) == MISALIGNED
    # with 2 K/V heads K spans 2*128*64*2 = 32 KiB: an O that starts 16 KiB in overlaps it,
    # one that starts 32 KiB in does not reach Q, K or V (its 128 KiB end before 3 * M1)
    assert fwd_gqa(lib, 2, O=2 * M1 + 16384) == INVALID
    assert bwd_gqa(lib, 2, dK=2 * M1 + 16384) == INVALID      # dK overlaps K
    assert bwd_gqa(lib, 2, dK=7 * M1 + 65536) == INVALID      # dK inside dQ (128 KiB)
    assert bwd_gqa(lib, 4, ws_bytes=16) == INVALID


@pytest.mark.parametrize("window", [0, -1, -128])
def test_sliding_window_rejects_empty_windows(lib, window):
    a = [ctypes.c_void_p(M1 * i) for i in range(1, 6)]
    assert lib.fa_fwd_swa(*a, 1, 8, 2, 128, 64, window, 0.125, 1, None) == INVALID
    b = [ctypes.c_void_p(M1 * i) for i in range(1, 11)]
    assert lib.fa_bwd_swa(*b, 1 << 20, 1, 8, 2, 128, 64, window, 0.125, 1, None) == INVALID


def test_sliding_window_checks_heads(lib):
    a = [ctypes.c_void_p(M1 * i) for i in range(1, 6)]
    assert lib.fa_fwd_swa(*a, 1, 8, 3, 128, 64, 16, 0.125, 1, None) == INVALID
    assert lib.fa_fwd_swa(*a, 1, 8, 2, 128, 48, 16, 0.125, 1, None) == UNSUPPORTED


def fwd_varlen(lib, **kw):
    a = dict(Q=M1, K=2 * M1, V=3 * M1, O=4 * M1, L=5 * M1, cu=6 * M1, B=2, total=300,
             max_len=200, H=4, Hkv=2, d=64, causal=1, window=0, scale=0.125, dtype=1)
    a.update(kw)
    ptrs = [ctypes.c_void_p(a[k]) for k in ("Q", "K", "V", "O", "L", "cu")]
    return lib.fa_fwd_varlen(*ptrs, a["B"], a["total"], a["max_len"], a["H"], a["Hkv"], a["d"],
                             a["causal"], a["window"], a["scale"], a["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(cu=0), INVALID), (dict(total=0), INVALID), (dict(window=-1), INVALID),
    (dict(window=16, causal=0), INVALID), (dict(cu=6 * M1 + 2), MISALIGNED),
    (dict(Hkv=3), INVALID), (dict(max_len=0), INVALID), (dict(d=48), UNSUPPORTED),
    (dict(O=M1 + 4096), INVALID),                     # O inside Q (300 x 4 x 64 x 2 bytes)
])
def test_varlen_rejects(lib, kw, code):
    assert fwd_varlen(lib, **kw) == code


def test_varlen_workspace_size(lib):
    assert lib.fa_bwd_varlen_workspace_size(2, 200, 4, 64) == lib.fa_bwd_workspace_size(
        2, 4, 200, 64, 1)
    assert lib.fa_bwd_varlen_workspace_size(2, 0, 4, 64) == 0


def test_workspace_size(lib):
    f = lib.fa_bwd_workspace_size
    # D and L*log2(e), fp32, padded to 128-row blocks
    assert f(1, 1, 128, 64, 0) == 2 * 128 * 4
    assert f(4, 8, 1000, 32, 1) == 2 * 32 * 1024 * 4
    assert f(1, 32, 8192, 128, 1) == 2 * 32 * 8192 * 4
    assert f(2, 3, 1000, 128, 0) == 2 * 6 * 1024 * 4
    assert f(1, 1, 1, 32, 1) == 2 * 128 * 4
    assert f(1, 1, 128, 48, 0) == 0 and f(0, 1, 128, 64, 0) == 0


def test_binding_refuses_without_library(tmp_path):
    import exact_io_aware_22_gb300 as fa
    with pytest.raises(RuntimeError, match="not built"):
        fa.load_library(str(tmp_path / "missing.so"))


def decode(lib, **kw):
    a = dict(Q=M1, K=2 * M1, V=3 * M1, lens=4 * M1, O=5 * M1, L=6 * M1, ws=0, ws_bytes=0, B=2,
             H=8, Hkv=2, Nmax=300, d=64, scale=0.125, dtype=1)
    a.update(kw)
    ptrs = [ctypes.c_void_p(a[k]) for k in ("Q", "K", "V", "lens", "O", "L", "ws")]
    return lib.fa_decode(*ptrs, a["ws_bytes"], a["B"], a["H"], a["Hkv"], a["Nmax"], a["d"],
                         a["scale"], a["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(Q=0), INVALID), (dict(lens=0), INVALID), (dict(L=0), INVALID),
    (dict(B=0), INVALID), (dict(Nmax=0), INVALID), (dict(Hkv=3), INVALID),
    (dict(Hkv=0), INVALID), (dict(scale=0.0), INVALID), (dict(scale=float("nan")), INVALID),
    (dict(d=48), UNSUPPORTED), (dict(dtype=7), UNSUPPORTED), (dict(Nmax=(1 << 30) + 1), UNSUPPORTED),
    (dict(K=2 * M1 + 8), MISALIGNED), (dict(lens=4 * M1 + 2), MISALIGNED),
    (dict(O=M1 + 512), INVALID),                        # O inside Q (2 x 8 x 64 x 2 bytes)
    (dict(O=3 * M1 + 4096), INVALID),                   # O inside the V cache
    (dict(ws=8 * M1, ws_bytes=16), INVALID),            # workspace too small
    (dict(ws=5 * M1 + 64, ws_bytes=1 << 19), INVALID),  # workspace over O
])
def test_decode_rejects(lib, kw, code):
    assert decode(lib, **kw) == code


def test_decode_workspace_size(lib):
    f = lib.fa_decode_workspace_size
    # (B*H rows) x splits partial states of d + 4 floats.  16 x 8 K/V heads, 32768
    # cached keys: 128 CTA rows, 19 splits of 1728 keys (a multiple of 64)
    assert f(16, 32, 8, 32768, 128) == 16 * 32 * 19 * 132 * 4
    # one key: one split
    assert f(1, 1, 1, 1, 32) == 1 * 1 * 1 * 36 * 4
    assert f(0, 1, 1, 1, 32) == 0 and f(1, 4, 3, 10, 64) == 0 and f(1, 1, 1, 10, 48) == 0


def fwd_fp8(lib, **kw):
    a = dict(Q=M1, K=2 * M1, V=3 * M1, O=4 * M1, L=5 * M1, B=1, H=4, Hkv=2, N=256, d=128,
             causal=1, scale=0.088, qs=0.01, ks=0.01, vs=0.01)
    a.update(kw)
    ptrs = [ctypes.c_void_p(a[k]) for k in ("Q", "K", "V", "O", "L")]
    return lib.fa_fwd_fp8(*ptrs, a["B"], a["H"], a["Hkv"], a["N"], a["d"], a["causal"],
                          a["scale"], a["qs"], a["ks"], a["vs"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=64), UNSUPPORTED), (dict(N=200), UNSUPPORTED), (dict(Hkv=3), INVALID),
    (dict(qs=0.0), INVALID), (dict(vs=float("inf")), INVALID), (dict(ks=-1.0), INVALID),
    (dict(Q=0), INVALID), (dict(L=0), INVALID), (dict(B=0), INVALID),
    (dict(K=2 * M1 + 8), MISALIGNED), (dict(L=5 * M1 + 2), MISALIGNED),
    (dict(O=M1 + 4096), INVALID),                       # O over Q8 (4 x 256 x 128 bytes)
])
def test_fwd_fp8_rejects(lib, kw, code):
    assert fwd_fp8(lib, **kw) == code


@pytest.mark.parametrize("args,code", [
    ((0, 1, 1, 1.0, 0), INVALID), ((1, 0, 1, 1.0, 0), INVALID), ((1, 1, 1, 0.0, 0), INVALID),
    ((1, 1, 1, 1.0, 2), INVALID), ((70000, 4, 4, 1.0, 1), UNSUPPORTED),
])
def test_quantize_rejects(lib, args, code):
    mats, rows, cols, inv, tr = args
    assert lib.fa_quantize_fp8(ctypes.c_void_p(M1), ctypes.c_void_p(8 * M1), mats, rows, cols,
                               inv, tr, 1, None) == code
    assert lib.fa_quantize_fp8(ctypes.c_void_p(M1 + 1), ctypes.c_void_p(8 * M1), 1, 4, 4, 1.0,
                               0, 1, None) == MISALIGNED
    assert lib.fa_quantize_fp8(ctypes.c_void_p(M1), ctypes.c_void_p(M1 + 8), 1, 4, 4, 1.0,
                               0, 1, None) == INVALID
    assert lib.fa_quantize_fp8(ctypes.c_void_p(M1), ctypes.c_void_p(8 * M1), 1, 4, 4, 1.0,
                               0, 7, None) == UNSUPPORTED


def test_decode_fp8_rejects(lib):
    a = [ctypes.c_void_p(M1 * i) for i in (1, 2, 3, 4, 5, 6)]
    ws = ctypes.c_void_p(0)
    # d = 64: unsupported for E4M3 caches; non-positive descale factors; bad heads
    assert lib.fa_decode_fp8(*a, ws, 0, 2, 8, 2, 300, 64, 0.125, 0.01, 0.01, 1, None) == UNSUPPORTED
    assert lib.fa_decode_fp8(*a, ws, 0, 2, 8, 2, 300, 128, 0.125, 0.0, 0.01, 1, None) == INVALID
    assert lib.fa_decode_fp8(*a, ws, 0, 2, 8, 2, 300, 128, 0.125, 0.01, -1.0, 1, None) == INVALID
    assert lib.fa_decode_fp8(*a, ws, 0, 2, 8, 3, 300, 128, 0.125, 0.01, 0.01, 1, None) == INVALID
    b = list(a)
    b[1] = ctypes.c_void_p(2 * M1 + 8)
    assert lib.fa_decode_fp8(*b, ws, 0, 2, 8, 2, 300, 128, 0.125, 0.01, 0.01, 1, None) == MISALIGNED


def test_trace_kind_names_and_read_rejects(lib):
    # the per-kernel trace kinds of include/fa.h, in order; none past the last
    names = [lib.fa_trace_kind_name(k) for k in range(7)]
    assert names == [b"fwd_kernel", b"bwd_pre_kernel", b"bwd_dkdv_kernel", b"bwd_dq_kernel",
                     b"decode_split_kernel", b"decode_merge_kernel", b"fwd_fp8_kernel"]
    assert lib.fa_trace_kind_name(7) is None and lib.fa_trace_kind_name(-1) is None
    t, n = ctypes.c_double(), ctypes.c_longlong()
    assert lib.fa_trace_read(7, ctypes.byref(t), ctypes.byref(n)) == INVALID
    assert lib.fa_trace_read(-1, ctypes.byref(t), ctypes.byref(n)) == INVALID
    assert lib.fa_trace_read(0, None, ctypes.byref(n)) == INVALID
    assert lib.fa_trace_read(0, ctypes.byref(t), None) == INVALID


def test_wait_limit_setter(lib):
    # any value is accepted (0 restores the default); no CUDA call is made
    assert lib.fa_set_wait_limit_ns(1_000_000) == OK
    assert lib.fa_set_wait_limit_ns(0) == OK
