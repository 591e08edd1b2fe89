"""The C-ABI library builds, loads and exports every entry point include/fa.h
declares; host-side argument checks return their documented codes without
touching a GPU (CPU only: no compute call is made)."""
import ctypes
import math
import os
import re
import shutil

import pytest

import transformer_attention_flashattention_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|const char\s*\*)\s*(fa_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from transformer_attention_flashattention_gb300 import _build
    _build.build()
    return fa.load_library()


def test_header_declares_the_boundary():
    assert _declared() == sorted(["fa_fwd", "fa_quantize_fp8", "fa_fwd_fp8", "fa_strerror",
                                  "fa_last_device_status", "fa_debug_inject_stall", "fa_version",
                                  "fa_decode", "fa_decode_workspace_size", "fa_decode_noalloc",
                                  "fa_bwd", "fa_bwd_workspace_size", "fa_quantize_fp8_ex",
                                  "fa_fwd_host", "fa_fwd_host_workspace_size", "fa_fwd_fp8_host",
                                  "fa_fwd_fp8_host_workspace_size", "fa_build_id", "fa_fwd_2cta", "fa_quantize_fp8_qkv",
                                  "fa_fwd_naive", "fa_fwd_naive_workspace_size"])


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert sorted(fa.exported_symbols()) == _declared()


def test_library_carries_the_build_id_of_these_sources(lib, tmp_path, capsys):
    from transformer_attention_flashattention_gb300 import _build
    sid = _build.source_id()
    assert lib.fa_build_id().decode() == sid == _build.built_id()
    _build.build()                                  # up to date: nothing is compiled
    assert "up to date" in capsys.readouterr().out
    # a library file carrying another id is stale; one with no id at all too
    other = tmp_path / "libfa.so"
    other.write_bytes(b"\x7fELF..." + _build.BUILD_ID_TAG + b"0123456789abcdef" + b"\0")
    assert _build.built_id(str(other)) == "0123456789abcdef" != sid
    other.write_bytes(b"\x7fELF...")
    assert _build.built_id(str(other)) is None


def test_strerror_and_version(lib):
    for code in range(-9, 1):
        assert lib.fa_strerror(code)
    assert lib.fa_strerror(-99) == b"unknown status"
    assert lib.fa_version() >= 100


A = 0x10000          # a 16-byte aligned fake address; never dereferenced by these calls


@pytest.mark.parametrize("args,want", [
    ((0, A, A, A, 0, 1, 1, 128, 64, 0.125, 0, 1), fa.FA_ERR_NULL),
    ((A, A, A, 0, 0, 1, 1, 128, 64, 0.125, 0, 1), fa.FA_ERR_NULL),
    ((A, A, A, A, 0, 1, 1, 128, 96, 0.125, 0, 1), fa.FA_ERR_UNSUPPORTED),
    ((A, A, A, A, 0, 1, 1, 128, 64, 0.125, 0, 7), fa.FA_ERR_UNSUPPORTED),
    ((A, A, A, A, 0, 1, 1, 128, 64, 0.125, 2, 1), fa.FA_ERR_UNSUPPORTED),
    ((A, A, A, A, 0, 1, 1, 128, 64, float("nan"), 0, 1), fa.FA_ERR_UNSUPPORTED),
    ((A, A, A, A, 0, 1, 1, 128, 64, 0.0, 0, 1), fa.FA_ERR_UNSUPPORTED),
    ((A, A, A, A, 0, 1, 1, 128, 64, -0.125, 0, 1), fa.FA_ERR_UNSUPPORTED),
    ((A, A, A, A, 0, 0, 1, 128, 64, 0.125, 0, 1), fa.FA_ERR_SHAPE),
    ((A, A, A, A, 0, 1, 1, 0, 64, 0.125, 0, 1), fa.FA_ERR_SHAPE),
    ((A, A, A, A, 0, 1, -3, 128, 64, 0.125, 0, 1), fa.FA_ERR_SHAPE),
    ((A, A, A, A, 0, 65536, 65536, 65536, 64, 0.125, 0, 1), fa.FA_ERR_SHAPE),
    ((A + 8, A, A, A, 0, 1, 1, 128, 64, 0.125, 0, 1), fa.FA_ERR_ALIGN),
    ((A, A, A, A + 2, 0, 1, 1, 128, 64, 0.125, 0, 1), fa.FA_ERR_ALIGN),
    ((A, A, A, A, A + 2, 1, 1, 128, 64, 0.125, 0, 1), fa.FA_ERR_ALIGN),
])
def test_fwd_rejects_bad_arguments_on_the_host(lib, args, want):
    q, k, v, o, lse, B, H, N, d, scale, causal, dtype = args
    assert lib.fa_fwd(q or None, k or None, v or None, o or None, lse or None, B, H, N, d, scale,
                      causal, dtype, None) == want


@pytest.mark.parametrize("args,want", [
    ((0, A, A, A, 0, 1, 1, 1, 128, 64, 0.125, 0, 1, 0, 0, 0), fa.FA_ERR_NULL),
    ((A, A, A, A, 0, 1, 1, 17, 128, 64, 0.125, 0, 1, 0, 0, 0), fa.FA_ERR_SHAPE),    # N_q > 16
    ((A, A, A, A, 0, 1, 1, 4, 3, 64, 0.125, 0, 1, 0, 0, 0), fa.FA_ERR_SHAPE),       # N_q > N_k
    ((A, A, A, A, 0, 1, 1, 1, 128, 80, 0.125, 0, 1, 0, 0, 0), fa.FA_ERR_UNSUPPORTED),
    ((A, A, A, A, 0, 1, 1, 1, 128, 64, 0.125, 3, 1, 0, 0, 0), fa.FA_ERR_UNSUPPORTED),
    ((A, A, A, A, 0, 1, 1, 1, 128, 64, 0.125, 0, 1, 0, A + 16, 1024), fa.FA_ERR_ALIGN),
])
def test_decode_rejects_bad_arguments_on_the_host(lib, args, want):
    q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype, splits, ws, wsb = args
    assert lib.fa_decode(q or None, k or None, v or None, o or None, lse or None, B, H, Nq, Nk, d, scale,
                         causal, dtype, splits, ws or None, wsb, None) == want


@pytest.mark.parametrize("Nq,Nk,d,want", [
    (17, 128, 64, fa.FA_ERR_SHAPE),      # N_q > 16
    (4, 3, 64, fa.FA_ERR_SHAPE),         # N_q > N_k
    (0, 128, 64, fa.FA_ERR_SHAPE),
    (1, 128, 80, fa.FA_ERR_UNSUPPORTED),
])
def test_decode_noalloc_rejects_bad_shapes_on_the_host(lib, Nq, Nk, d, want):
    assert lib.fa_decode_noalloc(A, A, A, A, None, 1, 1, Nq, Nk, d, 0.125, 0, 1, 0, None) == want


def test_decode_noalloc_checks_arguments_before_the_scratch_limit(lib):
    """With a num_splits far past the scratch area, a call that is also malformed reports
    what fa_decode would report, not FA_ERR_WORKSPACE."""
    call = lambda q=A, o=A, lse=0, scale=0.125, causal=0, dtype=1: lib.fa_decode_noalloc(
        q or None, A, A, o or None, lse or None, 1, 1, 1, 128, 64, scale, causal, dtype, 1 << 20, None)
    assert call(q=0) == fa.FA_ERR_NULL
    assert call(o=0) == fa.FA_ERR_NULL
    assert call(dtype=9) == fa.FA_ERR_UNSUPPORTED
    assert call(causal=2) == fa.FA_ERR_UNSUPPORTED
    assert call(scale=float("inf")) == fa.FA_ERR_UNSUPPORTED
    assert call(scale=0.0) == fa.FA_ERR_UNSUPPORTED
    assert call(q=A + 8) == fa.FA_ERR_ALIGN
    assert call(lse=A + 2) == fa.FA_ERR_ALIGN
    # fa_decode checks the shape before the scale
    assert lib.fa_decode_noalloc(A, A, A, A, None, 1, 1, 0, 128, 64, 0.0, 0, 1, 1 << 20, None) == fa.FA_ERR_SHAPE


def test_bwd_rejects_bad_arguments_on_the_host(lib):
    args = [A] * 9
    ws = 0x100000
    call = lambda a, B=1, H=1, N=128, d=64, scale=0.125, causal=0, dtype=1, wsp=ws, wsb=1 << 20: lib.fa_bwd(
        *a, B, H, N, d, scale, causal, dtype, wsp, wsb, None)
    assert call([0] + args[1:]) == fa.FA_ERR_NULL
    assert call(args, d=96) == fa.FA_ERR_UNSUPPORTED
    assert call(args, causal=2) == fa.FA_ERR_UNSUPPORTED
    assert call(args, scale=-1.0) == fa.FA_ERR_UNSUPPORTED
    assert call(args, N=0) == fa.FA_ERR_SHAPE
    assert call(args, wsp=ws + 16) == fa.FA_ERR_ALIGN
    assert call(args, wsb=512) == fa.FA_ERR_WORKSPACE     # 1 x 1 x 128 needs 1024
    n = ctypes.c_ulonglong(0)
    assert lib.fa_bwd_workspace_size(2, 3, 200, 64, ctypes.byref(n)) == fa.FA_OK and n.value == 2 * 2 * 3 * 256 * 4


def test_quantize_ex_rejects_bad_options_on_the_host(lib):
    call = lambda had=1, lo=0, hi=0, ph=0, d=128: lib.fa_quantize_fp8_ex(A, A, A, 1, 1, 64, d, had, lo, hi, ph, 0, None)
    assert call(had=0, lo=1) == fa.FA_ERR_UNSUPPORTED          # signs without the rotation
    assert call(d=64, hi=1) == fa.FA_ERR_UNSUPPORTED           # sign bit past d
    assert call(ph=2) == fa.FA_ERR_UNSUPPORTED
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED


def test_fwd_host_rejects_bad_arguments_on_the_host(lib):
    n = ctypes.c_ulonglong(0)
    assert lib.fa_fwd_host_workspace_size(2, 3, 100, 64, ctypes.byref(n)) == fa.FA_OK
    assert n.value == 4 * ((2 * 2 * 3 * 100 * 64 + 255) // 256 * 256) + (4 * 2 * 3 * 100 + 255) // 256 * 256
    ws = 0x100000
    call = lambda wsp=ws, wsb=1 << 30, chunks=0, dtype=1, d=64: lib.fa_fwd_host(
        A, A, A, A, None, 2, 3, 100, d, 0.125, 0, dtype, chunks, wsp, wsb, None)
    assert call(wsb=1024) == fa.FA_ERR_WORKSPACE
    assert call(wsp=ws + 64) == fa.FA_ERR_ALIGN
    assert call(chunks=-1) == fa.FA_ERR_UNSUPPORTED
    assert call(dtype=5) == fa.FA_ERR_UNSUPPORTED
    assert call(d=80) == fa.FA_ERR_UNSUPPORTED


def test_fwd_fp8_host_rejects_bad_arguments_on_the_host(lib):
    n = ctypes.c_ulonglong(0)
    assert lib.fa_fwd_fp8_host_workspace_size(2, 3, 96, 128, ctypes.byref(n)) == fa.FA_OK
    r = lambda x: (x + 255) // 256 * 256
    e = 2 * 3 * 96 * 128
    assert n.value == 4 * r(2 * e) + 3 * r(e) + 3 * r(4 * 2 * 3 * 2) + r(4 * 2 * 3 * 96)
    assert lib.fa_fwd_fp8_host_workspace_size(2, 3, 96, 64, ctypes.byref(n)) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_fwd_fp8_host_workspace_size(2, 3, 100, 128, ctypes.byref(n)) == fa.FA_ERR_SHAPE
    ws = 0x100000
    call = lambda wsp=ws, wsb=1 << 30, chunks=0, had=1, causal=0, N=96, q=A: lib.fa_fwd_fp8_host(
        q or None, A, A, A, None, 2, 3, N, 128, 0.125, causal, had, chunks, wsp, wsb, None)
    assert call(q=0) == fa.FA_ERR_NULL
    assert call(wsb=1024) == fa.FA_ERR_WORKSPACE
    assert call(wsp=ws + 64) == fa.FA_ERR_ALIGN
    assert call(chunks=-1) == fa.FA_ERR_UNSUPPORTED
    assert call(had=2) == fa.FA_ERR_UNSUPPORTED
    assert call(causal=3) == fa.FA_ERR_UNSUPPORTED
    assert call(N=100) == fa.FA_ERR_SHAPE


def test_fwd_2cta_rejects_bad_arguments_on_the_host(lib):
    call = lambda q=A, d=128, dtype=1, causal=0, scale=0.125, N=128: lib.fa_fwd_2cta(
        q or None, A, A, A, None, 1, 1, N, d, scale, causal, dtype, None)
    assert call(q=0) == fa.FA_ERR_NULL
    assert call(d=64) == fa.FA_ERR_UNSUPPORTED          # head dim 128 only
    assert call(dtype=3) == fa.FA_ERR_UNSUPPORTED
    assert call(causal=2) == fa.FA_ERR_UNSUPPORTED
    assert call(scale=-1.0) == fa.FA_ERR_UNSUPPORTED
    assert call(N=0) == fa.FA_ERR_SHAPE
    assert call(q=A + 8) == fa.FA_ERR_ALIGN


def test_quantize_qkv_rejects_bad_arguments_on_the_host(lib):
    call = lambda q=A, had=1, N=128, d=128, vs=A: lib.fa_quantize_fp8_qkv(q or None, A, A, A, A, A, A, A, vs or None,
                                                                      1, 1, N, d, had, None)
    assert call(q=0) == fa.FA_ERR_NULL
    assert call(vs=0) == fa.FA_ERR_NULL
    assert call(had=2) == fa.FA_ERR_UNSUPPORTED
    assert call(d=80) == fa.FA_ERR_UNSUPPORTED
    assert call(N=100) == fa.FA_ERR_SHAPE               # V is written transposed: N % 16 == 0
    assert call(q=A + 8) == fa.FA_ERR_ALIGN
    assert call(vs=A + 2) == fa.FA_ERR_ALIGN


def test_fwd_naive_rejects_bad_arguments_on_the_host(lib):
    n = ctypes.c_ulonglong(0)
    # fp32 scores, rows rounded up to whole float4 vectors
    assert lib.fa_fwd_naive_workspace_size(2, 3, 130, 64, ctypes.byref(n)) == fa.FA_OK
    assert n.value == (2 * 3 * 130 * 132 * 4 + 255) // 256 * 256 + (32 << 20)
    assert lib.fa_fwd_naive_workspace_size(1, 1, 32768, 128, ctypes.byref(n)) == fa.FA_OK
    assert lib.fa_fwd_naive_workspace_size(1, 1, 32769, 128, ctypes.byref(n)) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_fwd_naive_workspace_size(1, 1, 128, 96, ctypes.byref(n)) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_fwd_naive_workspace_size(1 << 16, 1 << 10, 64, 64, ctypes.byref(n)) == fa.FA_ERR_SHAPE
    assert lib.fa_fwd_naive_workspace_size(1, 1, 128, 64, None) == fa.FA_ERR_NULL
    ws = 0x100000
    call = lambda q=A, wsp=ws, wsb=1 << 30, dtype=1, causal=0, scale=0.125, d=64, N=130: lib.fa_fwd_naive(
        q or None, A, A, A, None, 2, 3, N, d, scale, causal, dtype, wsp or None, wsb, None)
    assert call(q=0) == fa.FA_ERR_NULL
    assert call(wsp=0) == fa.FA_ERR_NULL
    assert call(wsb=1024) == fa.FA_ERR_WORKSPACE
    assert call(wsp=ws + 64) == fa.FA_ERR_ALIGN
    assert call(dtype=4) == fa.FA_ERR_UNSUPPORTED
    assert call(causal=2) == fa.FA_ERR_UNSUPPORTED
    assert call(scale=-1.0) == fa.FA_ERR_UNSUPPORTED
    assert call(d=80) == fa.FA_ERR_UNSUPPORTED
    assert call(N=40000) == fa.FA_ERR_UNSUPPORTED
