"""GB300 (sm_103a) attention forward: a thin ctypes binding over libfa.so.

Every step of the computation runs in the library's CUDA kernels; this module
only checks arguments, allocates outputs with torch (device memory and streams
are all torch is used for) and passes raw pointers through the C ABI declared
in ``include/fa.h``.  There is no fallback: if the library is missing or the
device is not an sm_103 GPU, calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

__all__ = [
    "FAError",
    "load_library",
    "library_path",
    "exported_symbols",
    "attention",
    "attention_host",
    "attention_2cta",
    "attention_fp8_host",
    "quantize_fp8",
    "quantize_fp8_qkv",
    "attention_fp8",
    "decode",
    "decode_noalloc",
    "attention_backward",
    "attention_naive",
    "DECODE_NOALLOC_SCRATCH_BYTES",
    "last_device_status",
    "inject_stall",
    "FA_OK",
    "FA_ERR_NULL",
    "FA_ERR_ALIGN",
    "FA_ERR_SHAPE",
    "FA_ERR_UNSUPPORTED",
    "FA_ERR_LAUNCH",
    "FA_ERR_DEVICE_TIMEOUT",
    "FA_ERR_ARCH",
    "FA_ERR_CUDA",
    "FA_ERR_WORKSPACE",
]

FA_OK = 0
FA_ERR_NULL = -1
FA_ERR_ALIGN = -2
FA_ERR_SHAPE = -3
FA_ERR_UNSUPPORTED = -4
FA_ERR_LAUNCH = -5
FA_ERR_DEVICE_TIMEOUT = -6
FA_ERR_ARCH = -7
FA_ERR_CUDA = -8
FA_ERR_WORKSPACE = -9

# Size of the static scratch area behind decode_noalloc (FA_DECODE_NOALLOC_SCRATCH_BYTES).
DECODE_NOALLOC_SCRATCH_BYTES = 8 << 20

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
_LIB: Optional[ctypes.CDLL] = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_SIGNATURES = {
    "fa_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _vp]),
    "fa_fwd_2cta": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _vp]),
    "fa_quantize_fp8": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp]),
    "fa_quantize_fp8_ex": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, ctypes.c_ulonglong, ctypes.c_ulonglong,
                                _i, _i, _vp]),
    "fa_fwd_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _vp, _vp, _i, _vp]),
    "fa_quantize_fp8_qkv": (_i, [_vp] * 9 + [_i, _i, _i, _i, _i, _vp]),
    "fa_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _i, _vp, ctypes.c_ulonglong, _vp]),
    "fa_decode_workspace_size": (_i, [_i, _i, _i, _i, _i, _i, ctypes.POINTER(ctypes.c_ulonglong)]),
    "fa_decode_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _i, _vp]),
    "fa_bwd": (_i, [_vp] * 9 + [_i, _i, _i, _i, _f, _i, _i, _vp, ctypes.c_ulonglong, _vp]),
    "fa_bwd_workspace_size": (_i, [_i, _i, _i, _i, ctypes.POINTER(ctypes.c_ulonglong)]),
    "fa_fwd_naive": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _vp, ctypes.c_ulonglong, _vp]),
    "fa_fwd_naive_workspace_size": (_i, [_i, _i, _i, _i, ctypes.POINTER(ctypes.c_ulonglong)]),
    "fa_fwd_host": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _i, _vp, ctypes.c_ulonglong, _vp]),
    "fa_fwd_host_workspace_size": (_i, [_i, _i, _i, _i, ctypes.POINTER(ctypes.c_ulonglong)]),
    "fa_fwd_fp8_host": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _i, _vp, ctypes.c_ulonglong,
                             _vp]),
    "fa_fwd_fp8_host_workspace_size": (_i, [_i, _i, _i, _i, ctypes.POINTER(ctypes.c_ulonglong)]),
    "fa_strerror": (ctypes.c_char_p, [_i]),
    "fa_last_device_status": (_i, [_vp, ctypes.POINTER(ctypes.c_uint)]),
    "fa_debug_inject_stall": (_i, [_i, _i]),
    "fa_build_id": (ctypes.c_char_p, []),
    "fa_version": (_i, []),
}


class FAError(RuntimeError):
    """A non-zero status returned by the C ABI."""

    def __init__(self, status: int, where: str):
        self.status = status
        msg = _LIB.fa_strerror(status).decode() if _LIB is not None else str(status)
        super().__init__(f"{where}: {msg} (status {status})")


def library_path() -> str:
    return os.environ.get("FA_LIBRARY", os.path.join(_PKG_DIR, "libfa.so"))


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libfa.so (built by ``__graft_entry__.build()``) and declare its signatures."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libfa.so not found at {path}: build it with "
                           "`python -m transformer_attention_flashattention_gb300._build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    # the in-tree library must be built from the sources as they are now
    if path == library_path() and os.path.isdir(os.path.join(_PKG_DIR, "csrc")):
        from . import _build
        have, want = lib.fa_build_id().decode(), _build.source_id()
        if have != want:
            raise RuntimeError(f"libfa.so carries build id {have}, but the sources are {want}: rebuild it "
                               "with `python -m transformer_attention_flashattention_gb300._build`")
    _LIB = lib
    return lib


def exported_symbols():
    return list(_SIGNATURES)


def _check(status: int, where: str) -> None:
    if status != FA_OK:
        raise FAError(status, where)


def _stream_handle(stream: Optional[torch.cuda.Stream], device: torch.device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


_DTYPES = {torch.float16: 0, torch.bfloat16: 1}


def _check_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor):
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError(f"q, k, v must share one [B, H, N, d] shape; got {tuple(q.shape)}, "
                         f"{tuple(k.shape)}, {tuple(v.shape)}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device != q.device or t.dtype != q.dtype:
            raise ValueError("q, k, v must share device and dtype")


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
              scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
              lse: Optional[torch.Tensor] = None, return_lse: bool = True,
              stream: Optional[torch.cuda.Stream] = None,
              check: bool = False) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """O = softmax(scale * Q K^T [+ causal mask]) V and the natural-log LSE.

    q, k, v: contiguous CUDA tensors [B, H, N, d], float16 or bfloat16, d in {64, 128}.
    Returns (O [B, H, N, d] of q's dtype, LSE [B, H, N] float32 or None).

    The kernel's pipeline waits are bounded.  One that gives up (a stalled or heavily
    preempted GPU) leaves O and LSE undefined while the call itself still succeeds;
    only the device status word records it.  ``check=True`` synchronises the stream
    after the launch and raises ``FAError(FA_ERR_DEVICE_TIMEOUT)`` if the word is set.
    """
    lib = load_library()
    _check_qkv(q, k, v)
    if q.dtype not in _DTYPES:
        raise ValueError(f"dtype must be float16 or bfloat16, got {q.dtype}")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    st = lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d, float(scale),
                    int(bool(causal)), _DTYPES[q.dtype], _stream_handle(stream, q.device))
    _check(st, "fa_fwd")
    if check:
        with torch.cuda.device(q.device):
            _check(lib.fa_last_device_status(_stream_handle(stream, q.device), None), "fa_fwd (device status)")
    return out, lse


def attention_2cta(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                   scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                   lse: Optional[torch.Tensor] = None, return_lse: bool = True,
                   stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """``attention`` computed by CTA pairs (``fa_fwd_2cta``; head dim 128 only)."""
    lib = load_library()
    _check_qkv(q, k, v)
    if q.dtype not in _DTYPES:
        raise ValueError(f"dtype must be float16 or bfloat16, got {q.dtype}")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    st = lib.fa_fwd_2cta(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d, float(scale),
                         int(bool(causal)), _DTYPES[q.dtype], _stream_handle(stream, q.device))
    _check(st, "fa_fwd_2cta")
    return out, lse


_HOST_WS = {}


def attention_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                   scale: Optional[float] = None, device: Optional[torch.device] = None,
                   stream: Optional[torch.cuda.Stream] = None, out: Optional[torch.Tensor] = None,
                   lse_out: Optional[torch.Tensor] = None, chunks: int = 0):
    """End-to-end call on HOST tensors through ``fa_fwd_host``: the library copies Q, K,
    V to the GPU, computes and copies O and LSE back, overlapping the copies of one chunk
    of heads with the computation of another.  Pinned host tensors let the copies run
    asynchronously.  Returns host tensors (``out``/``lse_out`` if given)."""
    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.is_cuda or t.dim() != 4 or t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor shaped and typed like q")
    if q.dtype not in _DTYPES:
        raise ValueError(f"dtype must be float16 or bfloat16, got {q.dtype}")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    pin = q.is_pinned()
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=pin)
    if lse_out is None:
        lse_out = torch.empty((B, H, N), dtype=torch.float32, pin_memory=pin)
    need = ctypes.c_ulonglong(0)
    _check(lib.fa_fwd_host_workspace_size(B, H, N, d, ctypes.byref(need)), "fa_fwd_host_workspace_size")
    ws = _HOST_WS.get(dev)
    if ws is None or ws.numel() < need.value:
        ws = torch.empty(need.value, device=dev, dtype=torch.uint8)
        _HOST_WS[dev] = ws
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        st = lib.fa_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse_out), B, H, N, d, float(scale),
                             int(bool(causal)), _DTYPES[q.dtype], int(chunks), _ptr(ws), ws.numel(),
                             s.cuda_stream)
    _check(st, "fa_fwd_host")
    s.synchronize()
    return out, lse_out


def attention_fp8_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                       scale: Optional[float] = None, hadamard: bool = True,
                       device: Optional[torch.device] = None, stream: Optional[torch.cuda.Stream] = None,
                       out: Optional[torch.Tensor] = None, lse_out: Optional[torch.Tensor] = None,
                       chunks: int = 0):
    """The FP8 mode end to end on bf16 HOST tensors through ``fa_fwd_fp8_host``: the
    library copies Q, K, V to the GPU, quantises them there (Q and K rotated when
    ``hadamard``), runs the E4M3 forward and copies the bf16 O and the LSE back, chunk
    by chunk.  Returns host tensors (``out``/``lse_out`` if given)."""
    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.is_cuda or t.dim() != 4 or t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bfloat16 host tensor shaped like q")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    pin = q.is_pinned()
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin)
    if lse_out is None:
        lse_out = torch.empty((B, H, N), dtype=torch.float32, pin_memory=pin)
    need = ctypes.c_ulonglong(0)
    _check(lib.fa_fwd_fp8_host_workspace_size(B, H, N, d, ctypes.byref(need)), "fa_fwd_fp8_host_workspace_size")
    ws = _HOST_WS.get(dev)
    if ws is None or ws.numel() < need.value:
        ws = torch.empty(need.value, device=dev, dtype=torch.uint8)
        _HOST_WS[dev] = ws
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        st = lib.fa_fwd_fp8_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse_out), B, H, N, d, float(scale),
                                 int(bool(causal)), int(bool(hadamard)), int(chunks), _ptr(ws), ws.numel(),
                                 s.cuda_stream)
    _check(st, "fa_fwd_fp8_host")
    s.synchronize()
    return out, lse_out


def quantize_fp8(x: torch.Tensor, hadamard: bool = False, transpose_out: bool = False,
                 stream: Optional[torch.cuda.Stream] = None, sign_flips: int = 0,
                 per_head: bool = False,
                 out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Block absmax E4M3 quantisation of bf16 ``x [B,H,N,d]`` (optionally Hadamard-rotated).

    ``sign_flips`` (an integer bit mask, bit c negates coordinate c before the
    rotation) randomises the rotation; ``per_head`` takes one scale per (b, h).
    ``out`` = (codes, scales) to write into instead of new tensors.
    Returns (codes as uint8 [B,H,N,d] or [B,H,d,N] when transposed, scales fp32 [B,H,ceil(N/64)]).
    """
    lib = load_library()
    if x.dim() != 4 or not x.is_cuda or not x.is_contiguous() or x.dtype != torch.bfloat16:
        raise ValueError("x must be a contiguous CUDA bfloat16 tensor [B, H, N, d]")
    B, H, N, d = x.shape
    shape = (B, H, d, N) if transpose_out else (B, H, N, d)
    if out is not None:
        x8, sc = out
        if (tuple(x8.shape) != shape or x8.dtype != torch.uint8 or tuple(sc.shape) != (B, H, (N + 63) // 64)
                or sc.dtype != torch.float32 or not x8.is_contiguous() or not sc.is_contiguous()):
            raise ValueError("out must be (uint8 codes, float32 scales) shaped for x")
    else:
        x8 = torch.empty(shape, device=x.device, dtype=torch.uint8)
        sc = torch.empty((B, H, (N + 63) // 64), device=x.device, dtype=torch.float32)
    if sign_flips or per_head:
        if not 0 <= int(sign_flips) < (1 << 128):
            raise ValueError("sign_flips must be a 128-bit mask")
        st = lib.fa_quantize_fp8_ex(_ptr(x), _ptr(x8), _ptr(sc), B, H, N, d, int(bool(hadamard)),
                                    int(sign_flips) & ((1 << 64) - 1), int(sign_flips) >> 64, int(bool(per_head)),
                                    int(bool(transpose_out)), _stream_handle(stream, x.device))
        _check(st, "fa_quantize_fp8_ex")
        return x8, sc
    st = lib.fa_quantize_fp8(_ptr(x), _ptr(x8), _ptr(sc), B, H, N, d, int(bool(hadamard)),
                             int(bool(transpose_out)), _stream_handle(stream, x.device))
    _check(st, "fa_quantize_fp8")
    return x8, sc


def quantize_fp8_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, hadamard: bool = True,
                     stream: Optional[torch.cuda.Stream] = None, out=None):
    """The FP8 prologue in one launch (``fa_quantize_fp8_qkv``): Q and K quantised (rotated
    when ``hadamard``), V quantised and transposed.  ``out`` = (q8, k8, v8t, qs, ks, vs) to
    write into.  Returns (q8, k8, v8t, q_scale, k_scale, v_scale)."""
    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dim() != 4 or not t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16 or t.shape != q.shape:
            raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor shaped like q")
    B, H, N, d = q.shape
    nb = (N + 63) // 64
    if out is None:
        out = (torch.empty((B, H, N, d), device=q.device, dtype=torch.uint8),
               torch.empty((B, H, N, d), device=q.device, dtype=torch.uint8),
               torch.empty((B, H, d, N), device=q.device, dtype=torch.uint8),
               *(torch.empty((B, H, nb), device=q.device, dtype=torch.float32) for _ in range(3)))
    q8, k8, v8t, qs, ks, vs = out
    st = lib.fa_quantize_fp8_qkv(_ptr(q), _ptr(k), _ptr(v), _ptr(q8), _ptr(k8), _ptr(v8t), _ptr(qs), _ptr(ks),
                                 _ptr(vs), B, H, N, d, int(bool(hadamard)), _stream_handle(stream, q.device))
    _check(st, "fa_quantize_fp8_qkv")
    return q8, k8, v8t, qs, ks, vs


def attention_fp8(q8: torch.Tensor, k8: torch.Tensor, v8t: torch.Tensor, q_scale: torch.Tensor,
                  k_scale: torch.Tensor, v_scale: torch.Tensor, causal: bool = False,
                  scale: Optional[float] = None, hadamard: bool = False,
                  out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                  return_lse: bool = True, stream: Optional[torch.cuda.Stream] = None):
    """Attention forward from E4M3 codes (see ``quantize_fp8``); bf16 output."""
    lib = load_library()
    B, H, N, d = q8.shape
    if k8.shape != q8.shape or v8t.shape != (B, H, d, N):
        raise ValueError("k8 must be [B,H,N,d] and v8t [B,H,d,N]")
    for t in (q8, k8, v8t, q_scale, k_scale, v_scale):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all inputs must be contiguous CUDA tensors")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, N, d), device=q8.device, dtype=torch.bfloat16)
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), device=q8.device, dtype=torch.float32)
    st = lib.fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8t), _ptr(out), _ptr(lse), B, H, N, d, float(scale),
                        int(bool(causal)), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
                        int(bool(hadamard)), _stream_handle(stream, q8.device))
    _check(st, "fa_fwd_fp8")
    return out, lse


def decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
           scale: Optional[float] = None, num_splits: int = 0, out: Optional[torch.Tensor] = None,
           lse: Optional[torch.Tensor] = None, return_lse: bool = True,
           workspace: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
    """Attention of q [B,H,N_q,d] (N_q <= 16) against a key cache k, v [B,H,N_k,d].

    Split-KV on the CUDA cores with a log-sum-exp merge; a scratch workspace is
    allocated with torch unless one is given.  Returns (O, LSE).
    """
    lib = load_library()
    B, H, Nq, d = q.shape
    if k.dim() != 4 or k.shape != v.shape or k.shape[:2] != (B, H) or k.shape[3] != d:
        raise ValueError(f"k, v must be [B, H, N_k, d] matching q; got {tuple(k.shape)}, {tuple(v.shape)}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype:
            raise ValueError(f"{name} must be a contiguous CUDA tensor of q's dtype")
    if q.dtype not in _DTYPES:
        raise ValueError(f"dtype must be float16 or bfloat16, got {q.dtype}")
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = ctypes.c_ulonglong(0)
    with torch.cuda.device(q.device):
        _check(lib.fa_decode_workspace_size(B, H, Nq, Nk, d, int(num_splits), ctypes.byref(need)),
               "fa_decode_workspace_size")
    if workspace is None and need.value > 0:
        workspace = torch.empty(need.value, device=q.device, dtype=torch.uint8)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.fa_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq, Nk, d, float(scale),
                       int(bool(causal)), _DTYPES[q.dtype], int(num_splits), _ptr(workspace), ws_bytes,
                       _stream_handle(stream, q.device))
    _check(st, "fa_decode")
    return out, lse


def decode_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                   scale: Optional[float] = None, num_splits: int = 0, out: Optional[torch.Tensor] = None,
                   lse: Optional[torch.Tensor] = None, return_lse: bool = True,
                   stream: Optional[torch.cuda.Stream] = None):
    """``decode`` through ``fa_decode_noalloc``: the split scratch is the library's
    static per-device area, so the C call allocates nothing (pass ``out`` and
    ``lse`` to keep this wrapper from allocating them).  Calls that can overlap on
    the GPU share that area and race; the first call on a device does a one-time
    address look-up and belongs outside stream capture.  Raises FAError
    (FA_ERR_WORKSPACE) when these sizes need more than DECODE_NOALLOC_SCRATCH_BYTES.
    """
    lib = load_library()
    B, H, Nq, d = q.shape
    if k.dim() != 4 or k.shape != v.shape or k.shape[:2] != (B, H) or k.shape[3] != d:
        raise ValueError(f"k, v must be [B, H, N_k, d] matching q; got {tuple(k.shape)}, {tuple(v.shape)}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype:
            raise ValueError(f"{name} must be a contiguous CUDA tensor of q's dtype")
    if q.dtype not in _DTYPES:
        raise ValueError(f"dtype must be float16 or bfloat16, got {q.dtype}")
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32)
    with torch.cuda.device(q.device):
        st = lib.fa_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq, Nk, d,
                                   float(scale), int(bool(causal)), _DTYPES[q.dtype], int(num_splits),
                                   _stream_handle(stream, q.device))
    if st == FA_ERR_WORKSPACE:
        raise FAError(st, f"fa_decode_noalloc (these sizes need more than the "
                          f"{DECODE_NOALLOC_SCRATCH_BYTES}-byte static scratch: lower num_splits or use decode)")
    _check(st, "fa_decode_noalloc")
    return out, lse


def attention_backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                       lse: torch.Tensor, dout: torch.Tensor, causal: bool = False,
                       scale: Optional[float] = None, dq: Optional[torch.Tensor] = None,
                       dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None):
    """(dQ, dK, dV) of ``attention``'s output for the upstream gradient ``dout``.

    ``o`` and ``lse`` are ``attention``'s outputs for the same inputs, scale and
    mask.  A scratch workspace is allocated with torch unless one is given.
    """
    lib = load_library()
    _check_qkv(q, k, v)
    for name, t in (("o", o), ("dout", dout)):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor shaped and typed like q")
    B, H, N, d = q.shape
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = ctypes.c_ulonglong(0)
    _check(lib.fa_bwd_workspace_size(B, H, N, d, ctypes.byref(need)), "fa_bwd_workspace_size")
    if workspace is None:
        workspace = torch.empty(max(need.value, 256), device=q.device, dtype=torch.uint8)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    with torch.cuda.device(q.device):
        st = lib.fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                        B, H, N, d, float(scale), int(bool(causal)), _DTYPES[q.dtype], _ptr(workspace),
                        workspace.numel() * workspace.element_size(), _stream_handle(stream, q.device))
    _check(st, "fa_bwd")
    return dq, dk, dv


def attention_naive(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                    scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                    lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """``attention`` computed the standard way, with the N x N score matrix in HBM
    (``fa_fwd_naive``: a cuBLAS GEMM for S, the library's row softmax, a cuBLAS GEMM
    for O).  The comparison the tiled kernels are measured against; N <= 32768.  The
    fp32 score workspace (4 * B * H * N * N bytes, about) is allocated with torch unless
    one is given.
    """
    lib = load_library()
    _check_qkv(q, k, v)
    if q.dtype not in _DTYPES:
        raise ValueError(f"dtype must be float16 or bfloat16, got {q.dtype}")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = ctypes.c_ulonglong(0)
    _check(lib.fa_fwd_naive_workspace_size(B, H, N, d, ctypes.byref(need)), "fa_fwd_naive_workspace_size")
    if workspace is None:
        workspace = torch.empty(max(need.value, 256), device=q.device, dtype=torch.uint8)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    with torch.cuda.device(q.device):
        st = lib.fa_fwd_naive(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d, float(scale),
                              int(bool(causal)), _DTYPES[q.dtype], _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream_handle(stream, q.device))
    _check(st, "fa_fwd_naive")
    return out, lse


def last_device_status(stream: Optional[torch.cuda.Stream] = None) -> Tuple[int, int]:
    """Synchronise and read/clear the device status word: (status, raw bits)."""
    lib = load_library()
    bits = ctypes.c_uint(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    st = lib.fa_last_device_status(_stream_handle(stream, dev), ctypes.byref(bits))
    return st, bits.value


def inject_stall(load_index: int, timeout_ms: int = 100) -> None:
    """Test hook: the next ``attention`` call leaves out one K/V load (see include/fa.h)."""
    _check(load_library().fa_debug_inject_stall(int(load_index), int(timeout_ms)), "fa_debug_inject_stall")
