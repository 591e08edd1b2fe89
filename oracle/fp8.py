"""fp64 reference for the FP8 block quantisation with an optional Hadamard rotation.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources.  The news piece "Ignorierst du FlashAttention-3, rechnet deine KI jetzt
doppelt so langsam – 1,2 PFLOPs auf H100 erklärt" (section "Drei technische
Hebel", item 3 "FP8-Blockquantisierung", and section "Praxischeck", paragraph
"Präzision") says matrices are processed block by block in eight bits and that a
Hadamard transform reduces the quantisation error.  The concept card
"FlashAttention 2 + 3 — speicherbewusste Attention-Kernels" (section
"Kernpunkte", FP8 item) adds absmax scaling.  The pages fix neither the block,
the 8-bit format nor the transform size; the readings used here:

* format: OCP FP8 E4M3 ("fn": no infinities, largest finite 448, NaN = S.1111.111),
  round to nearest even, saturating to +-448;
* block: 64 consecutive rows of N for one (b, h), all d columns;
* scale: ``s = absmax / 448`` over the block, ``s = 1`` when the block is all zero;
  stored value ``x8 = e4m3(x / s)``, dequantised ``x8 * s``;
* rotation: the natural-order Sylvester matrix, normalised, ``x -> x @ H_d / sqrt(d)``
  applied along the head dimension to Q and K (the same matrix for both, so
  (QH)(KH)^T = QK^T); V is never rotated.

Variants (the next steps after the plain path, not on the pages beyond the words
"Hadamard-Transformation" and "Absmax"):

* randomised rotation: ``x -> (x * sigma) @ H_d / sqrt(d)`` with a +-1 sign vector
  sigma, the same for Q and K, so scores are still unchanged; sigma is an input
  (drawn by the caller from a seeded generator), given as a bit mask where bit c
  set means sigma_c = -1;
* per-head scale: one absmax over all N rows of a (b, h) instead of one per block,
  stored in every block entry of the scale array.

The e4m3 grid is written out from the format definition: a normal value is
``(1 + m/8) * 2^(E-7)`` for exponent field E in 1..15 (E=15, m=7 is NaN) and a
subnormal is ``m * 2^-9``.
"""
from __future__ import annotations

import numpy as np

from .sdpa import _f64, attention

__all__ = [
    "E4M3_MAX",
    "sign_vector",
    "sylvester_hadamard",
    "hadamard_rotate",
    "round_to_e4m3",
    "e4m3_encode",
    "e4m3_decode",
    "quantize_fp8_blocks",
    "dequantize_fp8_blocks",
    "emulate_fp8_attention",
]

E4M3_MAX = 448.0
_MIN_NORMAL_EXP = -6        # smallest normal: 2^-6
_MANT_BITS = 3
_SUBNORMAL_QUANTUM = 2.0 ** (_MIN_NORMAL_EXP - _MANT_BITS)   # 2^-9


def sylvester_hadamard(d: int) -> np.ndarray:
    """Unnormalised +-1 Hadamard matrix of order d (a power of two), Sylvester's
    recursion H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]]."""
    if d < 1 or d & (d - 1):
        raise ValueError(f"Hadamard order must be a power of two, got {d}")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def sign_vector(flips: int, d: int) -> np.ndarray:
    """+-1 vector of length d: entry c is -1 where bit c of the integer mask is set."""
    return np.array([-1.0 if (flips >> c) & 1 else 1.0 for c in range(d)])


def hadamard_rotate(x, signs=None) -> np.ndarray:
    """(x * signs) @ H_d / sqrt(d) along the last axis, in fp64 (signs: None or +-1 of length d).

    The +-1 matrix is applied first (sums of the inputs, exact in fp64 for
    bf16 data) and the result divided by sqrt(d) once."""
    x = _f64(x)
    d = x.shape[-1]
    if signs is not None:
        x = x * np.asarray(signs, dtype=np.float64)
    return (x @ sylvester_hadamard(d)) / np.sqrt(d)


def round_to_e4m3(x) -> np.ndarray:
    """Nearest E4M3 value (ties to even), saturating at +-448; fp64 in, fp64 out."""
    x = _f64(x)
    a = np.abs(x)
    _, e2 = np.frexp(a)                      # a = f * 2^e2, f in [0.5, 1)
    exp = (e2 - 1).astype(np.float64)        # floor(log2 a) for a > 0
    quantum = np.where(a >= 2.0 ** _MIN_NORMAL_EXP, np.exp2(exp - _MANT_BITS), _SUBNORMAL_QUANTUM)
    r = quantum * np.rint(a / quantum)       # np.rint rounds half to even; a/quantum is exact
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, x)


def e4m3_encode(values) -> np.ndarray:
    """Bit pattern (uint8) of values that already lie on the E4M3 grid."""
    v = _f64(values)
    sign = (np.signbit(v)).astype(np.uint8) << 7
    a = np.abs(v)
    code = np.zeros(a.shape, dtype=np.uint8)
    sub = (a > 0) & (a < 2.0 ** _MIN_NORMAL_EXP)
    code[sub] = np.rint(a[sub] / _SUBNORMAL_QUANTUM).astype(np.uint8)
    nrm = a >= 2.0 ** _MIN_NORMAL_EXP
    _, e2 = np.frexp(a[nrm])
    e = e2 - 1
    mant = np.rint((a[nrm] / np.exp2(e.astype(np.float64)) - 1.0) * 8.0).astype(np.int64)
    code[nrm] = ((e + 7) << 3 | mant).astype(np.uint8)
    return code | sign


def e4m3_decode(codes) -> np.ndarray:
    """fp64 value of E4M3 bit patterns (uint8)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    E = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(E == 0, m * _SUBNORMAL_QUANTUM, (1.0 + m / 8.0) * np.exp2(E.astype(np.float64) - 7.0))
    val = np.where((E == 0xF) & ((c & 0x7) == 0x7), np.nan, val)
    return sign * val


def quantize_fp8_blocks(x, block: int = 64, hadamard: bool = False, signs=None, per_head: bool = False):
    """Block absmax quantisation of ``x [B,H,N,d]`` to E4M3.

    Returns ``(codes uint8 [B,H,N,d], scales fp64 [B,H,ceil(N/block)])``; the
    rotation (with ``signs`` if given), when asked for, is applied before the
    absmax is taken.  With ``per_head`` the absmax runs over the whole head and
    every block of it gets that one scale.
    """
    y = hadamard_rotate(x, signs) if hadamard else _f64(x)
    B, H, N, d = y.shape
    nb = -(-N // block)
    scales = np.empty((B, H, nb))
    codes = np.empty((B, H, N, d), dtype=np.uint8)
    head_amax = np.abs(y).max(axis=(2, 3))
    for i in range(nb):
        blk = y[:, :, i * block:(i + 1) * block, :]
        amax = head_amax if per_head else np.abs(blk).max(axis=(2, 3))
        s = np.where(amax > 0, amax / E4M3_MAX, 1.0)
        scales[:, :, i] = s
        codes[:, :, i * block:(i + 1) * block, :] = e4m3_encode(round_to_e4m3(blk / s[:, :, None, None]))
    return codes, scales


def dequantize_fp8_blocks(codes, scales, block: int = 64) -> np.ndarray:
    """codes * scale of their block, fp64."""
    vals = e4m3_decode(codes)
    N = vals.shape[2]
    rep = np.repeat(_f64(scales), block, axis=2)[:, :, :N]
    return vals * rep[..., None]


def emulate_fp8_attention(q, k, v, scale: float, causal: bool, hadamard: bool, block: int = 64,
                          round_p: bool = False, signs=None, v_per_head: bool = False):
    """Predictor, not a reference: fp64 attention on dequantised E4M3 inputs.

    The reference for the FP8 path is ``attention`` on the unquantised inputs;
    this function only predicts, on the CPU, how far a quantised kernel lands
    from it with and without the rotation.  With ``round_p`` the softmax weights
    are also stored in E4M3 before the weighted sum over V, with V's per-block
    scales folded into them relative to the head's largest V scale:
    ``P~_ij = e4m3(p_ij * s_v(j) / max s_v)`` and
    ``O_i = max s_v * sum_j P~_ij * v8_j / sum_j p_ij``.
    ``signs`` randomises the rotation of Q and K; ``v_per_head`` gives V one scale
    per head.
    Returns ``(O, LSE)`` (the LSE is that of the dequantised scores).
    """
    qc, qs = quantize_fp8_blocks(q, block, hadamard, signs)
    kc, ks = quantize_fp8_blocks(k, block, hadamard, signs)
    vc, vs = quantize_fp8_blocks(v, block, False, per_head=v_per_head)
    qd, kd = dequantize_fp8_blocks(qc, qs, block), dequantize_fp8_blocks(kc, ks, block)
    if not round_p:
        return attention(qd, kd, dequantize_fp8_blocks(vc, vs, block), scale, causal)
    v8 = e4m3_decode(vc)
    B, H, N, d = qd.shape
    o = np.empty((B, H, N, d))
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            s = scale * (qd[b, h] @ kd[b, h].T)
            if causal:
                s = np.where(np.tril(np.ones((N, N), dtype=bool)), s, -np.inf)
            m = s.max(axis=1)
            p = np.exp(s - m[:, None])
            l = p.sum(axis=1)
            g = np.repeat(vs[b, h], block)[:N]
            p8 = round_to_e4m3(p * (g / g.max())[None, :])
            o[b, h] = g.max() * (p8 @ v8[b, h]) / l[:, None]
            lse[b, h] = m + np.log(l)
    return o, lse
