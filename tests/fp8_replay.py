"""CPU replay of the roundings of the E4M3 attention forward (test infrastructure).

The exact reference for the FP8 path is the fp64 attention on the unquantised
inputs, and E4M3 storage keeps the kernel several per cent away from it.  That
distance says little about the kernel itself: an error of a few per cent of its
own (a wrong block scale, a weight folded with the wrong factor) hides inside
it.  This replay closes the gap so the kernel can be checked element by element.

It takes the SAME E4M3 codes and fp32 block scales that the kernel reads (made on
the CPU by the oracle's quantiser and uploaded to the GPU, never read back from
it) and performs, in fp64, the roundings that the kernel's schedule performs on
them:

* scores are products of E4M3 values summed exactly, times the row's and the
  key block's dequantisation factors (formed in fp32, as the kernel forms them);
* keys are taken in tiles of 128; each row keeps a running maximum (log2
  units) that is moved only when a tile's maximum exceeds it by more than 8,
  with the partial output and sum corrected by 2^(old - new) when it moves;
* each softmax weight 2^(score - running max), times V's block scale relative to
  the head's largest, is rounded to E4M3 (nearest, ties to even: the oracle's
  ``round_to_e4m3``) before the weighted sum over the V codes;
* the row sum is of the unrounded weights; the output is the weighted sum times
  the largest V scale over the row sum, and LSE = ln 2 * (max + log2 sum).

In real arithmetic the running maximum cancels, so without the rounding of the
weights the replay equals the fp64 attention on the dequantised inputs (a pin in
``test_oracle.py``).  What is left between the kernel and the replay: the final
bf16 rounding of O, and the fp32 arithmetic of the exponent, of ``ex2`` and of
the MMA accumulation, which move a weight's E4M3 rounding only where the exact
value lies within about 1e-5 (relative) of a midpoint between two codes.
"""
from __future__ import annotations

import math

import numpy as np

import oracle

TILE = 128              # keys per tile of the kernel's schedule
BLOCK = 64              # rows per quantisation block
LAZY_THRESHOLD = 8.0    # log2 units the row maximum must grow by before it is moved
LOG2E = 1.4426950408889634


def _f32(x):
    return np.asarray(x, dtype=np.float32)


def replay_fp8_attention(q8, k8, v8, qs, ks, vs, scale: float, causal: bool, round_p: bool = True,
                         threshold: float = LAZY_THRESHOLD):
    """Replay of the E4M3 forward on codes ``q8, k8, v8`` (uint8 ``[B,H,N,d]``, V not
    transposed) with fp32 block scales ``qs, ks, vs`` (``[B,H,ceil(N/64)]``).

    Returns ``(O, LSE, W)`` in fp64, where ``W[b,h,i,c] = s_v,max / l_i *
    sum_j |P~_ij| |v8_jc|`` is the magnitude of the weighted sum behind O (the
    scale of any error in the weights).
    """
    qv, kv, vv = oracle.e4m3_decode(q8), oracle.e4m3_decode(k8), oracle.e4m3_decode(v8)
    qs, ks, vs = _f32(qs), _f32(ks), _f32(vs)
    B, H, N, d = qv.shape
    sl2 = _f32(np.float32(scale) * np.float32(LOG2E))
    rows = np.arange(N)
    o = np.empty((B, H, N, d))
    w = np.empty((B, H, N, d))
    lse = np.empty((B, H, N))
    n_tiles = -(-N // TILE)
    for b in range(B):
        for h in range(H):
            acc = qv[b, h] @ kv[b, h].T                                  # exact in fp64
            c_row = _f32(sl2 * qs[b, h][rows // BLOCK]).astype(np.float64)  # fp32 like the kernel
            f_col = _f32(c_row[:, None].astype(np.float32) * ks[b, h][None, np.arange(N) // BLOCK])
            s = acc * f_col.astype(np.float64)                           # log2 units
            if causal:
                s = np.where(np.arange(N)[None, :] <= rows[:, None], s, -np.inf)
            sv_max = np.float32(vs[b, h].max())
            inv_sv = np.float32(np.float32(1.0) / sv_max)
            bcol = np.log2((vs[b, h][np.arange(N) // BLOCK] * inv_sv).astype(np.float64))  # <= 0
            m = np.full(N, -np.inf)
            l = np.zeros(N)
            acc_o = np.zeros((N, d))
            acc_w = np.zeros((N, d))
            for j in range(n_tiles):
                cols = slice(j * TILE, min(N, (j + 1) * TILE))
                st = s[:, cols]
                if causal:
                    live = rows >= j * TILE           # rows whose tiles reach this one
                else:
                    live = np.ones(N, dtype=bool)
                m_new = np.maximum(m, st.max(axis=1))
                if j == 0:
                    m_use = np.where(np.isfinite(m_new), m_new, 0.0)
                    alpha = np.ones(N)
                else:
                    need = m_new > m + threshold
                    m_use = np.where(need, m_new, m)
                    alpha = np.where(need, np.exp2(m - m_new), 1.0)
                m_use = np.where(live, m_use, m)
                alpha = np.where(live, alpha, 1.0)
                x = st + bcol[None, cols] - m_use[:, None]
                pw = np.where(live[:, None], np.exp2(x), 0.0)
                pr = oracle.round_to_e4m3(pw) if round_p else pw
                l = l * alpha + (pw * np.exp2(-bcol[None, cols])).sum(axis=1)
                acc_o = acc_o * alpha[:, None] + pr @ vv[b, h, cols]
                acc_w = acc_w * alpha[:, None] + np.abs(pr) @ np.abs(vv[b, h, cols])
                m = m_use
            with np.errstate(divide="ignore", invalid="ignore"):
                o[b, h] = acc_o * (float(sv_max) / l)[:, None]
                w[b, h] = acc_w * (float(sv_max) / l)[:, None]
                lse[b, h] = math.log(2.0) * (m + np.log2(l))
    return o, lse, w


def quantize_for_both(x, hadamard: bool, signs=None, per_head: bool = False):
    """Oracle E4M3 codes and their fp32 scales: the inputs both the kernel and the replay read."""
    codes, sc = oracle.quantize_fp8_blocks(x, BLOCK, hadamard, signs, per_head)
    return codes, sc.astype(np.float32)
