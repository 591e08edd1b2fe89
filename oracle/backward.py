"""Plain fp64 gradient of the attention forward pass: the chain rule, written out.

TEST INFRASTRUCTURE ONLY (see the package docstring).  The probability matrix is
materialised (row-chunked only to bound memory); nothing is tiled, fused or
reordered beyond what the formulas below state.

The pages name the backward pass (the concept card "FlashAttention 2 + 3 —
speicherbewusste Attention-Kernels", section "Kernpunkte": FlashAttention-2's
better parallelism in the backward pass; the "Flash Attention" glossary, section
"/02 Technische Vorteile im Überblick": faster training) but print no formula
for it.  The gradient is therefore the calculus of the forward definition in
``sdpa.py``.  For an upstream gradient dO of the output O, per (b, h):

    S      = scale * Q K^T, masked entries -inf       (causal: key j visible iff j <= i)
    P      = row-wise softmax of S                     (masked entries 0)
    dV     = P^T dO
    dP     = dO V^T
    D_i    = sum_j P_ij dP_ij  (= sum_c dO_ic O_ic)
    dS     = P * (dP - D)                              (elementwise, D broadcast along j)
    dQ     = scale * dS K
    dK     = scale * dS^T Q

Inputs are converted to float64 from the values the GPU sees.
"""
from __future__ import annotations

import math

import numpy as np

from .sdpa import _MAX_BLOCK_ELEMS, _check, _f64

__all__ = ["attention_backward", "brute_force_attention_backward", "attention_backward_delta"]


def _probs_rows(qh, kh, scale: float, causal: bool, r0: int, r1: int) -> np.ndarray:
    """Rows r0..r1-1 of P for one head (fp64), masked entries exactly 0."""
    s = scale * (qh[r0:r1] @ kh.T)
    if causal:
        rows = np.arange(r0, r1)[:, None]
        s = np.where(np.arange(kh.shape[0])[None, :] > rows, -np.inf, s)
    m = s.max(axis=1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m)
    lsum = e.sum(axis=1, keepdims=True)
    return np.divide(e, lsum, out=np.zeros_like(e), where=lsum > 0)


def attention_backward(q, k, v, do, scale: float, causal: bool):
    """(dQ, dK, dV) in float64, each [B, H, N, d], for upstream gradient ``do``."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    _check(q, k, v)
    if do.shape != q.shape:
        raise ValueError(f"dO must be shaped like Q; got {do.shape} vs {q.shape}")
    B, H, N, d = q.shape
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    step = max(1, _MAX_BLOCK_ELEMS // max(N, 1))
    for b in range(B):
        for h in range(H):
            qh, kh, vh, doh = q[b, h], k[b, h], v[b, h], do[b, h]
            for r0 in range(0, N, step):
                r1 = min(N, r0 + step)
                p = _probs_rows(qh, kh, scale, causal, r0, r1)        # rows x N
                dv[b, h] += p.T @ doh[r0:r1]
                dp = doh[r0:r1] @ vh.T
                delta = (p * dp).sum(axis=1, keepdims=True)
                ds = p * (dp - delta)
                dq[b, h, r0:r1] = scale * (ds @ kh)
                dk[b, h] += scale * (ds.T @ qh[r0:r1])
    return dq, dk, dv


def attention_backward_delta(o, do) -> np.ndarray:
    """D_i = sum_c dO_ic O_ic, [B, H, N] float64 (equal to sum_j P_ij dP_ij)."""
    return (_f64(o) * _f64(do)).sum(axis=-1)


def brute_force_attention_backward(q, k, v, do, scale: float, causal: bool):
    """The same gradient with explicit Python loops over every index (tiny inputs only)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, d = q.shape
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            for i in range(N):
                vis = [j for j in range(N) if not (causal and j > i)]
                s = {j: scale * sum(q[b, h, i, c] * k[b, h, j, c] for c in range(d)) for j in vis}
                m = max(s.values())
                z = sum(math.exp(s[j] - m) for j in vis)
                p = {j: math.exp(s[j] - m) / z for j in vis}
                dp = {j: sum(do[b, h, i, c] * v[b, h, j, c] for c in range(d)) for j in vis}
                delta = sum(p[j] * dp[j] for j in vis)
                for j in vis:
                    ds = p[j] * (dp[j] - delta)
                    for c in range(d):
                        dv[b, h, j, c] += p[j] * do[b, h, i, c]
                        dq[b, h, i, c] += scale * ds * k[b, h, j, c]
                        dk[b, h, j, c] += scale * ds * q[b, h, i, c]
    return dq, dk, dv
