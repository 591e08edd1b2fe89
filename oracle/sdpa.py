"""Plain fp64 scaled-dot-product attention: the definition, written out.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Nothing here is tiled,
fused or reordered beyond what the definition states; the score matrix is
materialised (row-chunked only to bound memory, which changes no arithmetic of
any single row).

What is computed, per (b, h) and query row i (the pages' problem statement:
"FlashAttention 2 + 3 — speicherbewusste Attention-Kernels", section
"Kernpunkte": the same output as softmax(QK^T/sqrt(d)) V; the "Flash Attention"
glossary, section "/01 Was ist Flash Attention?": the same results as classic
attention):

    s_ij   = scale * <q_i, k_j>                 (scale passed in; 1/sqrt(d) in the workloads)
    s_ij   = -inf  for j > i                    (causal only; key j visible iff j <= i)
    m_i    = max_j s_ij
    p_ij   = exp(s_ij - m_i)
    l_i    = sum_j p_ij
    O_i    = (sum_j p_ij v_j) / l_i
    LSE_i  = m_i + log(l_i)                     (natural log, scale included)

A row with no visible key (cannot occur when N_q = N_k and the mask is causal)
gives O_i = 0 and LSE_i = -inf.

Inputs are converted to float64 from the values the GPU sees (the already
rounded fp16/bf16 tensors), so the oracle and the kernel start from identical
numbers.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

__all__ = [
    "attention",
    "attention_decode",
    "attention_probs",
    "brute_force_attention",
    "online_softmax_attention",
    "rel_rms",
]

# Largest fp64 score block (rows x keys) materialised at once: 32 Mi entries = 256 MB.
_MAX_BLOCK_ELEMS = 32 * 1024 * 1024


def _f64(x) -> np.ndarray:
    """Any array-like (numpy or a CPU torch tensor) as a float64 numpy array."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def _check(q, k, v):
    if q.ndim != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError(f"expected Q, K, V of one shape [B,H,N,d]; got {q.shape} {k.shape} {v.shape}")


def _rows_of_head(qh, kh, vh, scale: float, causal: bool, rows: np.ndarray):
    """O and LSE for the query rows ``rows`` of one head (fp64)."""
    n_keys = kh.shape[0]
    s = scale * (qh[rows] @ kh.T)                       # [len(rows), N] scores
    if causal:
        visible = np.arange(n_keys)[None, :] <= rows[:, None]
        s = np.where(visible, s, -np.inf)
    m = s.max(axis=1)                                   # row max
    m_safe = np.where(np.isfinite(m), m, 0.0)
    p = np.exp(s - m_safe[:, None])                     # exp(-inf) = 0 for masked keys
    l = p.sum(axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        o = (p @ vh) / l[:, None]
        lse = m + np.log(l)
    empty = l == 0.0
    o[empty] = 0.0
    lse[empty] = -np.inf
    return o, lse


def attention(q, k, v, scale: float, causal: bool, rows: Optional[Sequence[int]] = None):
    """Exact attention forward in fp64.

    q, k, v: ``[B, H, N, d]`` (numpy or CPU torch).  ``rows``: optional sorted
    query-row indices, the same for every head; only those rows are computed.
    Returns ``(O [B,H,R,d], LSE [B,H,R])`` as float64 numpy arrays, R = N or
    len(rows).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    _check(q, k, v)
    B, H, N, d = q.shape
    row_idx = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    R = row_idx.shape[0]
    o = np.empty((B, H, R, d), dtype=np.float64)
    lse = np.empty((B, H, R), dtype=np.float64)
    chunk = max(1, min(R, _MAX_BLOCK_ELEMS // max(N, 1)))
    for b in range(B):
        for h in range(H):
            for r0 in range(0, R, chunk):
                sel = row_idx[r0:r0 + chunk]
                o[b, h, r0:r0 + chunk], lse[b, h, r0:r0 + chunk] = _rows_of_head(
                    q[b, h], k[b, h], v[b, h], scale, causal, sel)
    return o, lse


def attention_probs(q, k, v, scale: float, causal: bool) -> np.ndarray:
    """The full softmax matrix P = softmax(scale*QK^T [+mask]) (small inputs only)."""
    q, k = _f64(q), _f64(k)
    N = q.shape[-2]
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    if causal:
        s = np.where(np.tril(np.ones((N, N), dtype=bool)), s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    p = np.exp(s - m)
    return p / p.sum(axis=-1, keepdims=True)


def brute_force_attention(q, k, v, scale: float, causal: bool):
    """The same definition with pure-Python loops and ``math`` (tiny inputs)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    _check(q, k, v)
    B, H, N, d = q.shape
    o = np.zeros((B, H, N, d))
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                keys = range(i + 1) if causal else range(N)
                scores = []
                for j in keys:
                    acc = 0.0
                    for c in range(d):
                        acc += float(q[b, h, i, c]) * float(k[b, h, j, c])
                    scores.append(scale * acc)
                mx = max(scores)
                weights = [math.exp(s - mx) for s in scores]
                total = sum(weights)
                for c in range(d):
                    acc = 0.0
                    for w, j in zip(weights, keys):
                        acc += w * float(v[b, h, j, c])
                    o[b, h, i, c] = acc / total
                lse[b, h, i] = mx + math.log(total)
    return o, lse


def online_softmax_attention(q, k, v, scale: float, causal: bool, block: int):
    """The streaming form of the same result, block of ``block`` keys at a time.

    Follows the online softmax as the concept card "FlashAttention 2 + 3 —
    speicherbewusste Attention-Kernels" describes it ("Begriffe auf dieser
    Seite", Online-Softmax): a running maximum per row, and a correction factor
    applied to the partial sums at every tile boundary, so the normaliser is
    never formed over all keys at once.  In exact arithmetic it equals
    ``attention``; the tests check that in fp64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    _check(q, k, v)
    B, H, N, d = q.shape
    o = np.zeros((B, H, N, d))
    lse = np.zeros((B, H, N))
    rows = np.arange(N)
    for b in range(B):
        for h in range(H):
            m = np.full(N, -np.inf)          # running max
            l = np.zeros(N)                  # running sum of exp(s - m)
            acc = np.zeros((N, d))           # running un-normalised output
            for j0 in range(0, N, block):
                cols = np.arange(j0, min(N, j0 + block))
                s = scale * (q[b, h] @ k[b, h, cols].T)
                if causal:
                    s = np.where(cols[None, :] <= rows[:, None], s, -np.inf)
                m_new = np.maximum(m, s.max(axis=1))
                m_use = np.where(np.isfinite(m_new), m_new, 0.0)
                corr = np.exp(np.where(np.isfinite(m), m, m_use) - m_use)   # correction factor
                corr = np.where(np.isfinite(m), corr, 0.0)
                p = np.exp(s - m_use[:, None])
                l = corr * l + p.sum(axis=1)
                acc = corr[:, None] * acc + p @ v[b, h, cols]
                m = m_new
            with np.errstate(invalid="ignore", divide="ignore"):
                o[b, h] = acc / l[:, None]
                lse[b, h] = m + np.log(l)
    return o, lse


def rel_rms(x, ref) -> float:
    """||x - ref||_F / ||ref||_F over all elements."""
    x, ref = _f64(x), _f64(ref)
    return float(np.linalg.norm((x - ref).ravel()) / np.linalg.norm(ref.ravel()))


def attention_decode(q, k, v, scale: float, causal: bool):
    """Attention of N_q query rows against N_k >= N_q keys (a KV-cache step), fp64.

    q: ``[B, H, N_q, d]``; k, v: ``[B, H, N_k, d]``.  The queries are the last N_q
    positions of the sequence, so with ``causal`` query row i sees keys
    0 .. N_k - N_q + i (bottom-right alignment); without it every row sees all
    keys.  Same definition as ``attention`` otherwise; returns
    ``(O [B,H,N_q,d], LSE [B,H,N_q])``.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim != 4 or k.shape != v.shape or k.shape[:2] != q.shape[:2] or k.shape[3] != q.shape[3]:
        raise ValueError(f"bad decode shapes {q.shape} {k.shape} {v.shape}")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if Nq > Nk:
        raise ValueError("N_q must not exceed N_k")
    o = np.empty((B, H, Nq, d))
    lse = np.empty((B, H, Nq))
    for b in range(B):
        for h in range(H):
            s = scale * (q[b, h] @ k[b, h].T)                       # [N_q, N_k]
            if causal:
                last = (Nk - Nq) + np.arange(Nq)                    # last visible key per row
                s = np.where(np.arange(Nk)[None, :] <= last[:, None], s, -np.inf)
            m = s.max(axis=1)
            p = np.exp(s - m[:, None])
            l = p.sum(axis=1)
            o[b, h] = (p @ v[b, h]) / l[:, None]
            lse[b, h] = m + np.log(l)
    return o, lse
