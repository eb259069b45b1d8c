"""Materialised-softmax attention in fp64: the definition the fused kernel must reach.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What is computed, per batch b, head h and query row i, with J(i) the visible
keys (all keys, or keys j <= i under the causal mask):

    s_ij   = scale * sum_d q[b,i,h,d] * k[b,j,h,d]
    m_i    = max_{j in J(i)} s_ij
    l_i    = sum_{j in J(i)} exp(s_ij - m_i)
    O[b,i,h,:] = sum_{j in J(i)} exp(s_ij - m_i) / l_i * v[b,j,h,:]
    lse[b,h,i] = m_i + ln(l_i)

Sources: the hada.io FA3 summary ("FlashAttention-3: Schnellere und präzisere
Attention ..."), section "Rückblick auf den FlashAttention-Ansatz": tiling
plus softmax rescaling gives the correct output blockwise, without
approximation -- so the fused kernel's target is the plain softmax(QK^T)V of
section "Überlappung von GEMM und Softmax" (GEMM Q-K, softmax, GEMM P-V).
The NL page ("FlashAttention-3 (NL)", "Het probleem van het
aandachtsmechanisme") names the S x S intermediate that the naive form
materialises; this oracle materialises it on purpose, one block of query rows
at a time.

Readings where the pages are silent: the layout is [B, S, H, D] (a row is one
token of one head); ``scale`` multiplies the logits (1/sqrt(D) by default);
the causal mask lets query i see key j iff j <= i (equal query and key
lengths); lse is the natural log of the sum of exponentials of the scaled,
masked logits.
"""

import numpy as np

__all__ = ["attention_weights", "attention", "online_softmax_attention", "default_scale"]

# Rows of the materialised score matrix handled at once (bounds memory only).
_ROW_CHUNK = 512


def default_scale(D):
    """Softmax scale used when the caller gives none: 1/sqrt(D)."""
    return 1.0 / np.sqrt(float(D))


def _visible(rows, S, causal):
    """Boolean [R, S] matrix: True where query rows[r] may attend to key j."""
    keys = np.arange(S)
    if not causal:
        return np.ones((len(rows), S), dtype=bool)
    return keys[None, :] <= np.asarray(rows)[:, None]


def attention_weights(q_bh, k_bh, scale, causal, rows=None):
    """Softmax weights P[r, j] for one (b, h): q_bh [S, D], k_bh [S, D], fp64.

    ``rows`` selects query rows (default: all).  Masked weights are exactly 0.
    Returns (P [R, S], m [R], l [R]) with m the row max of the scaled, masked
    logits and l the sum of exp(s - m) over visible keys.
    """
    S = k_bh.shape[0]
    rows = np.arange(q_bh.shape[0]) if rows is None else np.asarray(rows)
    s = scale * (q_bh[rows] @ k_bh.T)
    s = np.where(_visible(rows, S, causal), s, -np.inf)
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])
    l = e.sum(axis=1)
    return e / l[:, None], m, l


def attention(q, k, v, scale=None, causal=False, rows=None):
    """Exact attention forward, fp64.

    q, k, v: arrays [B, S, H, D] (converted to float64).  ``rows``: optional
    query-row indices (same for every b, h) to compute only a sample.
    Returns (O [B, R, H, D], lse [B, H, R]).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, S, H, D = q.shape
    if scale is None:
        scale = default_scale(D)
    rows = np.arange(S) if rows is None else np.asarray(rows, dtype=np.int64)
    R = len(rows)
    O = np.empty((B, R, H, D))
    lse = np.empty((B, H, R))
    for b in range(B):
        for h in range(H):
            for c0 in range(0, R, _ROW_CHUNK):
                r = rows[c0:c0 + _ROW_CHUNK]
                P, m, l = attention_weights(q[b, :, h, :], k[b, :, h, :], scale, causal, r)
                O[b, c0:c0 + len(r), h, :] = P @ v[b, :, h, :]
                lse[b, h, c0:c0 + len(r)] = m + np.log(l)
    return O, lse


def online_softmax_attention(q, k, v, scale=None, causal=False, block=128):
    """Blockwise recomputation with running max / running sum (fp64).

    Follows the hada.io summary, "Rückblick auf den FlashAttention-Ansatz":
    key/value blocks are visited one at a time; each block's scores update a
    running row max m and a running sum l, and the partial output is rescaled
    by exp(m_old - m_new) whenever the max grows.  Used only to pin
    :func:`attention` (the two must agree to rounding).
    Returns (O [B, S, H, D], lse [B, H, S]).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, S, H, D = q.shape
    if scale is None:
        scale = default_scale(D)
    O = np.empty_like(q)
    lse = np.empty((B, H, S))
    rows = np.arange(S)
    for b in range(B):
        for h in range(H):
            Q, K, V = q[b, :, h, :], k[b, :, h, :], v[b, :, h, :]
            m = np.full(S, -np.inf)
            l = np.zeros(S)
            acc = np.zeros((S, D))
            for j0 in range(0, S, block):
                cols = np.arange(j0, min(j0 + block, S))
                s = scale * (Q @ K[cols].T)
                if causal:
                    s = np.where(cols[None, :] <= rows[:, None], s, -np.inf)
                m_new = np.maximum(m, s.max(axis=1))
                # rows that have seen no visible key yet keep m = -inf
                safe = np.where(np.isfinite(m_new), m_new, 0.0)
                alpha = np.where(np.isfinite(m), np.exp(m - safe), 0.0)
                p = np.exp(s - safe[:, None])
                l = alpha * l + p.sum(axis=1)
                acc = alpha[:, None] * acc + p @ V[cols]
                m = m_new
            O[b, :, h, :] = acc / l[:, None]
            lse[b, h, :] = m + np.log(l)
    return O, lse
