"""Gradients of exact attention (the backward pass from the saved log-sum-exp), fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources: "FlashAttention-3 (NL)" and the hada.io FA3 summary ("Rückblick auf den
FlashAttention-Ansatz") describe FlashAttention as tiling plus recomputation: the score
matrix is never stored, and what the backward pass needs of the forward is recomputed from
Q, K, V and the per-row log-sum-exp.  The pages give no backward formulas; these are the
derivatives of the definition in ``attention`` (plain calculus), per (b, h):

    S   = scale * Q K^T  (masked entries -inf),   P = softmax_rows(S),   O = P V
    dV  = P^T dO
    dP  = dO V^T
    Delta_i = sum_j P_ij dP_ij = sum_d dO_id O_id
    dS  = P * (dP - Delta[:, None])
    dQ  = scale * dS K,     dK = scale * dS^T Q

O and P here are the oracle's own fp64 values computed from Q, K, V (never the GPU's).

Grouped-query attention (``gqa.attention_gqa``: query head h reads key/value head h // G) is
multi-head attention with every key/value head repeated G times, so its gradients are those
of the repeated problem with dK and dV summed over each group (the gradient of a repeated
input is the sum of the copies' gradients): ``attention_backward_gqa``.
"""

import numpy as np

from .attention import attention, attention_weights, default_scale

__all__ = ["attention_backward", "attention_backward_gqa", "attention_backward_rows"]


def attention_backward(q, k, v, do, scale=None, causal=False):
    """(dQ, dK, dV) [B, S, H, D] for inputs q, k, v and output gradient do [B, S, H, D]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, S, H, D = q.shape
    if scale is None:
        scale = default_scale(D)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            P, _, _ = attention_weights(q[b, :, h], k[b, :, h], scale, causal)
            o = P @ v[b, :, h]
            g = do[b, :, h]
            dv[b, :, h] = P.T @ g
            dP = g @ v[b, :, h].T
            delta = (g * o).sum(axis=1)
            dS = P * (dP - delta[:, None])
            dq[b, :, h] = scale * dS @ k[b, :, h]
            dk[b, :, h] = scale * dS.T @ q[b, :, h]
    return dq, dk, dv


def attention_backward_gqa(q, k, v, do, scale=None, causal=False):
    """(dQ [B, S, Hq, D], dK, dV [B, S, Hkv, D]) of grouped-query attention."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    Hq, Hkv = q.shape[2], k.shape[2]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    dq, dk_rep, dv_rep = attention_backward(q, np.repeat(k, G, axis=2), np.repeat(v, G, axis=2), do, scale, causal)
    B, S, _, D = k.shape
    return dq, dk_rep.reshape(B, S, Hkv, G, D).sum(axis=3), dv_rep.reshape(B, S, Hkv, G, D).sum(axis=3)


def attention_backward_rows(q, k, v, do, q_rows, k_rows, scale=None, causal=False):
    """The same gradients on sampled rows only, for sequences too long for an S x S matrix.

    Returns (dQ [B, len(q_rows), H, D], dK and dV [B, len(k_rows), H, D]).  Every entry is the
    formula above evaluated for one row or one column: O and lse of all query rows first
    (``attention``, row blocks), then, for query row i, P_i = exp(S_i - lse_i), dP_i = dO_i V^T,
    dS_i = P_i * (dP_i - Delta_i), dQ_i = scale * dS_i K; and for key j the column
    P_:j = exp(S_:j - lse), dV_j = P_:j^T dO, dS_:j = P_:j * (dO v_j - Delta),
    dK_j = scale * dS_:j^T Q."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, S, H, D = q.shape
    if scale is None:
        scale = default_scale(D)
    q_rows = np.asarray(q_rows, dtype=np.int64)
    k_rows = np.asarray(k_rows, dtype=np.int64)
    O, lse = attention(q, k, v, scale, causal)
    delta = (do * O).sum(axis=3)                                   # [B, S, H]
    dq = np.zeros((B, len(q_rows), H, D))
    dk = np.zeros((B, len(k_rows), H, D))
    dv = np.zeros((B, len(k_rows), H, D))
    keys = np.arange(S)
    for b in range(B):
        for h in range(H):
            Q, K, V, G = q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h]
            L, dl = lse[b, h], delta[b, :, h]
            # query rows
            s = scale * (Q[q_rows] @ K.T)
            vis = (keys[None, :] <= q_rows[:, None]) if causal else np.ones(s.shape, dtype=bool)
            P = np.where(vis, np.exp(s - L[q_rows, None]), 0.0)
            dS = P * (G[q_rows] @ V.T - dl[q_rows, None])
            dq[b, :, h] = scale * dS @ K
            # key columns
            sc = scale * (Q @ K[k_rows].T)                         # [S, n_k]
            visc = (keys[:, None] >= k_rows[None, :]) if causal else np.ones(sc.shape, dtype=bool)
            Pc = np.where(visc, np.exp(sc - L[:, None]), 0.0)
            dv[b, :, h] = Pc.T @ G
            dSc = Pc * (G @ V[k_rows].T - dl[:, None])
            dk[b, :, h] = scale * dSc.T @ Q
    return dq, dk, dv
