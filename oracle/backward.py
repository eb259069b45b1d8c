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

from .attention import attention_weights, default_scale

__all__ = ["attention_backward", "attention_backward_gqa"]


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
