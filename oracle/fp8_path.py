"""The FP8 attention path end to end, in fp64 arithmetic with E4M3 rounding emulated.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Steps, in the order of "FlashAttention-3 (NL)", "Technische innovaties",
item 3, and the hada.io summary, "Niedrige FP8-Präzision und incoherent
processing":

1. (optional) rotate Q and K with the same random-sign Hadamard matrix;
2. quantise Q, K and V to E4M3 with one scale per (b, h, 128-token block);
3. attention on the de-quantised values, with both GEMMs in FP8: the scores
   come from the E4M3 Q and K, and the softmax numerators exp(s - m) are
   rounded to E4M3 before the P-V product (the second GEMM's A operand);
   the row sum l uses the unrounded numerators.

Readings where the pages are silent: the numerators are rounded relative to
the exact row max m (so they lie in (0, 1]); the output is O = (E4M3(P~) @ V)
/ l with P~ = exp(s - m).  The rotation is orthogonal, so without
quantisation the result equals plain attention ("FlashAttention-3 (NL)",
item 3, step 4).

V's block scales can be folded into the numerators instead of into V (the
reading of the V descale used for the FP8 attention step): with sv_j the
scale of key j's block and sv_max the largest of the head's block scales,
the E4M3 operand is the numerator times r_j = sv_j / sv_max <= 1, and the
product with the codes of V is scaled back by sv_max.  In real arithmetic
this is the same O; with the rounding it is E4M3(P~_ij * r_j) / r_j that
multiplies V (``v_ratio``).
"""

import numpy as np

from .attention import default_scale, _visible
from .e4m3 import round_e4m3
from .quantise import quantise_blocks, dequantise

__all__ = ["quantise_qkv", "attention_rounded_p", "fp8_attention", "v_block_ratio"]


def quantise_qkv(q, k, v, signs=None):
    """Quantise Q, K (rotated when ``signs`` is given) and V (never rotated)."""
    Qq = quantise_blocks(q, signs)
    Kq = quantise_blocks(k, signs)
    Vq = quantise_blocks(v, None)
    return Qq, Kq, Vq


def v_block_ratio(v_scale, S, block=128):
    """r [B, H, S]: the block scale of each key over the largest block scale of its head
    (0 for every key of a head whose scales are all 0)."""
    v_scale = np.asarray(v_scale, dtype=np.float64)
    per_key = v_scale[:, :, np.arange(S) // block]
    mx = v_scale.max(axis=2, keepdims=True)
    return np.where(mx > 0, per_key / np.where(mx > 0, mx, 1.0), 0.0)


def attention_rounded_p(qd, kd, vd, scale, causal=False, rows=None, round_p=True, v_ratio=None):
    """Attention on de-quantised fp64 inputs with the numerators rounded to E4M3.

    qd, kd, vd: [B, S, H, D] fp64.  With ``round_p=False`` this is plain exact
    attention on the given inputs.  ``v_ratio`` [B, H, S] (see v_block_ratio):
    the rounded quantity is the numerator times the key's ratio, divided by it
    again after rounding.  Returns (O [B,R,H,D], lse [B,H,R]).
    """
    B, S, H, D = qd.shape
    rows = np.arange(S) if rows is None else np.asarray(rows, dtype=np.int64)
    O = np.empty((B, len(rows), H, D))
    lse = np.empty((B, H, len(rows)))
    vis = _visible(rows, S, causal)
    for b in range(B):
        for h in range(H):
            s = scale * (qd[b, rows, h, :] @ kd[b, :, h, :].T)
            s = np.where(vis, s, -np.inf)
            m = s.max(axis=1)
            e = np.exp(s - m[:, None])
            l = e.sum(axis=1)
            if not round_p:
                p = e
            elif v_ratio is None:
                p = round_e4m3(e)
            else:
                # a key whose block scale is 0 has V = 0: its term vanishes (the limit r -> 0)
                r = np.asarray(v_ratio, dtype=np.float64)[b, h][None, :]
                rs = np.where(r > 0, r, 1.0)
                p = np.where(r > 0, round_e4m3(e * rs) / rs, 0.0)
            O[b, :, h, :] = (p @ vd[b, :, h, :]) / l[:, None]
            lse[b, h, :] = m + np.log(l)
    return O, lse


def fp8_attention(q, k, v, signs=None, scale=None, causal=False, rows=None, round_p=True, fold_v=False):
    """Rotate (optional), quantise, and attend.  Inputs [B,S,H,D] fp64 values.

    ``fold_v``: round the numerators with V's block ratios folded in (v_ratio).
    Returns (O, lse, (Qq, Kq, Vq)) with the quantiser outputs of
    :func:`oracle.quantise.quantise_blocks`.
    """
    q = np.asarray(q, dtype=np.float64)
    D = q.shape[-1]
    if scale is None:
        scale = default_scale(D)
    Qq, Kq, Vq = quantise_qkv(q, k, v, signs)
    qd = dequantise(Qq["q"], Qq["scale"])
    kd = dequantise(Kq["q"], Kq["scale"])
    vd = dequantise(Vq["q"], Vq["scale"])
    ratio = v_block_ratio(Vq["scale"], vd.shape[1]) if fold_v else None
    O, lse = attention_rounded_p(qd, kd, vd, scale, causal, rows, round_p, ratio)
    return O, lse, (Qq, Kq, Vq)
