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

"""

import numpy as np

from .attention import default_scale, _visible
from .e4m3 import round_e4m3
from .quantise import quantise_blocks, dequantise

__all__ = ["quantise_qkv", "attention_rounded_p", "fp8_attention"]


def quantise_qkv(q, k, v, signs=None, granularity="block"):
    """Quantise Q, K (rotated when ``signs`` is given) and V (never rotated)."""
    Qq = quantise_blocks(q, signs, granularity=granularity)
    Kq = quantise_blocks(k, signs, granularity=granularity)
    Vq = quantise_blocks(v, None, granularity=granularity)
    return Qq, Kq, Vq


def attention_rounded_p(qd, kd, vd, scale, causal=False, rows=None, round_p=True):
    """Attention on de-quantised fp64 inputs with the numerators rounded to E4M3.

    qd, kd, vd: [B, S, H, D] fp64.  With ``round_p=False`` this is plain exact
    attention on the given inputs.  Returns (O [B,R,H,D], lse [B,H,R]).
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
            p = round_e4m3(e) if round_p else e
            O[b, :, h, :] = (p @ vd[b, :, h, :]) / l[:, None]
            lse[b, h, :] = m + np.log(l)
    return O, lse


def fp8_attention(q, k, v, signs=None, scale=None, causal=False, rows=None, round_p=True,
                  granularity="block"):
    """Rotate (optional), quantise, and attend.  Inputs [B,S,H,D] fp64 values.

    ``granularity``: the quantiser's scale granularity ("block" or "tensor").
    Returns (O, lse, (Qq, Kq, Vq)) with the quantiser outputs of
    :func:`oracle.quantise.quantise_blocks`.
    """
    q = np.asarray(q, dtype=np.float64)
    D = q.shape[-1]
    if scale is None:
        scale = default_scale(D)
    Qq, Kq, Vq = quantise_qkv(q, k, v, signs, granularity)
    qd = dequantise(Qq["q"], Qq["scale"])
    kd = dequantise(Kq["q"], Kq["scale"])
    vd = dequantise(Vq["q"], Vq["scale"])
    O, lse = attention_rounded_p(qd, kd, vd, scale, causal, rows, round_p)
    return O, lse, (Qq, Kq, Vq)
