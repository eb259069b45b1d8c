"""Blockwise-scaled E4M3 quantiser with optional random-sign Hadamard rotation, fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources: "FlashAttention-3 (NL)", "Technische innovaties", item 3 (Lage
precisie (FP8)), steps 1-3: multiply Q and K by a random orthogonal matrix,
which spreads outlier magnitude over all coordinates, then quantise to FP8
with a smaller error.  hada.io FA3 summary, "Niedrige FP8-Präzision und
incoherent processing": outliers in activations make quantisation hard and
enlarge its error.

Readings where the pages are silent: one fp32 scale per (batch b, head h,
block of 128 consecutive tokens), equal to amax / 448 over the block's
(rotated) values, or 1 when the block is all zero; each value is divided by
its block's scale and rounded to E4M3 (nearest even, saturating).  The
de-quantised value is code_value * scale.  Q, K and V all use this
quantiser; only Q and K are rotated (V is quantised as is).

Precision of the rounding decision: the quotient x' / scale is formed in
fp32, the precision of the GPU kernel, as fl32(y) * fl32(448 / amax(fl32(y)))
with y = (x * signs) H_D the unnormalised transform (exact in fp64 for bf16
inputs; x' = y / sqrt(D)).  In real arithmetic this equals x' / scale, but
when amax has odd factors (amax = 26 gives x * 224 / 13) a fraction of the
quotients are exact E4M3 rounding midpoints, and fp64 and fp32 would break
those ties differently; taking the decision in the kernel's precision makes
the codes a single well-defined answer.  The stored scale is the fp64 value
amax(x') / 448.
"""

import numpy as np

from .e4m3 import E4M3_MAX, round_e4m3, encode
from .hadamard import sylvester

__all__ = ["TOKEN_BLOCK", "quantise_blocks", "dequantise"]

TOKEN_BLOCK = 128


def quantise_blocks(x, signs=None, block=TOKEN_BLOCK):
    """Quantise x [B, S, H, D] (fp64 values) per (b, h, token block).

    ``signs``: length-D vector of +-1 to rotate with, or None for no rotation.
    Returns a dict with
      ``rotated`` [B,S,H,D]  the (rotated) values before scaling,
      ``scale``   [B,H,nblk] amax / 448 per block (1 for an all-zero block),
      ``pre``     [B,S,H,D]  rotated / scale formed in fp32, the value that is rounded,
      ``q``       [B,S,H,D]  the E4M3 value of each element (pre rounded),
      ``codes``   [B,S,H,D]  uint8 E4M3 bytes.
    """
    x = np.asarray(x, dtype=np.float64)
    B, S, H, D = x.shape
    if signs is not None:
        y = (x * np.asarray(signs, dtype=np.float64)) @ sylvester(D)   # unnormalised transform
        norm = 1.0 / np.sqrt(float(D))
    else:
        y, norm = x, 1.0
    xr = y * norm
    y32 = y.astype(np.float32)
    nblk = (S + block - 1) // block
    scale = np.empty((B, H, nblk))
    pre = np.empty_like(xr)
    for i in range(nblk):
        t0, t1 = i * block, min((i + 1) * block, S)
        amax = np.abs(y[:, t0:t1]).max(axis=(1, 3))                 # [B, H], fp64
        scale[:, :, i] = np.where(amax > 0, amax * norm / E4M3_MAX, 1.0)
        amax32 = np.abs(y32[:, t0:t1]).max(axis=(1, 3))             # [B, H], fp32
        with np.errstate(divide="ignore"):
            inv32 = np.where(amax32 > 0, np.float32(E4M3_MAX) / amax32, np.float32(0)).astype(np.float32)
        pre[:, t0:t1] = (y32[:, t0:t1] * inv32[:, None, :, None]).astype(np.float64)
    q = round_e4m3(pre)
    return {"rotated": xr, "scale": scale, "pre": pre, "q": q, "codes": encode(q)}


def dequantise(q, scale, block=TOKEN_BLOCK):
    """Values q [B,S,H,D] times their block's scale [B,H,nblk]."""
    q = np.asarray(q, dtype=np.float64)
    S = q.shape[1]
    tok_blk = np.arange(S) // block                              # [S]
    per_tok = np.transpose(scale, (0, 2, 1))[:, tok_blk, :]      # [B, S, H]
    return q * per_tok[..., None]
