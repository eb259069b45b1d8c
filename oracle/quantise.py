"""Blockwise-scaled E4M3 quantiser with optional random-sign Hadamard rotation, fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources: "FlashAttention-3 (NL)", "Technische innovaties", item 3 (Lage
precisie (FP8)), steps 1-3: multiply Q and K by a random orthogonal matrix,
which spreads outlier magnitude over all coordinates, then quantise to FP8
with a smaller error.  hada.io FA3 summary, "Niedrige FP8-Präzision und
incoherent processing": outliers in activations make quantisation hard and
enlarge its error.

Readings where the pages are silent: one scale per (batch b, head h, block of
128 consecutive tokens), equal to amax / 448 over the block's (rotated)
values, or 1 when the block is all zero; each value is divided by its block's
scale and rounded to E4M3 (nearest, ties to even, saturating).  The
de-quantised value is code_value * scale.  Q, K and V all use this
quantiser; only Q and K are rotated (V is quantised as is).  The alternative
reading of "standard FP8" -- one scale for the whole tensor -- is
``granularity="tensor"``.

The rounding is the plain definition, decided exactly: the quotient
x' / scale equals 448 * y / amax(y) in real arithmetic, with y = (x * s) H_D
the unnormalised transform (x' = y / sqrt(D)) and amax(y) the block's (or
tensor's) largest |y|.  It is evaluated in fp64, with a forward error bound:
a D-term sum of +-x errs by at most D 2^-53 sum_d |x_d| in any order, so the
quotient's error is bounded element by element.  Every element whose fp64
quotient lies within that bound (plus 2^-30 of a grid step) of an E4M3
rounding midpoint is decided again in exact rational arithmetic
(``fractions.Fraction``): its y, and the exact maximum of its block, are
recomputed from the input values.  Exact midpoints thus go to the even
neighbour, whatever the precision of the input values.
"""

from fractions import Fraction

import numpy as np

from .e4m3 import E4M3_MAX, round_e4m3, encode
from .hadamard import sylvester

__all__ = ["TOKEN_BLOCK", "quantise_blocks", "dequantise", "rne_e4m3_fraction", "grid_step"]

TOKEN_BLOCK = 128
_NEAR = 2.0 ** -30          # extra distance to a midpoint, in grid steps, decided exactly


def rne_e4m3_fraction(F):
    """The E4M3 value nearest to the exact rational F (ties to even, saturating), as a float."""
    F = Fraction(F)
    if F == 0:
        return 0.0
    sign = -1.0 if F < 0 else 1.0
    a = abs(F)
    e = a.numerator.bit_length() - a.denominator.bit_length()     # 2^(e-1) < a < 2^(e+1)
    if Fraction(2) ** e > a:
        e -= 1
    if Fraction(2) ** (e + 1) <= a:
        e += 1
    step = Fraction(2) ** (max(e, -6) - 3)                        # spacing of E4M3 values there
    t = a / step
    n = t.numerator // t.denominator
    rem = t - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * min(float(n * step), E4M3_MAX)


def grid_step(v):
    """Spacing of E4M3 values in the binade of |v| (2^(e-3); 2^-9 below 2^-6), fp64 arrays."""
    av = np.abs(np.asarray(v, dtype=np.float64))
    _, ex = np.frexp(np.where(av > 0, av, 1.0))
    return np.exp2((np.maximum(ex - 1, -6) - 3).astype(np.float64))


def _y_exact(x_row, signs, H, c):
    """Element c of (x_row * signs) @ H (or of x_row, without signs) as an exact Fraction."""
    if signs is None:
        return Fraction(float(x_row[c]))
    return sum(Fraction(float(x_row[d])) * int(signs[d]) * int(H[d, c]) for d in range(len(x_row)))


def quantise_blocks(x, signs=None, block=TOKEN_BLOCK, granularity="block"):
    """Quantise x [B, S, H, D] (fp64 values) per (b, h, token block), or per tensor.

    ``signs``: length-D vector of +-1 to rotate with, or None for no rotation.
    ``granularity``: "block" (one scale per (b, h, 128-token block)) or "tensor" (one
    scale for the whole tensor, repeated in every block entry).
    Returns a dict with
      ``rotated`` [B,S,H,D]  the (rotated) values before scaling,
      ``scale``   [B,H,nblk] amax / 448 (1 for an all-zero block or tensor),
      ``pre``     [B,S,H,D]  x' / scale evaluated in fp64 (the value that is rounded),
      ``q``       [B,S,H,D]  the E4M3 value of each element (x' / scale rounded exactly),
      ``codes``   [B,S,H,D]  uint8 E4M3 bytes.
    """
    if granularity not in ("block", "tensor"):
        raise ValueError("granularity must be 'block' or 'tensor'")
    x = np.asarray(x, dtype=np.float64)
    B, S, H, D = x.shape
    sg = None if signs is None else np.asarray(signs, dtype=np.float64)
    Hm = None if signs is None else sylvester(D)
    if sg is not None:
        y = (x * sg) @ Hm                                           # unnormalised transform
        norm = 1.0 / np.sqrt(float(D))
        err = np.broadcast_to(D * 2.0 ** -53 * np.abs(x).sum(axis=-1, keepdims=True), x.shape)
    else:
        y, norm = x, 1.0
        err = np.zeros_like(x)
    nblk = (S + block - 1) // block
    ay = np.abs(y)
    scale = np.empty((B, H, nblk))
    amax_el = np.empty_like(y)          # the group (block or tensor) max |y| of each element
    err_el = np.empty_like(y)           # the group's largest error bound of y
    if granularity == "tensor":
        amax = ay.max() if y.size else 0.0
        scale[:] = amax * norm / E4M3_MAX if amax > 0 else 1.0
        amax_el[:] = amax
        err_el[:] = err.max() if y.size else 0.0
    else:
        for i in range(nblk):
            t0, t1 = i * block, min((i + 1) * block, S)
            amax = ay[:, t0:t1].max(axis=(1, 3))                    # [B, H]
            scale[:, :, i] = np.where(amax > 0, amax * norm / E4M3_MAX, 1.0)
            amax_el[:, t0:t1] = amax[:, None, :, None]
            err_el[:, t0:t1] = err[:, t0:t1].max(axis=(1, 3))[:, None, :, None]
    live = amax_el > 0
    den = np.where(live, amax_el, 1.0)
    pre = np.where(live, E4M3_MAX * y / den, 0.0)
    q = round_e4m3(pre)
    # bound on |pre - 448 y / amax(y)| (exact), and the elements whose decision it can flip
    dpre = 1.01 * E4M3_MAX * (err + np.abs(y) * 2 * err_el / den) / den + 2.0 ** -50 * np.abs(pre)
    step = grid_step(pre)
    t = np.abs(pre) / step
    near = live & (np.abs(t - np.floor(t) - 0.5) * step <= dpre + _NEAR * step)

    cache = {}

    def group_max(b, s, h):
        """Exact max |y| over the element's group, from the elements that can reach it."""
        if granularity == "tensor":
            key, off = "all", (0, 0, 0, 0)
            sub = ay
        else:
            t0 = s // block * block
            key, off = (b, t0, h), (b, t0, h, 0)
            sub = ay[b:b + 1, t0:min(S, t0 + block), h:h + 1]
        if key not in cache:
            cand = np.argwhere(sub >= amax_el[b, s, h, 0] - 2 * err_el[b, s, h, 0])
            best = Fraction(0)
            for c in cand:
                bb, ss, hh, cc = (int(c[i]) + off[i] for i in range(4))
                best = max(best, abs(_y_exact(x[bb, ss, hh], sg, Hm, cc)))
            cache[key] = best
        return cache[key]

    for b, s, h, c in np.argwhere(near):
        Y = _y_exact(x[b, s, h], sg, Hm, c)
        q[b, s, h, c] = rne_e4m3_fraction(Fraction(int(E4M3_MAX)) * Y / group_max(b, s, h))
    return {"rotated": y * norm, "scale": scale, "pre": pre, "q": q, "codes": encode(q)}


def dequantise(q, scale, block=TOKEN_BLOCK):
    """Values q [B,S,H,D] times their block's scale [B,H,nblk]."""
    q = np.asarray(q, dtype=np.float64)
    S = q.shape[1]
    tok_blk = np.arange(S) // block                              # [S]
    per_tok = np.transpose(scale, (0, 2, 1))[:, tok_blk, :]      # [B, S, H]
    return q * per_tok[..., None]
