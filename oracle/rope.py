"""Rotary position embedding (RoPE) of Q and K, fp64, and its fusion with the FP8 quantiser.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: hada.io FA3 summary, "Niedrige FP8-Präzision und incoherent processing":
the Hadamard transform is memory-bandwidth-bound, and fused with a preceding
operation that is memory-bandwidth-bound as well -- rotary embedding is the
pages' example -- it costs nothing extra.  The pages name rotary embedding
but do not define it.

Reading (the original definition, Su et al., "RoFormer: Enhanced Transformer
with Rotary Position Embedding", 2021, section 3.2): a D-element row at token
position p is split into the D/2 consecutive pairs (x[2i], x[2i+1]), and pair i
is turned by the angle p * theta_i, theta_i = base^(-2i/D), base = 10000:

    x'[2i]   = x[2i] cos(p theta_i) - x[2i+1] sin(p theta_i)
    x'[2i+1] = x[2i] sin(p theta_i) + x[2i+1] cos(p theta_i)

Position p of the token at index s of a [B, S, H, D] tensor is s (every
sequence starts at 0).  RoPE is applied to Q and K, not to V.  Fused with the
FP8 path, each Q/K row becomes  quantise((rope(x) * signs) H_D / sqrt(D)):
rotary embedding first, then the random-sign Hadamard rotation, then the
per-block quantiser, with no rounding in between.
"""

import numpy as np

from .quantise import quantise_blocks

__all__ = ["DEFAULT_BASE", "theta", "angles", "cos_sin_table", "rope", "rope_quantise_blocks"]

DEFAULT_BASE = 10000.0


def theta(D, base=DEFAULT_BASE):
    """Frequencies theta_i = base^(-2i/D), i = 0 .. D/2 - 1."""
    if D < 2 or D % 2:
        raise ValueError("D must be even")
    i = np.arange(D // 2, dtype=np.float64)
    return float(base) ** (-2.0 * i / D)


def angles(n_pos, D, base=DEFAULT_BASE):
    """[n_pos, D/2] angles p * theta_i for p = 0 .. n_pos - 1."""
    p = np.arange(n_pos, dtype=np.float64)
    return p[:, None] * theta(D, base)[None, :]


def cos_sin_table(n_pos, D, base=DEFAULT_BASE):
    """[n_pos, D/2, 2]: (cos, sin) of p * theta_i."""
    a = angles(n_pos, D, base)
    return np.stack([np.cos(a), np.sin(a)], axis=-1)


def rope(x, base=DEFAULT_BASE):
    """Rotary embedding of x [B, S, H, D] (fp64), positions 0 .. S-1 along axis 1."""
    x = np.asarray(x, dtype=np.float64)
    B, S, H, D = x.shape
    a = angles(S, D, base)[None, :, None, :]        # [1, S, 1, D/2]
    c, s = np.cos(a), np.sin(a)
    even, odd = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = even * c - odd * s
    out[..., 1::2] = even * s + odd * c
    return out


def rope_quantise_blocks(x, signs=None, base=DEFAULT_BASE):
    """Rotary embedding, then the (optionally rotated) per-block E4M3 quantiser of
    ``quantise.quantise_blocks`` on the result; same return dict."""
    return quantise_blocks(rope(x, base), signs)
