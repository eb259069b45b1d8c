"""The FP8 E4M3 number format, written from its definition (fp64 arithmetic).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages only say "FP8" ("FlashAttention-3 (NL)", "Nieuwe
hardwaremogelijkheden": an 8-bit floating-point format with limited dynamic
range; hada.io summary, "Hopper-GPU-Funktionen: WGMMA, TMA, FP8").  The
reading taken here is E4M3 as defined for 8-bit floating point on NVIDIA
tensor cores: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no
infinities, the single NaN pattern S.1111.111, so the largest finite value
is 1.75 * 2^8 = 448.  Normal values are (1 + m/8) * 2^(E-7) for E = 1..15;
subnormals (E = 0) are m * 2^-9.  Conversion from a wider type rounds to
nearest, ties to even, and saturates to +-448 ("satfinite").
"""

import numpy as np

__all__ = ["E4M3_MAX", "decode", "round_e4m3", "encode"]

E4M3_MAX = 448.0
_MIN_NORMAL_EXP = -6          # smallest normal value is 2^-6
_SUBNORMAL_QUANTUM = 2.0 ** -9


def decode(codes):
    """Value (fp64) of each E4M3 byte in ``codes`` (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    E = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2((E - 7).astype(np.float64))
    sub = m * _SUBNORMAL_QUANTUM
    val = np.where(E == 0, sub, normal)
    val = np.where((E == 15) & ((c & 0x7) == 7), np.nan, val)
    return sign * val


def _quantum(ax):
    """Spacing of E4M3 values in the binade of |x| (2^(e-3), or 2^-9 below 2^-6)."""
    _, ex = np.frexp(ax)              # ax = f * 2^ex, f in [0.5, 1)  =>  floor(log2 ax) = ex - 1
    e = np.maximum(ex - 1, _MIN_NORMAL_EXP)
    return np.exp2((e - 3).astype(np.float64))


def round_e4m3(x):
    """Round fp64 values to the nearest E4M3 value (ties to even), saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    q = _quantum(np.where(ax > 0, ax, 1.0))
    y = np.rint(ax / q) * q           # np.rint rounds half to even; /q is exact (power of two)
    y = np.minimum(y, E4M3_MAX)
    y = np.where(ax > 0, y, 0.0)
    out = np.copysign(y, x)
    return np.where(np.isnan(x), np.nan, out)


def encode(x):
    """E4M3 byte codes of fp64 values (round to nearest even, saturating)."""
    y = round_e4m3(x)
    sign = np.where(np.signbit(y), 0x80, 0).astype(np.int64)
    ay = np.abs(y)
    code = np.zeros(ay.shape, dtype=np.int64)
    sub = (ay > 0) & (ay < 2.0 ** _MIN_NORMAL_EXP)
    code = np.where(sub, np.rint(ay / _SUBNORMAL_QUANTUM).astype(np.int64), code)
    norm = ay >= 2.0 ** _MIN_NORMAL_EXP
    _, ex = np.frexp(np.where(norm, ay, 1.0))
    e = ex - 1
    mant = np.rint((np.where(norm, ay, 1.0) / np.exp2(e.astype(np.float64)) - 1.0) * 8.0).astype(np.int64)
    code = np.where(norm, ((e + 7) << 3) | mant, code)
    code = np.where(np.isnan(y), 0x7F, code)
    return (code | sign).astype(np.uint8)
