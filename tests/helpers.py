"""Shared helpers for the GPU parity tests: seeded inputs, row sampling, error statistics."""

import numpy as np
import torch

from exact_attention_46_gb300 import synth

# Tolerances of the BF16 path against the fp64 oracle (N(0,1) inputs, D <= 128):
#   max |O - O_ref| - half_ulp_bf16(O_ref) <= 1e-2   (the error beyond the unavoidable rounding
#                                                     of the exact result to the bf16 output;
#                                                     at |O| >= 4 that rounding alone is 0.0156)
#   RMS(O - O_ref) <= 2e-3,  max |lse - lse_ref| <= 1e-3.
BF16_MAX_ABS = 1e-2
BF16_RMS = 2e-3
LSE_MAX_ABS = 1e-3


def half_ulp_bf16(x):
    """Half the spacing of bf16 values at |x| (8 significant bits)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    _, ex = np.frexp(np.where(ax > 0, ax, 1.0))          # ax = f * 2^ex, f in [0.5, 1)
    return np.where(ax > 0, np.exp2((ex - 1 - 8).astype(np.float64)), 0.0)


def sample_rows(S, n_random=24, seed=0):
    """Query rows checked at large S: tile edges, both ends, and seeded random rows."""
    fixed = {0, 1, 63, 127, 128, 129, 255, 256, 257, S // 2, S - 129, S - 128, S - 2, S - 1}
    rng = np.random.default_rng(seed + S)
    rnd = set(rng.integers(0, S, size=n_random).tolist())
    return np.array(sorted(r for r in fixed | rnd if 0 <= r < S), dtype=np.int64)


def to64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def stats(gpu, ref):
    err = gpu - ref
    return float(np.abs(err).max()), float(np.sqrt(np.mean(err ** 2)))


def bf16_stats(gpu, ref):
    """(max error beyond the bf16 output rounding, RMS error, raw max error)."""
    err = np.abs(gpu - ref)
    return float((err - half_ulp_bf16(ref)).max()), float(np.sqrt(np.mean(err ** 2))), float(err.max())


def check_codes(gpu_codes, ref, tie_rtol, tie_atol):
    """E4M3 codes vs the oracle's: equal, except where the oracle's pre-rounding quotient lies
    within tie_rtol * |pre| + tie_atol of a rounding midpoint (the oracle decides midpoints
    exactly, ties to even; a kernel working in fp32 may land on either side); there the two
    codes must be the neighbouring grid values around that midpoint.  Returns the number of
    differing codes."""
    from oracle import e4m3
    diff = gpu_codes != ref["codes"]
    n_diff = int(diff.sum())
    if n_diff:
        pre = ref["pre"][diff]
        a = e4m3.decode(gpu_codes[diff])
        b = e4m3.decode(ref["codes"][diff])
        mid = (a + b) / 2
        assert np.all(np.abs(pre - mid) <= tie_rtol * np.abs(pre) + tie_atol), "non-tie code mismatch"
        # neighbours on the grid: nothing representable strictly between them
        lo, hi = np.minimum(a, b), np.maximum(a, b)
        assert np.all(e4m3.round_e4m3((lo + mid) / 2) == lo) and np.all(e4m3.round_e4m3((hi + mid) / 2) == hi)
    assert not np.any((gpu_codes & 0x7F) == 0x7F), "NaN code produced"
    return n_diff


def inputs(B, S, H, D, case, dist="normal"):
    return synth.make_qkv(B, S, H, D, case, dist)
