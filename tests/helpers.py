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


def inputs(B, S, H, D, case, dist="normal"):
    return synth.make_qkv(B, S, H, D, case, dist)
