"""Seeded synthetic inputs, shared by the tests, the bench and the oracle runs.

This module holds no attention, rotation or quantisation arithmetic: it only
draws numbers.  Recipe (the pages' own experiment, hada.io FA3 summary,
"Niedrige FP8-Präzision und incoherent processing": Q, K, V drawn from a
standard normal distribution, with 0.1 % of the entries given a large
magnitude to simulate outliers):

* counter-based SplitMix64 (Steele, Lea & Flood 2014): the i-th 64-bit word
  of stream ``seed`` is mix(seed + (i + 1) * 0x9E3779B97F4A7C15);
* uniform in (0, 1): the top 53 bits, offset by half a unit;
* normal: Box-Muller in fp64 on the two 32-bit halves of one word, each
  taken as (half + 0.5) * 2^-32, then rounded to fp32;
* ``outliers``: each entry independently, with probability 1e-3, is replaced
  by an independent N(0, sigma = 10) draw;
* bf16 tensors are the fp32 draws rounded to nearest even (torch's cast).

Seeds: ``seed_for(case, stream)`` = 0xA77E000 + 16 * case + stream, with
streams 0 = Q, 1 = K, 2 = V, 3 = Hadamard signs, 4 = outlier mask,
5 = outlier values, 6 = sequence lengths of a packed batch.
"""

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

__all__ = ["seed_for", "uniform", "normal", "normal_with_outliers", "signs", "seqlens",
           "make_qkv", "STREAM_Q", "STREAM_K", "STREAM_V", "STREAM_SIGNS"]

STREAM_Q, STREAM_K, STREAM_V, STREAM_SIGNS, STREAM_OUT_MASK, STREAM_OUT_VAL, STREAM_LENGTHS = range(7)
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 21
_POOL = ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))


def seed_for(case, stream):
    """Seed of one input stream of one test / bench case."""
    return 0xA77E000 + 16 * int(case) + int(stream)


def _splitmix64(counter, seed):
    z = np.uint64(seed) + (counter + np.uint64(1)) * _GOLDEN
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _chunks(n):
    return [(c0, min(n, c0 + _CHUNK)) for c0 in range(0, n, _CHUNK)]


def uniform(shape, seed):
    """fp64 uniforms in (0, 1), deterministic in (shape, seed)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float64)

    def fill(c):
        ctr = np.arange(c[0], c[1], dtype=np.uint64)
        w = _splitmix64(ctr, seed)
        out[c[0]:c[1]] = ((w >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)

    list(_POOL.map(fill, _chunks(n)))
    return out.reshape(shape)


def normal(shape, seed):
    """fp32 standard normals by Box-Muller on SplitMix64 words."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)

    def fill(c):
        ctr = np.arange(c[0], c[1], dtype=np.uint64)
        w = _splitmix64(ctr, seed)
        u1 = ((w >> np.uint64(32)).astype(np.float64) + 0.5) * (2.0 ** -32)
        u2 = ((w & np.uint64(0xFFFFFFFF)).astype(np.float64) + 0.5) * (2.0 ** -32)
        np.log(u1, out=u1)
        u1 *= -2.0
        np.sqrt(u1, out=u1)
        u2 *= 2.0 * np.pi
        np.cos(u2, out=u2)
        u1 *= u2
        out[c[0]:c[1]] = u1

    list(_POOL.map(fill, _chunks(n)))
    return out.reshape(shape)


def normal_with_outliers(shape, seed_base, prob=1e-3, sigma=10.0, case_streams=None):
    """N(0,1) draws where each entry, w.p. ``prob``, is replaced by N(0, sigma).

    ``seed_base`` is the stream seed of the tensor's own normals; the outlier
    mask and values use ``case_streams`` = (mask_seed, value_seed), derived
    from it when not given.
    """
    x = normal(shape, seed_base)
    if case_streams is None:
        case_streams = ((seed_base << 8) | 0x41, (seed_base << 8) | 0x42)
    mask = uniform(shape, case_streams[0]) < prob
    big = normal(shape, case_streams[1]) * np.float32(sigma)
    return np.where(mask, big, x).astype(np.float32)


def signs(D, seed):
    """fp32 vector of D random signs (+1 / -1)."""
    return np.where(uniform((D,), seed) < 0.5, 1.0, -1.0).astype(np.float32)


def seqlens(total, lo, hi, seed):
    """Sequence lengths drawn uniformly from the integers lo .. hi until they sum to ``total``
    (the last one cut short); returns (lengths, cu_seqlens) as int32 numpy arrays."""
    u = uniform((total // max(lo, 1) + 1,), seed)
    lens, acc = [], 0
    while acc < total:
        n = min(lo + int(u[len(lens)] * (hi - lo + 1)), total - acc)
        lens.append(n)
        acc += n
    lens = np.array(lens, dtype=np.int32)
    return lens, np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def make_qkv(B, S, H, D, case, dist="normal", dtype=torch.bfloat16):
    """Q, K, V as CPU torch tensors [B, S, H, D] (bf16 by default).

    dist: "normal" (N(0,1)) or "outliers" (N(0,1) with 0.1 % N(0, 10) entries).
    """
    out = []
    for stream in (STREAM_Q, STREAM_K, STREAM_V):
        sd = seed_for(case, stream)
        if dist == "normal":
            x = normal((B, S, H, D), sd)
        elif dist == "outliers":
            x = normal_with_outliers((B, S, H, D), sd, case_streams=(
                (seed_for(case, STREAM_OUT_MASK) << 4) | stream,
                (seed_for(case, STREAM_OUT_VAL) << 4) | stream))
        else:
            raise ValueError(f"unknown distribution {dist!r}")
        out.append(torch.from_numpy(x).to(dtype))
    return tuple(out)
