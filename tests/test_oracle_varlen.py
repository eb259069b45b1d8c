"""Pins for the variable-length (packed batch) attention oracle (CPU only).

The pages name variable-length sequences (hada.io FA3 summary, "Weitere Optimierungen und
künftige Integration") without defining them; the reading is a packed batch in which every
sequence attends only to itself.  Pins: a library routine on a different formulation (torch
fp64 scaled_dot_product_attention over the whole packed axis with a block-diagonal mask),
closed forms at the segment boundaries (zero queries give the mean of the sequence's visible
values and lse = ln(count); per-sequence constant values come back exactly, so nothing leaks
across sequences), single-token and empty sequences, and sampled rows.
"""

import math

import numpy as np
import pytest
import torch

from oracle import varlen

RNG = np.random.default_rng(777)
CU = [0, 5, 5, 133, 134, 390, 391, 600]          # lengths 5, 0, 128, 1, 256, 1, 209


def _packed(total, H, D):
    return (RNG.standard_normal((total, H, D)) for _ in range(3))


@pytest.mark.parametrize("causal", [False, True])
def test_matches_block_diagonal_sdpa(causal):
    H, D = 2, 16
    q, k, v = _packed(CU[-1], H, D)
    O, lse = varlen.attention_varlen(q, k, v, CU, causal=causal)
    seg = np.zeros(CU[-1], dtype=np.int64)
    pos = np.zeros(CU[-1], dtype=np.int64)
    for s, (s0, n) in enumerate(varlen.segments(CU)):
        seg[s0:s0 + n] = s
        pos[s0:s0 + n] = np.arange(n)
    allowed = seg[:, None] == seg[None, :]
    if causal:
        allowed &= pos[None, :] <= pos[:, None]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a.transpose(1, 0, 2)))[None]
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=torch.from_numpy(allowed)[None, None],
                                                           scale=1 / math.sqrt(D))[0].numpy().transpose(1, 0, 2)
    np.testing.assert_allclose(O, ref, atol=1e-12)
    s = np.einsum("ihd,jhd->hij", q, k) / math.sqrt(D)
    s = np.where(allowed[None], s, -np.inf)
    np.testing.assert_allclose(lse, torch.logsumexp(torch.from_numpy(s), dim=-1).numpy(), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_the_mean_of_visible_values(causal):
    H, D = 3, 8
    _, k, v = _packed(CU[-1], H, D)
    q = np.zeros_like(k)
    O, lse = varlen.attention_varlen(q, k, v, CU, causal=causal)
    for s0, n in varlen.segments(CU):
        for i in range(n):
            vis = v[s0:s0 + (i + 1 if causal else n)]
            np.testing.assert_allclose(O[s0 + i], vis.mean(axis=0), atol=1e-13)
            np.testing.assert_allclose(lse[:, s0 + i], math.log(len(vis)), atol=1e-13)


def test_constant_values_per_sequence_do_not_leak():
    H, D = 2, 8
    q, k, _ = _packed(CU[-1], H, D)
    v = np.empty((CU[-1], H, D))
    for s, (s0, n) in enumerate(varlen.segments(CU)):
        v[s0:s0 + n] = 10.0 * s + np.arange(D)
    for causal in (False, True):
        O, _ = varlen.attention_varlen(q, k, v, CU, causal=causal)
        for s, (s0, n) in enumerate(varlen.segments(CU)):
            np.testing.assert_allclose(O[s0:s0 + n], np.broadcast_to(10.0 * s + np.arange(D), (n, H, D)), atol=1e-12)


def test_single_token_sequence_and_sampled_rows():
    H, D = 2, 16
    q, k, v = _packed(CU[-1], H, D)
    O, lse = varlen.attention_varlen(q, k, v, CU)
    np.testing.assert_allclose(O[133], v[133], atol=1e-15)               # the 1-token sequence
    np.testing.assert_allclose(lse[:, 133], np.einsum("hd,hd->h", q[133], k[133]) / math.sqrt(D), atol=1e-13)
    rows = np.array([0, 4, 5, 132, 133, 134, 389, 390, 599])
    Os, ls = varlen.attention_varlen(q, k, v, CU, rows=rows)
    np.testing.assert_allclose(Os, O[rows], atol=1e-13)       # BLAS may sum a subset differently
    np.testing.assert_allclose(ls, lse[:, rows], atol=1e-13)


def test_rejects_bad_offsets():
    q = np.zeros((10, 1, 4))
    for cu in ([1, 10], [0, 6, 4, 10], [0, 9]):
        with pytest.raises(ValueError):
            varlen.attention_varlen(q, q, q, cu)
