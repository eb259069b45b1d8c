"""Pins for the grouped-query / decoding oracle (CPU only).

Independent references: torch fp64 scaled_dot_product_attention with each key/value head
repeated G times and an explicit bottom-right causal mask (a library routine), the
fixed-length definition when G = 1 and S_q = S_k (torch's own is_causal), closed forms (zero
queries give the mean of the visible values with lse = ln(count); one query token under the
mask sees every key), and that query heads of one group read the same values.
"""

import math

import numpy as np
import pytest
import torch

from oracle import gqa

RNG = np.random.default_rng(31)


def _sdpa(q, k, v, G, mask):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a.transpose(0, 2, 1, 3)))
    kk = t(np.repeat(k, G, axis=2))
    vv = t(np.repeat(v, G, axis=2))
    o = torch.nn.functional.scaled_dot_product_attention(t(q), kk, vv, attn_mask=torch.from_numpy(mask),
                                                         scale=1 / math.sqrt(q.shape[-1]))
    return o.numpy().transpose(0, 2, 1, 3)


@pytest.mark.parametrize("Sq,Sk,Hq,Hkv", [(1, 300, 8, 2), (5, 64, 6, 3), (16, 16, 4, 1), (3, 130, 4, 4)])
@pytest.mark.parametrize("causal", [False, True])
def test_matches_sdpa_with_repeated_heads(Sq, Sk, Hq, Hkv, causal):
    D = 16
    q = RNG.standard_normal((2, Sq, Hq, D))
    k, v = RNG.standard_normal((2, Sk, Hkv, D)), RNG.standard_normal((2, Sk, Hkv, D))
    mask = np.ones((Sq, Sk), dtype=bool)
    if causal:
        mask = np.tril(np.ones((Sq, Sk), dtype=bool), k=Sk - Sq)
    O, lse = gqa.attention_gqa(q, k, v, causal=causal)
    np.testing.assert_allclose(O, _sdpa(q, k, v, Hq // Hkv, mask), atol=1e-12)


def test_equal_lengths_single_group_is_plain_causal_attention():
    q, k, v = (RNG.standard_normal((1, 40, 2, 8)) for _ in range(3))
    O, _ = gqa.attention_gqa(q, k, v, causal=True)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a.transpose(0, 2, 1, 3)))
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True).numpy().transpose(0, 2, 1, 3)
    np.testing.assert_allclose(O, ref, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_and_group_sharing(causal):
    B, Sq, Sk, Hq, Hkv, D = 1, 4, 50, 6, 2, 8
    k, v = RNG.standard_normal((B, Sk, Hkv, D)), RNG.standard_normal((B, Sk, Hkv, D))
    O, lse = gqa.attention_gqa(np.zeros((B, Sq, Hq, D)), k, v, causal=causal)
    for i in range(Sq):
        n = Sk - Sq + i + 1 if causal else Sk
        for h in range(Hq):
            np.testing.assert_allclose(O[0, i, h], v[0, :n, h // 3].mean(axis=0), atol=1e-13)
            np.testing.assert_allclose(lse[0, h, i], math.log(n), atol=1e-13)


def test_single_decode_token_sees_every_key():
    q = RNG.standard_normal((2, 1, 4, 8))
    k, v = RNG.standard_normal((2, 33, 2, 8)), RNG.standard_normal((2, 33, 2, 8))
    a, la = gqa.attention_gqa(q, k, v, causal=True)
    b, lb = gqa.attention_gqa(q, k, v, causal=False)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


def test_rejects_bad_shapes():
    with pytest.raises(ValueError):
        gqa.attention_gqa(np.zeros((1, 2, 3, 4)), np.zeros((1, 2, 2, 4)), np.zeros((1, 2, 2, 4)))
    with pytest.raises(ValueError):
        gqa.attention_gqa(np.zeros((1, 5, 2, 4)), np.zeros((1, 4, 2, 4)), np.zeros((1, 4, 2, 4)))


@pytest.mark.parametrize("causal", [False, True])
def test_rounded_numerators_match_the_fp8_path_at_one_group(causal):
    # G = 1 and Sq = Sk: the same computation as fp8_path.attention_rounded_p
    from oracle import fp8_path
    q, k, v = (RNG.standard_normal((2, 50, 3, 16)) for _ in range(3))
    a, la = gqa.attention_gqa(q, k, v, causal=causal, round_p=True)
    b, lb = fp8_path.attention_rounded_p(q, k, v, 1 / math.sqrt(16), causal)
    np.testing.assert_allclose(a, b, atol=1e-13)
    np.testing.assert_allclose(la, lb, atol=1e-13)
    c, _ = gqa.attention_gqa(q, k, v, causal=causal)
    assert np.abs(a - c).max() > 1e-4          # the rounding does change O
