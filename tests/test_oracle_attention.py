"""Pins for the fp64 attention oracle (CPU only).

Each test checks the oracle against something other than itself: a closed
form, an invariant of softmax attention, a library routine (torch's fp64 CPU
scaled_dot_product_attention), a blockwise recomputation (the tiling +
softmax-rescaling argument of the hada.io FA3 summary, "Rückblick auf den
FlashAttention-Ansatz"), or brute force on tiny inputs.
"""

import math

import numpy as np
import pytest
import torch

from oracle import attention as A

RNG = np.random.default_rng(1234)


def rand(*shape):
    return RNG.standard_normal(shape)


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_value_rows_return_that_row(causal):
    B, S, H, D = 2, 37, 3, 16
    q, k = rand(B, S, H, D), rand(B, S, H, D)
    u = rand(B, 1, H, D)
    v = np.broadcast_to(u, (B, S, H, D)).copy()
    O, _ = A.attention(q, k, v, causal=causal)
    np.testing.assert_allclose(O, np.broadcast_to(u, O.shape), rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_mean_of_visible_values(causal):
    B, S, H, D = 1, 50, 2, 8
    q = np.zeros((B, S, H, D))
    k, v = rand(B, S, H, D), rand(B, S, H, D)
    O, lse = A.attention(q, k, v, causal=causal)
    for i in range(S):
        n = i + 1 if causal else S
        np.testing.assert_allclose(O[:, i], v[:, :n].mean(axis=1), atol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], math.log(n), atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_rows_sum_to_one_and_mask_is_exact(causal):
    S, D = 64, 16
    q, k = rand(S, D), rand(S, D)
    P, m, l = A.attention_weights(q, k, 0.3, causal)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-15)
    assert (P >= 0).all()
    if causal:
        assert (P[np.triu_indices(S, 1)] == 0).all()
        assert (P[np.tril_indices(S)] > 0).all()


def test_single_key_and_causal_first_row():
    D = 8
    q, k, v = rand(1, 1, 1, D), rand(1, 1, 1, D), rand(1, 1, 1, D)
    O, lse = A.attention(q, k, v, scale=0.7)
    np.testing.assert_allclose(O, v, atol=1e-15)
    np.testing.assert_allclose(lse[0, 0, 0], 0.7 * float(q.ravel() @ k.ravel()), atol=1e-14)
    q, k, v = rand(1, 9, 2, D), rand(1, 9, 2, D), rand(1, 9, 2, D)
    O, lse = A.attention(q, k, v, scale=0.7, causal=True)
    np.testing.assert_allclose(O[:, 0], v[:, 0], atol=1e-15)
    np.testing.assert_allclose(lse[0, :, 0], 0.7 * np.einsum("hd,hd->h", q[0, 0], k[0, 0]), atol=1e-14)


def test_two_keys_hand_computed():
    # logits 0 and ln 3 -> weights 1/4, 3/4; O = 1/4 * 1 + 3/4 * 5 = 4; lse = ln 4
    q = np.array([1.0]).reshape(1, 1, 1, 1)
    k = np.array([0.0, math.log(3.0)]).reshape(1, 2, 1, 1)
    v = np.array([1.0, 5.0]).reshape(1, 2, 1, 1)
    O, lse = A.attention(q, k, v, scale=1.0, rows=[0])
    assert abs(O[0, 0, 0, 0] - 4.0) < 1e-14
    assert abs(lse[0, 0, 0] - math.log(4.0)) < 1e-14


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S,D", [(1, 4), (7, 8), (130, 64), (257, 32)])
def test_matches_torch_sdpa_fp64(S, D, causal):
    B, H = 2, 3
    q, k, v = rand(B, S, H, D), rand(B, S, H, D), rand(B, S, H, D)
    sc = 1.0 / math.sqrt(D)
    O, lse = A.attention(q, k, v, scale=sc, causal=causal)
    t = lambda x: torch.from_numpy(x).permute(0, 2, 1, 3)  # [B,H,S,D]
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=causal, scale=sc)
    np.testing.assert_allclose(O, ref.permute(0, 2, 1, 3).numpy(), atol=1e-12)
    s = torch.einsum("bhid,bhjd->bhij", t(q), t(k)) * sc
    if causal:
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block", [1, 16, 128])
def test_blockwise_online_softmax_equals_full_softmax(causal, block):
    B, S, H, D = 1, 300, 2, 32   # 300 = 2 full 128-blocks + a ragged tail
    q, k, v = rand(B, S, H, D) * 2, rand(B, S, H, D) * 2, rand(B, S, H, D)
    O1, l1 = A.attention(q, k, v, causal=causal)
    O2, l2 = A.online_softmax_attention(q, k, v, causal=causal, block=block)
    np.testing.assert_allclose(O1, O2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-12)


def test_brute_force_loops_tiny():
    B, S, H, D = 1, 5, 2, 3
    q, k, v = rand(B, S, H, D), rand(B, S, H, D), rand(B, S, H, D)
    for causal in (False, True):
        O, lse = A.attention(q, k, v, scale=0.9, causal=causal)
        for h in range(H):
            for i in range(S):
                keys = range(i + 1) if causal else range(S)
                logit = {j: 0.9 * sum(q[0, i, h, d] * k[0, j, h, d] for d in range(D)) for j in keys}
                w = {j: math.exp(x) for j, x in logit.items()}
                z = sum(w.values())
                for d in range(D):
                    assert abs(O[0, i, h, d] - sum(w[j] * v[0, j, h, d] for j in keys) / z) < 1e-13
                assert abs(lse[0, h, i] - math.log(z)) < 1e-13


def test_key_permutation_invariance_noncausal():
    B, S, H, D = 1, 40, 2, 8
    q, k, v = rand(B, S, H, D), rand(B, S, H, D), rand(B, S, H, D)
    perm = RNG.permutation(S)
    O1, l1 = A.attention(q, k, v)
    O2, l2 = A.attention(q, k[:, perm], v[:, perm])
    np.testing.assert_allclose(O1, O2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def test_logit_shift_invariance():
    # k_j -> k_j + w shifts every logit of row i by scale * q_i.w: O unchanged, lse shifted.
    B, S, H, D = 1, 33, 1, 8
    q, k, v = rand(B, S, H, D), rand(B, S, H, D), rand(B, S, H, D)
    w = rand(D)
    O1, l1 = A.attention(q, k, v, scale=0.5, causal=True)
    O2, l2 = A.attention(q, k + w, v, scale=0.5, causal=True)
    np.testing.assert_allclose(O1, O2, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, 0.5 * (q[0, :, 0, :] @ w)[None, None, :], atol=1e-12)


def test_row_sampling_matches_full_rows():
    B, S, H, D = 2, 200, 2, 16
    q, k, v = rand(B, S, H, D), rand(B, S, H, D), rand(B, S, H, D)
    rows = np.array([0, 5, 127, 128, 199])
    for causal in (False, True):
        O, lse = A.attention(q, k, v, causal=causal)
        Os, lses = A.attention(q, k, v, causal=causal, rows=rows)
        np.testing.assert_allclose(O[:, rows], Os, atol=1e-14)
        np.testing.assert_allclose(lse[:, :, rows], lses, atol=1e-14)
