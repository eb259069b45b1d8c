"""Pins for the attention-gradient oracle (CPU only).

The backward pass is plain calculus on the attention definition; its pins are independent of
the formulas in oracle/backward.py: central finite differences of the scalar
L = sum(dO * O) computed with the forward oracle (fp64, step 1e-6: truncation ~1e-12, rounding
~1e-10), torch fp64 autograd through scaled_dot_product_attention (a library routine), and
invariants: shifting every key by a common vector adds a constant to each row's logits,
which softmax ignores, so sum_j dK_j = 0 per (b, h); every row of P sums to one, so the
column sums of dV equal those of dO; with uniform V rows, O depends on neither Q nor K.
"""

import math

import numpy as np
import pytest
import torch

from oracle import attention, backward

RNG = np.random.default_rng(2024)


def loss(q, k, v, do, causal):
    o, _ = attention.attention(q, k, v, causal=causal)
    return float((o * do).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_matches_finite_differences(causal):
    B, S, H, D = 1, 9, 2, 4
    q, k, v, do = (RNG.standard_normal((B, S, H, D)) for _ in range(4))
    dq, dk, dv = backward.attention_backward(q, k, v, do, causal=causal)
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        for idx in [(0, 0, 0, 0), (0, 3, 1, 2), (0, 8, 0, 3), (0, 5, 1, 1)]:
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [xp if y is x else y for y in (q, k, v)]
            args_m = [xm if y is x else y for y in (q, k, v)]
            fd = (loss(*args_p, do, causal) - loss(*args_m, do, causal)) / (2 * eps)
            assert abs(fd - g[idx]) < 1e-7, (idx, fd, g[idx])


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_autograd(causal):
    B, S, H, D = 2, 70, 3, 16
    q, k, v, do = (RNG.standard_normal((B, S, H, D)) for _ in range(4))
    dq, dk, dv = backward.attention_backward(q, k, v, do, causal=causal)
    t = [torch.from_numpy(np.ascontiguousarray(x.transpose(0, 2, 1, 3))).requires_grad_(True) for x in (q, k, v)]
    o = torch.nn.functional.scaled_dot_product_attention(*t, is_causal=causal, scale=1 / math.sqrt(D))
    o.backward(torch.from_numpy(np.ascontiguousarray(do.transpose(0, 2, 1, 3))))
    for mine, ref in ((dq, t[0]), (dk, t[1]), (dv, t[2])):
        np.testing.assert_allclose(mine, ref.grad.numpy().transpose(0, 2, 1, 3), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_invariants(causal):
    B, S, H, D = 1, 40, 2, 8
    q, k, v, do = (RNG.standard_normal((B, S, H, D)) for _ in range(4))
    dq, dk, dv = backward.attention_backward(q, k, v, do, causal=causal)
    # a common shift of every key leaves each row's softmax unchanged
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    # every row of P sums to one, so dV's column sums equal dO's
    np.testing.assert_allclose(dv.sum(axis=1), do.sum(axis=1), atol=1e-12)
    # uniform V rows: O does not depend on Q or K at all
    vu = np.broadcast_to(RNG.standard_normal((1, 1, H, D)), v.shape).copy()
    dq0, dk0, _ = backward.attention_backward(q, k, vu, do, causal=causal)
    np.testing.assert_allclose(dq0, 0.0, atol=1e-12)
    np.testing.assert_allclose(dk0, 0.0, atol=1e-12)


def test_single_key_row_has_no_query_gradient():
    # causal row 0 sees only key 0: P = 1, dS = 0 for that row
    B, S, H, D = 1, 6, 1, 4
    q, k, v, do = (RNG.standard_normal((B, S, H, D)) for _ in range(4))
    dq, _, _ = backward.attention_backward(q, k, v, do, causal=True)
    np.testing.assert_allclose(dq[0, 0], 0.0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_gradients_match_finite_differences(causal):
    # the loss sum(dO * O) of grouped-query attention, differentiated numerically
    from oracle import gqa
    rng = np.random.default_rng(5)
    B, S, Hq, Hkv, D = 1, 6, 4, 2, 3
    q, do = rng.standard_normal((B, S, Hq, D)), rng.standard_normal((B, S, Hq, D))
    k, v = rng.standard_normal((B, S, Hkv, D)), rng.standard_normal((B, S, Hkv, D))
    dq, dk, dv = backward.attention_backward_gqa(q, k, v, do, 0.7, causal)
    loss = lambda q_, k_, v_: float((gqa.attention_gqa(q_, k_, v_, 0.7, causal)[0] * do).sum())
    h = 1e-6
    for arr, grad, idx in ((q, dq, (0, 3, 2, 1)), (k, dk, (0, 1, 1, 2)), (v, dv, (0, 4, 0, 0)), (k, dk, (0, 5, 0, 1))):
        plus, minus = arr.copy(), arr.copy()
        plus[idx] += h
        minus[idx] -= h
        args_p = [plus if a is arr else a for a in (q, k, v)]
        args_m = [minus if a is arr else a for a in (q, k, v)]
        fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (idx, fd, grad[idx])


def test_gqa_with_one_group_per_head_is_the_plain_backward():
    rng = np.random.default_rng(6)
    q, k, v, do = (rng.standard_normal((2, 9, 3, 4)) for _ in range(4))
    a = backward.attention_backward_gqa(q, k, v, do, causal=True)
    b = backward.attention_backward(q, k, v, do, causal=True)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_rows_equal_the_full_gradients(causal):
    B, S, H, D = 2, 300, 2, 32
    rng = np.random.default_rng(31)
    q, k, v, do = (rng.standard_normal((B, S, H, D)) for _ in range(4))
    full = backward.attention_backward(q, k, v, do, causal=causal)
    qr, kr = np.array([0, 1, 127, 128, 299]), np.array([0, 5, 150, 298, 299])
    dq, dk, dv = backward.attention_backward_rows(q, k, v, do, qr, kr, causal=causal)
    np.testing.assert_allclose(dq, full[0][:, qr], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk, full[1][:, kr], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, full[2][:, kr], rtol=1e-11, atol=1e-12)
