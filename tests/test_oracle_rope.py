"""Pins for the rotary-embedding oracle (CPU only).

Rotary embedding is not defined on the pages (hada.io FA3 summary, "Niedrige
FP8-Präzision und incoherent processing", names it only as the memory-bound op
to fuse the rotation with); the oracle follows RoFormer (Su et al., 2021,
section 3.2).  Its pins: closed-form angles (theta_0 = 1, so pair 0 turns by
exactly p radians; at D = 4, base 10^4, pair 1 turns by p / 100 radians), the
turning direction, the identity at p = 0, norm preservation, the defining
relative-position property, and invariance of QK^T under the Hadamard rotation
applied after it.
"""

import math

import numpy as np
import pytest

from oracle import hadamard, quantise, rope

RNG = np.random.default_rng(4242)


def _rows_at(x_row, S, D):
    """[1, S, 1, D] tensor holding the same row at every position."""
    return np.broadcast_to(np.asarray(x_row, dtype=np.float64), (1, S, 1, D)).copy()


def test_direction_and_angle_of_pair_zero():
    # D = 2: theta_0 = 1 for any base, so position p turns the pair by p radians,
    # counter-clockwise: (1, 0) -> (cos p, sin p) and (0, 1) -> (-sin p, cos p).
    for p in (1, 2, 7, 100):
        a = rope.rope(_rows_at([1.0, 0.0], p + 1, 2))[0, p, 0]
        b = rope.rope(_rows_at([0.0, 1.0], p + 1, 2))[0, p, 0]
        np.testing.assert_allclose(a, [math.cos(p), math.sin(p)], atol=1e-15)
        np.testing.assert_allclose(b, [-math.sin(p), math.cos(p)], atol=1e-15)
    # p = 1 written out: cos 1 = 0.5403023058681398, sin 1 = 0.8414709848078965
    a = rope.rope(_rows_at([1.0, 0.0], 2, 2))[0, 1, 0]
    np.testing.assert_allclose(a, [0.5403023058681398, 0.8414709848078965], atol=1e-15)


def test_frequency_exponent_and_pairing():
    # D = 4, base 10^4: theta = (1, 10^-2).  Position 100 turns pair (x0, x1) by 100 rad and
    # pair (x2, x3) by exactly 1 rad.  Adjacent elements pair up (not x_i with x_{i+D/2}).
    x = rope.rope(_rows_at([0.0, 0.0, 1.0, 0.0], 101, 4))[0, 100, 0]
    np.testing.assert_allclose(x, [0.0, 0.0, math.cos(1.0), math.sin(1.0)], atol=1e-14)
    x = rope.rope(_rows_at([1.0, 0.0, 0.0, 0.0], 101, 4))[0, 100, 0]
    np.testing.assert_allclose(x, [math.cos(100.0), math.sin(100.0), 0.0, 0.0], atol=1e-14)
    np.testing.assert_allclose(rope.theta(128)[[0, 32, 63]],
                               [1.0, 10000.0 ** -0.5, 10000.0 ** (-126 / 128)], rtol=1e-15)


def test_table_closed_form():
    t = rope.cos_sin_table(300, 64)
    p = np.arange(300)
    np.testing.assert_allclose(t[:, 0, 0], np.cos(p), atol=1e-15)
    np.testing.assert_allclose(t[:, 0, 1], np.sin(p), atol=1e-15)
    np.testing.assert_allclose(t[0], np.stack([np.ones(32), np.zeros(32)], -1), atol=0)
    np.testing.assert_allclose(t[..., 0] ** 2 + t[..., 1] ** 2, 1.0, atol=1e-15)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_identity_at_zero_and_norm_of_every_pair(D):
    x = RNG.standard_normal((2, 50, 3, D))
    y = rope.rope(x)
    np.testing.assert_array_equal(y[:, 0], x[:, 0])
    n_in = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    n_out = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-13)


@pytest.mark.parametrize("D", [64, 128])
def test_relative_position_property(D):
    # <rope(q) at m, rope(k) at n> depends on m - n only (RoFormer's defining property).
    q, k = RNG.standard_normal(D), RNG.standard_normal(D)
    S = 400
    rq, rk = rope.rope(_rows_at(q, S, D))[0, :, 0], rope.rope(_rows_at(k, S, D))[0, :, 0]
    for m, n in [(5, 3), (17, 90), (250, 250), (399, 0)]:
        for t in (1, -m if m < n else -n, 7):
            if 0 <= m + t < S and 0 <= n + t < S:
                np.testing.assert_allclose(rq[m] @ rk[n], rq[m + t] @ rk[n + t], atol=1e-10)
    # and it is not a function of m or n alone
    assert abs(rq[5] @ rk[3] - rq[6] @ rk[3]) > 1e-3


@pytest.mark.parametrize("D", [64, 128, 256])
def test_scores_unchanged_by_the_hadamard_rotation_after_rope(D):
    s = RNG.choice([-1.0, 1.0], size=D)
    q = rope.rope(RNG.standard_normal((1, 40, 2, D)))
    k = rope.rope(RNG.standard_normal((1, 40, 2, D)))
    R = hadamard.rotation_matrix(s)
    for h in range(2):
        np.testing.assert_allclose((q[0, :, h] @ R) @ (k[0, :, h] @ R).T, q[0, :, h] @ k[0, :, h].T, atol=1e-11)


def test_fused_quantiser_is_rope_then_quantiser():
    x = RNG.standard_normal((1, 200, 2, 64))
    s = RNG.choice([-1.0, 1.0], size=64)
    a = rope.rope_quantise_blocks(x, s)
    b = quantise.quantise_blocks(rope.rope(x), s)
    np.testing.assert_array_equal(a["codes"], b["codes"])
    np.testing.assert_array_equal(a["scale"], b["scale"])


def test_rejects_odd_head_dim():
    with pytest.raises(ValueError):
        rope.theta(63)
