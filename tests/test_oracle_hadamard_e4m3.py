"""Pins for the Hadamard rotation, the E4M3 format and the blockwise quantiser (CPU only).

Library routines used as independent references: scipy.linalg.hadamard
(Sylvester construction) and torch's float8_e4m3fn conversion.  The rest are
closed forms and invariants fixed by the pages: the rotation is orthogonal so
QK^T is unchanged ("FlashAttention-3 (NL)", "Technische innovaties", item 3,
step 4), and it spreads an outlier over all coordinates (step 2).
"""

import math
from fractions import Fraction

import numpy as np
import pytest
import scipy.linalg
import torch

from oracle import e4m3, hadamard, quantise

RNG = np.random.default_rng(99)


# ---------------------------------------------------------------- Hadamard --

@pytest.mark.parametrize("D", [1, 2, 4, 64, 128, 256])
def test_sylvester_matches_scipy_and_is_orthogonal(D):
    H = hadamard.sylvester(D)
    np.testing.assert_array_equal(H, scipy.linalg.hadamard(D))
    np.testing.assert_array_equal(H @ H.T, D * np.eye(D))


def test_sylvester_rejects_non_power_of_two():
    with pytest.raises(ValueError):
        hadamard.sylvester(96)


def _fwht_butterfly(x):
    """Independent fast Walsh-Hadamard transform (natural order) for the pin."""
    x = x.copy()
    D = x.shape[-1]
    h = 1
    while h < D:
        for i in range(0, D, 2 * h):
            a = x[..., i:i + h].copy()
            b = x[..., i + h:i + 2 * h].copy()
            x[..., i:i + h] = a + b
            x[..., i + h:i + 2 * h] = a - b
        h *= 2
    return x


@pytest.mark.parametrize("D", [64, 128, 256])
def test_rotation_equals_fast_transform_and_preserves_norm(D):
    s = RNG.choice([-1.0, 1.0], size=D)
    x = RNG.standard_normal((5, 3, D))
    xr = hadamard.rotate(x, s)
    np.testing.assert_allclose(xr, _fwht_butterfly(x * s) / math.sqrt(D), atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(xr, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    R = hadamard.rotation_matrix(s)
    np.testing.assert_allclose(R @ R.T, np.eye(D), atol=1e-14)


@pytest.mark.parametrize("D", [64, 128])
def test_rotation_leaves_qk_products_unchanged(D):
    s = RNG.choice([-1.0, 1.0], size=D)
    q, k = RNG.standard_normal((40, D)), RNG.standard_normal((50, D))
    np.testing.assert_allclose(hadamard.rotate(q, s) @ hadamard.rotate(k, s).T, q @ k.T, atol=1e-12)
    # different signs for Q and K would not preserve it
    s2 = -s
    s2[0] = s[0]
    assert np.abs(hadamard.rotate(q, s) @ hadamard.rotate(k, s2).T - q @ k.T).max() > 1e-3


def test_rotation_spreads_an_outlier_evenly():
    D = 128
    s = RNG.choice([-1.0, 1.0], size=D)
    x = np.zeros(D)
    x[17] = 40.0
    np.testing.assert_allclose(np.abs(hadamard.rotate(x, s)), 40.0 / math.sqrt(D), atol=1e-12)
    e0 = np.zeros(D)
    e0[0] = 1.0
    np.testing.assert_allclose(hadamard.rotate(e0, np.ones(D)), np.full(D, 1 / math.sqrt(D)), atol=1e-15)


# -------------------------------------------------------------------- E4M3 --

def test_all_256_codes_round_trip_and_match_torch_decoding():
    codes = np.arange(256, dtype=np.uint8)
    vals = e4m3.decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(vals), np.isnan(ref))
    fin = ~np.isnan(vals)
    np.testing.assert_array_equal(vals[fin], ref[fin])
    assert np.isnan(vals).sum() == 2                 # 0x7F and 0xFF
    np.testing.assert_array_equal(e4m3.encode(vals[fin]), codes[fin])
    assert e4m3.decode(np.array([0x7E]))[0] == 448.0


def test_known_codes_and_ties_to_even():
    assert e4m3.encode(np.array([1.0]))[0] == 0x38
    assert e4m3.encode(np.array([448.0]))[0] == 0x7E
    assert e4m3.encode(np.array([2.0 ** -9]))[0] == 0x01
    assert e4m3.encode(np.array([2.0 ** -6]))[0] == 0x08
    assert e4m3.encode(np.array([7 * 2.0 ** -9]))[0] == 0x07
    # 1.0625 lies half-way between 1.0 (mantissa 0) and 1.125 (mantissa 1): even wins
    assert e4m3.round_e4m3(np.array([1.0625]))[0] == 1.0
    # 1.1875 lies half-way between 1.125 (mantissa 1) and 1.25 (mantissa 2): even wins
    assert e4m3.round_e4m3(np.array([1.1875]))[0] == 1.25
    assert e4m3.round_e4m3(np.array([-1.1875]))[0] == -1.25
    # half of the smallest subnormal rounds to zero (even), slightly more rounds up
    assert e4m3.round_e4m3(np.array([2.0 ** -10]))[0] == 0.0
    assert e4m3.round_e4m3(np.array([2.0 ** -10 * 1.01]))[0] == 2.0 ** -9


def test_saturation():
    np.testing.assert_array_equal(e4m3.round_e4m3(np.array([449.0, 464.0, 500.0, 1e9, -1e9])),
                                  [448.0, 448.0, 448.0, 448.0, -448.0])


def test_rounding_matches_torch_cast_in_range():
    fin = e4m3.decode(np.arange(0, 0x7F, dtype=np.uint8))          # non-negative finite grid
    mids = (fin[1:] + fin[:-1]) / 2                                  # exact ties
    rnd = RNG.uniform(0, 448, 20000) * np.exp2(-RNG.integers(0, 14, 20000))
    # perturbations are representable in fp32, the type torch converts through
    x = np.concatenate([fin, mids, rnd, mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20)])
    x = np.concatenate([x, -x]).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(e4m3.round_e4m3(x), ref)


# --------------------------------------------------------------- quantiser --

def test_block_scale_maps_block_max_to_448_and_error_bound():
    B, S, H, D = 2, 300, 3, 64                   # blocks of 128, 128, 44 tokens
    x = RNG.standard_normal((B, S, H, D))
    out = quantise.quantise_blocks(x)
    assert out["scale"].shape == (B, H, 3)
    for i, (t0, t1) in enumerate([(0, 128), (128, 256), (256, 300)]):
        amax = np.abs(x[:, t0:t1]).max(axis=(1, 3))
        np.testing.assert_allclose(out["scale"][:, :, i], amax / 448.0, rtol=1e-15)
        np.testing.assert_allclose(np.abs(out["q"][:, t0:t1]).max(axis=(1, 3)), 448.0)
    # relative error <= 2^-4 in the normal range, absolute <= 2^-10 below it (scaled units)
    pre, q = out["pre"], out["q"]
    err = np.abs(q - pre)
    bound = np.maximum(np.abs(pre) * 2.0 ** -4, 2.0 ** -10)
    assert (err <= bound * (1 + 1e-12)).all()
    np.testing.assert_array_equal(e4m3.decode(out["codes"]), q)


def test_zero_block_gets_unit_scale_and_planted_outlier_moves_one_scale():
    B, S, H, D = 1, 384, 2, 64
    x = RNG.standard_normal((B, S, H, D))
    x[:, 0:128, 1] = 0.0
    base = quantise.quantise_blocks(x)
    assert (base["scale"][0, 1, 0] == 1.0) and (base["codes"][:, 0:128, 1] == 0).all()
    y = x.copy()
    y[0, 200, 0, 5] = 1000.0
    moved = quantise.quantise_blocks(y)
    changed = moved["scale"] != base["scale"]
    assert changed.sum() == 1 and changed[0, 0, 1]
    assert moved["scale"][0, 0, 1] == 1000.0 / 448.0


def test_dequantise_of_grid_values_is_exact():
    # values already on the E4M3 grid times a power-of-two scale survive unchanged
    B, S, H, D = 1, 256, 2, 32
    codes = RNG.integers(0, 0x7E, size=(B, S, H, D)).astype(np.uint8)
    vals = e4m3.decode(codes) * np.where(RNG.random((B, S, H, D)) < 0.5, -1, 1)
    vals[:, 0, :, 0] = 448.0
    vals[:, 128, :, 0] = 448.0
    x = vals * 2.0 ** -5
    out = quantise.quantise_blocks(x)
    np.testing.assert_array_equal(out["scale"], 2.0 ** -5)
    np.testing.assert_array_equal(quantise.dequantise(out["q"], out["scale"]), x)


def test_rotated_quantiser_rotates_before_scaling():
    B, S, H, D = 1, 128, 1, 128
    s = RNG.choice([-1.0, 1.0], size=D)
    x = RNG.standard_normal((B, S, H, D))
    out = quantise.quantise_blocks(x, s)
    np.testing.assert_allclose(out["rotated"], hadamard.rotate(x, s), atol=1e-13)
    np.testing.assert_allclose(out["scale"][0, 0, 0], np.abs(hadamard.rotate(x, s)).max() / 448.0, rtol=1e-14)


def _brute_force(x, signs, granularity="block"):
    """Every element decided in exact rational arithmetic from x: exact transform, exact
    block (or tensor) maximum, exact quotient 448 y / amax, nearest E4M3 with ties to even."""
    B, S, H, D = x.shape
    Hm = hadamard.sylvester(D)
    y = np.empty(x.shape, dtype=object)
    for idx in np.ndindex(B, S, H):
        row = [Fraction(float(a)) for a in x[idx]]
        if signs is None:
            y[idx] = row
        else:
            xs = [row[d] * int(signs[d]) for d in range(D)]
            y[idx] = [sum(xs[d] * int(Hm[d, c]) for d in range(D)) for c in range(D)]
    q = np.empty(x.shape)
    A_all = max(abs(v) for v in y.reshape(-1)) if granularity == "tensor" else None
    for b, s, h in np.ndindex(B, S, H):
        if granularity == "tensor":
            A = A_all
        else:
            t0 = s // 128 * 128
            A = max(abs(v) for v in y[b, t0:min(S, t0 + 128), h].reshape(-1))
        for c in range(D):
            q[b, s, h, c] = quantise.rne_e4m3_fraction(448 * y[b, s, h, c] / A) if A > 0 else 0.0
    return q


def test_exact_rne_of_fractions_matches_torch_cast():
    fin = e4m3.decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = (fin[1:] + fin[:-1]) / 2
    rnd = RNG.uniform(0, 448, 3000) * np.exp2(-RNG.integers(0, 14, 3000))
    x = np.concatenate([fin, mids, rnd, mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20)])
    x = np.concatenate([x, -x]).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([quantise.rne_e4m3_fraction(Fraction(float(v))) for v in x])
    np.testing.assert_array_equal(got, ref)
    # beyond the range torch's cast gives NaN; the quantiser saturates ("satfinite")
    assert quantise.rne_e4m3_fraction(Fraction(500)) == 448.0
    assert quantise.rne_e4m3_fraction(Fraction(-10 ** 6)) == -448.0


def test_exact_midpoints_go_to_the_even_neighbour():
    # amax = 26 and x = 39 * 2^-5: the quotient 448 * 1.21875 / 26 = 21 lies exactly half-way
    # between the E4M3 values 20 (mantissa 2, even) and 22 (mantissa 3): even wins.  A rounding
    # decision taken in fp32 (x * fl32(448 / 26)) lands slightly above 21 and would pick 22.
    B, S, H, D = 1, 128, 1, 128
    x = torch.from_numpy(RNG.standard_normal((B, S, H, D))).to(torch.bfloat16).double().numpy()
    x[0, 0, 0, 0] = 26.0
    x[0, 1:40, 0, 1] = 39 * 2.0 ** -5
    out = quantise.quantise_blocks(x)
    assert (out["q"][0, 1:40, 0, 1] == 20.0).all()
    assert (out["pre"][0, 1:40, 0, 1] == 21.0).all()
    f32 = np.float32(39 * 2.0 ** -5) * (np.float32(448.0) / np.float32(26.0))
    assert e4m3.round_e4m3(np.array([float(f32)]))[0] == 22.0
    # and every element equals the decision taken in exact arithmetic
    np.testing.assert_array_equal(out["q"], _brute_force(x, None))


@pytest.mark.parametrize("rotate", [False, True])
def test_quantiser_equals_exact_arithmetic_brute_force(rotate):
    # bf16 inputs with outliers and planted ties, blocks of 128 and a ragged 44-token block
    B, S, H, D = 1, 172, 2, 16
    x = RNG.standard_normal((B, S, H, D))
    x[RNG.random(x.shape) < 0.01] *= 10
    x = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    x[0, 3, 1, :] = 0.0
    x[0, 5, 0, 0] = 26.0
    x[0, 6:20, 0, 2] = 39 * 2.0 ** -5
    s = RNG.choice([-1.0, 1.0], size=D) if rotate else None
    out = quantise.quantise_blocks(x, s)
    np.testing.assert_array_equal(out["q"], _brute_force(x, s))
    np.testing.assert_array_equal(e4m3.decode(out["codes"]), out["q"])


def test_rows_fp64_cannot_hold_are_transformed_exactly():
    # 100 and 2^-60 in one row: the +-sums need about 67 significant bits, beyond fp64
    B, S, H, D = 1, 130, 1, 16
    x = RNG.standard_normal((B, S, H, D))
    x[0, 7, 0, 0] = 100.0
    x[0, 7, 0, 1:] = 2.0 ** -60
    x[0, 129, 0, 3] = 2.0 ** -70
    s = RNG.choice([-1.0, 1.0], size=D)
    out = quantise.quantise_blocks(x, s)
    np.testing.assert_array_equal(out["q"], _brute_force(x, s))


def test_tensor_granularity_uses_one_scale():
    B, S, H, D = 2, 300, 2, 16
    x = RNG.standard_normal((B, S, H, D))
    x[1, 250, 1, 3] = 37.0
    out = quantise.quantise_blocks(x, granularity="tensor")
    np.testing.assert_array_equal(out["scale"], np.full((B, H, 3), 37.0 / 448.0))
    np.testing.assert_array_equal(out["q"], _brute_force(x, None, "tensor"))
    s = RNG.choice([-1.0, 1.0], size=D)
    rot = quantise.quantise_blocks(x, s, granularity="tensor")
    np.testing.assert_allclose(rot["scale"], np.abs(hadamard.rotate(x, s)).max() / 448.0, rtol=1e-14)
    np.testing.assert_array_equal(rot["q"], _brute_force(x, s, "tensor"))
    with pytest.raises(ValueError):
        quantise.quantise_blocks(x, granularity="row")
