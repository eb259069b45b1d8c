"""Pins for the fp64 emulation of the FP8 path, and the incoherent-processing experiment (CPU only).

The experiment follows the hada.io FA3 summary, "Niedrige FP8-Präzision und
incoherent processing": Q, K, V standard normal with 0.1 % of the entries
given a large magnitude; incoherent processing is reported there to cut the
FP8 quantisation error 2.6-fold.  Under the readings taken here (per
128-token-block scales, E4M3 with round-to-nearest-even, outliers N(0, 10),
error = RMS of O against exact fp64 attention on the unquantised inputs) the
reduction measured by this emulation is smaller (ratio about 0.6-0.75, not
1/2.6); the test records the ratio and checks its direction and range, it
does not tune the recipe to reach 2.6.
"""

import numpy as np
import pytest
import torch

from exact_attention_46_gb300 import synth
from oracle import attention as A
from oracle import e4m3, fp8_path, quantise

RNG = np.random.default_rng(7)


def _grid_inputs(B, S, H, D):
    """Inputs whose blockwise E4M3 quantisation is exact (scale 2^-5 per block)."""
    # codes 0x38..0x6F are the normal values 1 .. 120; divided by 64 they stay on the grid
    codes = RNG.integers(0x38, 0x70, size=(B, S, H, D)).astype(np.uint8)
    vals = e4m3.decode(codes) * np.where(RNG.random((B, S, H, D)) < 0.5, -1, 1) / 64.0
    for t0 in range(0, S, 128):
        vals[:, t0, :, 0] = 448.0
    return vals * 2.0 ** -5


@pytest.mark.parametrize("causal", [False, True])
def test_exactly_representable_inputs_reduce_to_plain_attention(causal):
    B, S, H, D = 1, 256, 2, 64
    q, k, v = _grid_inputs(B, S, H, D), _grid_inputs(B, S, H, D), _grid_inputs(B, S, H, D)
    O, lse, _ = fp8_path.fp8_attention(q, k, v, signs=None, causal=causal, round_p=False)
    O0, lse0 = A.attention(q, k, v, causal=causal)
    np.testing.assert_allclose(O, O0, atol=1e-13)
    np.testing.assert_allclose(lse, lse0, atol=1e-12)


def test_rotation_without_quantisation_error_is_invisible():
    # Rotated inputs, no rounding anywhere: the result equals plain attention,
    # because the rotation is orthogonal ("FlashAttention-3 (NL)", item 3, step 4).
    B, S, H, D = 1, 200, 2, 64
    s = np.where(RNG.random(D) < 0.5, -1.0, 1.0)
    q, k, v = RNG.standard_normal((3, B, S, H, D))
    Qq, Kq, Vq = fp8_path.quantise_qkv(q, k, v, s)
    qd = Qq["rotated"]
    kd = Kq["rotated"]
    O, lse = fp8_path.attention_rounded_p(qd, kd, v, 1 / np.sqrt(D), round_p=False)
    O0, lse0 = A.attention(q, k, v)
    np.testing.assert_allclose(O, O0, atol=1e-12)
    np.testing.assert_allclose(lse, lse0, atol=1e-12)


def test_rounding_p_error_bound():
    B, S, H, D = 1, 256, 2, 64
    q, k, v = RNG.standard_normal((3, B, S, H, D))
    Or, lr = fp8_path.attention_rounded_p(q, k, v, 0.125, round_p=True)
    Oe, le = fp8_path.attention_rounded_p(q, k, v, 0.125, round_p=False)
    np.testing.assert_array_equal(lr, le)
    # |dp| <= max(p 2^-4, 2^-10) for p in (0, 1]  =>  |dO| <= 2^-4 max|v| + 2^-10 S max|v| / l, l >= 1
    bound = (2.0 ** -4 + 2.0 ** -10 * S) * np.abs(v).max()
    assert np.abs(Or - Oe).max() <= bound
    assert np.abs(Or - Oe).max() > 0


def _experiment(case, S=512, H=4, D=128, dist="outliers"):
    """RMS of O against exact attention: (per-block FP8, per-block FP8 with the rotation,
    per-tensor FP8 without the rotation)."""
    q, k, v = (t.to(torch.float64).numpy() for t in synth.make_qkv(1, S, H, D, case, dist))
    s = synth.signs(D, synth.seed_for(case, synth.STREAM_SIGNS)).astype(np.float64)
    O_ref, _ = A.attention(q, k, v)
    O_none, _, _ = fp8_path.fp8_attention(q, k, v, signs=None)
    O_had, _, _ = fp8_path.fp8_attention(q, k, v, signs=s)
    O_tensor, _, _ = fp8_path.fp8_attention(q, k, v, signs=None, granularity="tensor")
    rms = lambda x: float(np.sqrt(np.mean(x ** 2)))
    return rms(O_none - O_ref), rms(O_had - O_ref), rms(O_tensor - O_ref)


@pytest.mark.parametrize("case", [40, 41])
def test_incoherent_processing_lowers_fp8_error_on_outlier_inputs(case):
    # reading 1: the baseline is the same per-block FP8 path without the rotation
    e_none, e_had, _ = _experiment(case)
    ratio = e_had / e_none
    print(f"case {case}: RMS no-rotation {e_none:.3e}  rotation {e_had:.3e}  ratio {ratio:.3f}")
    assert 0.4 < ratio < 0.85
    assert e_had < 2e-2


@pytest.mark.parametrize("case", [40, 41])
def test_incoherent_processing_against_standard_fp8(case):
    # reading 2: the baseline is standard FP8 -- one scale per tensor, no rotation.  A single
    # scale set by the largest outlier leaves the rest of the tensor with fewer significant
    # bits (more values in the subnormal range), so the baseline's error is larger than the
    # per-block one and the product's reduction against it larger too
    e_none, e_had, e_tensor = _experiment(case)
    print(f"case {case}: RMS per-tensor {e_tensor:.3e}  per-block + rotation {e_had:.3e}  "
          f"ratio {e_had / e_tensor:.3f}")
    assert e_tensor > e_none
    assert e_had / e_tensor < e_had / e_none


def test_per_tensor_scale_equals_per_block_when_every_block_shares_the_max():
    # with the same largest magnitude in every (b, h, block), the two granularities coincide
    B, S, H, D = 1, 256, 2, 32
    x = RNG.standard_normal((B, S, H, D))
    x[:, ::128, :, 0] = 9.0
    a = quantise.quantise_blocks(x)
    b = quantise.quantise_blocks(x, granularity="tensor")
    np.testing.assert_array_equal(a["codes"], b["codes"])
    np.testing.assert_array_equal(a["scale"], b["scale"])


def test_rotation_changes_little_without_outliers():
    e_none, e_had, _ = _experiment(42, dist="normal")
    assert 0.8 < e_had / e_none < 1.25
