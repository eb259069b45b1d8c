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
    q, k, v = (t.to(torch.float64).numpy() for t in synth.make_qkv(1, S, H, D, case, dist))
    s = synth.signs(D, synth.seed_for(case, synth.STREAM_SIGNS)).astype(np.float64)
    O_ref, _ = A.attention(q, k, v)
    O_none, _, _ = fp8_path.fp8_attention(q, k, v, signs=None)
    O_had, _, _ = fp8_path.fp8_attention(q, k, v, signs=s)
    rms = lambda x: float(np.sqrt(np.mean(x ** 2)))
    return rms(O_none - O_ref), rms(O_had - O_ref)


@pytest.mark.parametrize("case", [40, 41])
def test_incoherent_processing_lowers_fp8_error_on_outlier_inputs(case):
    e_none, e_had = _experiment(case)
    ratio = e_had / e_none
    print(f"case {case}: RMS no-rotation {e_none:.3e}  rotation {e_had:.3e}  ratio {ratio:.3f}")
    assert 0.4 < ratio < 0.85
    assert e_had < 2e-2


def test_rotation_changes_little_without_outliers():
    e_none, e_had = _experiment(42, dist="normal")
    assert 0.8 < e_had / e_none < 1.25


def test_v_ratio_of_one_is_plain_numerator_rounding():
    B, S, H, D = 1, 300, 2, 32
    q, k, v = (RNG.standard_normal((B, S, H, D)) for _ in range(3))
    a, la = fp8_path.attention_rounded_p(q, k, v, 0.2, causal=True, round_p=True)
    b, lb = fp8_path.attention_rounded_p(q, k, v, 0.2, causal=True, round_p=True, v_ratio=np.ones((B, H, S)))
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


def test_power_of_two_ratios_commute_with_rounding():
    # Scaling by 2^-k moves only the exponent, so E4M3(e * 2^-k) / 2^-k = E4M3(e) while e * 2^-k
    # stays in the normal range (>= 2^-6): a small key count keeps every numerator >= 2^-6 * 2^3.
    B, S, H, D = 1, 8, 1, 16
    q = np.zeros((B, S, H, D))
    k, v = RNG.standard_normal((B, S, H, D)), RNG.standard_normal((B, S, H, D))
    q[..., 0] = 0.3
    k[..., 0] = np.linspace(-1.0, 1.0, S)[None, :, None]     # logits in [-0.3, 0.3]: e in [0.5, 1]
    r = 2.0 ** -RNG.integers(0, 3, size=(B, H, S))
    a, _ = fp8_path.attention_rounded_p(q, k, v, 1.0, round_p=True)
    b, _ = fp8_path.attention_rounded_p(q, k, v, 1.0, round_p=True, v_ratio=r)
    np.testing.assert_array_equal(a, b)
    c, _ = fp8_path.attention_rounded_p(q, k, v, 1.0, round_p=True, v_ratio=np.full((B, H, S), 0.3))
    assert not np.array_equal(a, c)


def test_one_key_with_a_ratio_by_hand():
    # One key: e = 1, l = 1.  With r = 0.3 the operand is E4M3(0.3) = 0.3125 (0.3 = 1.2 * 2^-2 lies
    # between 1.125 * 2^-2 and 1.25 * 2^-2, nearer the latter), so O = (0.3125 / 0.3) * v.
    q = np.ones((1, 1, 1, 4))
    k = np.full((1, 1, 1, 4), 0.5)
    v = np.array([1.0, -2.0, 0.5, 4.0]).reshape(1, 1, 1, 4)
    O, lse = fp8_path.attention_rounded_p(q, k, v, 1.0, round_p=True, v_ratio=np.full((1, 1, 1), 0.3))
    np.testing.assert_allclose(O[0, 0, 0], (0.3125 / 0.3) * v[0, 0, 0], rtol=1e-15)
    np.testing.assert_allclose(lse[0, 0, 0], 2.0, rtol=1e-15)


def test_v_block_ratio_layout():
    sc = np.array([[[2.0, 4.0, 1.0]]])                        # [B=1, H=1, 3 blocks]
    r = fp8_path.v_block_ratio(sc, 300)
    assert r.shape == (1, 1, 300)
    assert r[0, 0, 0] == 0.5 and r[0, 0, 127] == 0.5 and r[0, 0, 128] == 1.0 and r[0, 0, 256] == 0.25


def test_ratios_belong_to_keys_by_hand():
    # Two queries, two keys with equal logits (e = 1 each, l = 2) and ratios 0.3 and 1:
    # O = (E4M3(0.3) / 0.3 * v_0 + v_1) / 2 for both queries.
    q = np.zeros((1, 2, 1, 4))
    k = np.zeros((1, 2, 1, 4))
    v = np.array([[1.0, 2.0, -1.0, 0.5], [3.0, -1.0, 2.0, 1.0]]).reshape(1, 2, 1, 4)
    O, _ = fp8_path.attention_rounded_p(q, k, v, 1.0, round_p=True, v_ratio=np.array([[[0.3, 1.0]]]))
    want = ((0.3125 / 0.3) * v[0, 0, 0] + v[0, 1, 0]) / 2
    np.testing.assert_allclose(O[0, 0, 0], want, rtol=1e-15)
    np.testing.assert_allclose(O[0, 1, 0], want, rtol=1e-15)


def test_zero_block_scale_terms_vanish():
    # a key of a zero-scale block has V = 0; its folded term is 0 (not 0/0) and l still counts it
    q = np.zeros((1, 2, 1, 4))
    k = np.zeros((1, 2, 1, 4))
    v = np.array([[0.0, 0.0, 0.0, 0.0], [3.0, -1.0, 2.0, 1.0]]).reshape(1, 2, 1, 4)
    O, lse = fp8_path.attention_rounded_p(q, k, v, 1.0, round_p=True, v_ratio=np.array([[[0.0, 1.0]]]))
    np.testing.assert_allclose(O[0, 0, 0], v[0, 1, 0] / 2, rtol=1e-15)
    np.testing.assert_allclose(lse[0, 0], np.log(2.0), rtol=1e-15)
    r = fp8_path.v_block_ratio(np.zeros((1, 1, 2)), 200)
    assert np.array_equal(r, np.zeros((1, 1, 200)))
