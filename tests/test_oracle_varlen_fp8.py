"""Pins for the packed-batch FP8 path of the oracle (CPU only)."""

import numpy as np
import pytest

from oracle import fp8_path, quantise
from oracle import varlen_fp8 as VF
from oracle.varlen import attention_varlen

RNG = np.random.default_rng(11)


def test_block_indices_by_hand():
    # lengths 1, 129, 0, 128 (cu = 0, 1, 130, 130, 258): bases 0, 1, 3, 4; NB = 2 + 4 + 1 = 7; sequence 1
    # takes indices 1 and 2, index 3 (the empty sequence) and 5, 6 carry nothing
    cu = np.array([0, 1, 130, 130, 258])
    assert list(VF.block_base(cu)) == [0, 0 + 1, 1 + 2, 1 + 3]
    assert VF.scale_blocks(258, 4) == 7
    x = RNG.standard_normal((258, 2, 16))
    r = VF.quantise_varlen(x, cu)
    sc = r["scale"]
    np.testing.assert_allclose(sc[:, 0], np.abs(x[0:1]).max(axis=(0, 2)) / 448, rtol=1e-15)
    np.testing.assert_allclose(sc[:, 1], np.abs(x[1:129]).max(axis=(0, 2)) / 448, rtol=1e-15)
    np.testing.assert_allclose(sc[:, 2], np.abs(x[129:130]).max(axis=(0, 2)) / 448, rtol=1e-15)
    np.testing.assert_allclose(sc[:, 4], np.abs(x[130:258]).max(axis=(0, 2)) / 448, rtol=1e-15)
    assert np.isnan(sc[:, 3]).all() and np.isnan(sc[:, 5:]).all()


@pytest.mark.parametrize("rotate", [False, True])
def test_whole_blocks_match_the_fixed_length_quantiser(rotate):
    # sequences whose lengths are multiples of 128: the blocks are those of the packed tensor
    cu = np.array([0, 128, 384, 512])
    x = RNG.standard_normal((512, 3, 32))
    s = np.where(RNG.random(32) < 0.5, -1.0, 1.0) if rotate else None
    r = VF.quantise_varlen(x, cu, s)
    ref = quantise.quantise_blocks(x[None], s)
    np.testing.assert_array_equal(r["codes"], ref["codes"][0])
    base = VF.block_base(cu)
    # packed block b of sequence s sits at index b + s
    for si, (b0, b1) in enumerate([(0, 1), (1, 3), (3, 4)]):
        np.testing.assert_array_equal(r["scale"][:, base[si]:base[si] + (b1 - b0)], ref["scale"][0][:, b0:b1])


def test_exact_values_reduce_to_the_varlen_definition():
    # without rounding of the numerators, the path on de-quantised inputs is exact attention
    cu = np.array([0, 5, 5, 200, 331])
    q, k, v = (RNG.standard_normal((331, 2, 16)) for _ in range(3))
    deq = [VF.quantise_varlen(t, cu)["deq"] for t in (q, k, v)]
    for causal in (False, True):
        O, lse = VF.fp8_attention_varlen(*deq, cu, 0.25, causal, round_p=False)
        O0, lse0 = attention_varlen(*deq, cu, 0.25, causal)
        np.testing.assert_allclose(O, O0, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, lse0, rtol=1e-12, atol=1e-13)


def test_one_sequence_is_the_fixed_length_fp8_path():
    S, H, D = 300, 2, 32
    cu = np.array([0, S])
    q, k, v = (RNG.standard_normal((S, H, D)) for _ in range(3))
    rv = VF.quantise_varlen(v, cu)
    deq = [VF.quantise_varlen(t, cu)["deq"] for t in (q, k)] + [rv["deq"]]
    O, lse = VF.fp8_attention_varlen(*deq, cu, 0.2, True)
    O1, lse1, _ = fp8_path.fp8_attention(q[None], k[None], v[None], None, 0.2, True)
    np.testing.assert_allclose(O, O1[0], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, lse1[0], rtol=1e-13)


def test_rotary_positions_restart_at_every_sequence():
    from oracle import rope as R
    cu = np.array([0, 200, 200, 330])
    x = RNG.standard_normal((330, 2, 16))
    s = np.where(RNG.random(16) < 0.5, -1.0, 1.0)
    r = VF.quantise_varlen(x, cu, s, rope_base=10000.0)
    a = R.rope_quantise_blocks(x[None, :200], s)                 # sequence 0 alone
    b = R.rope_quantise_blocks(x[None, 200:], s)                 # sequence 2 alone, positions from 0
    np.testing.assert_array_equal(r["codes"][:200], a["codes"][0])
    np.testing.assert_array_equal(r["codes"][200:], b["codes"][0])
    base = VF.block_base(cu)
    np.testing.assert_array_equal(r["scale"][:, base[2]:base[2] + 2], b["scale"][0])
    # not the embedding of the packed axis: positions 200 .. 329 would give other codes
    c = R.rope_quantise_blocks(x[None], s)
    assert not np.array_equal(r["codes"][200:], c["codes"][0, 200:])
