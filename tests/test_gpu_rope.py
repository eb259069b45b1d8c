"""Rotary embedding fused into the rotation + quantiser, vs the fp64 oracle, through the C ABI (GPU).

Table: every entry is the fp64 (cos, sin) rounded to fp32; the kernel evaluates in fp64 too,
so the two agree to one fp32 unit in the last place (1e-10 absolute near zero, where the
fp64 angles' last-bit differences show).

Fused quantiser: the kernel turns each pair in fp32 with (cos, sin) rebuilt by the
angle-addition identity from two table rows (about 3 fp32 ulps), so its pre-rounding values
differ from the oracle's fp64 ones by a few ulps of the row's largest values.  Block scales
agree to 1e-5 relative; codes agree except where the oracle's pre-rounding value lies within
TIE_ATOL (in code units; the grid spacing there is >= 2^-9) of a rounding midpoint, where the
two codes must be grid neighbours, at most 1e-4 of all codes.
"""

import numpy as np
import pytest
import torch

from exact_attention_46_gb300 import ops, synth
from oracle import rope
from tests.helpers import check_codes, inputs, to64

pytestmark = pytest.mark.gpu

TIE_RTOL = 1e-5
TIE_ATOL = 5e-4
SCALE_RTOL = 1e-5


def table_rows(S):
    return 128 * ((S + 127) // 128)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("n_pos,base", [(1, 10000.0), (300, 10000.0), (65536, 10000.0), (4096, 500000.0)])
def test_table_matches_oracle(n_pos, D, base):
    cs = ops.rope_cos_sin_table(n_pos, D, base)
    ops.check()
    g = cs.cpu().numpy()
    r = rope.cos_sin_table(n_pos, D, base).astype(np.float32)
    tol = np.maximum(np.spacing(np.abs(r)), 1e-10)
    assert np.all(np.abs(g.astype(np.float64) - r) <= tol), np.abs(g.astype(np.float64) - r).max()


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("rotate", [False, True])
@pytest.mark.parametrize("S", [1, 128, 300, 1024])
def test_fused_quantiser_matches_oracle(S, D, rotate):
    B, H = 2, 3
    x = inputs(B, S, H, D, case=30, dist="outliers")[0]
    s = synth.signs(D, synth.seed_for(30, synth.STREAM_SIGNS)) if rotate else None
    cs = ops.rope_cos_sin_table(table_rows(S), D)
    codes, scale = ops.rope_hadamard_rotate_quant_fp8(x.cuda(), cs, torch.from_numpy(s).cuda() if rotate else None)
    ops.check()
    ref = rope.rope_quantise_blocks(to64(x), None if s is None else s.astype(np.float64))
    np.testing.assert_allclose(scale.cpu().double().numpy(), ref["scale"], rtol=SCALE_RTOL, atol=0)
    check_codes(codes.cpu().numpy(), ref, TIE_RTOL, TIE_ATOL)


@pytest.mark.parametrize("B,S,H,D", [(1, 8192, 8, 128), (1, 65536, 1, 128), (1, 4096, 2, 256), (2, 2000, 4, 64)])
def test_fused_quantiser_long_positions(B, S, H, D):
    # positions up to 65535: the coarse table rows at large multiples of 16 and angles of
    # tens of thousands of radians
    x = inputs(B, S, H, D, case=31, dist="outliers")[0]
    s = synth.signs(D, synth.seed_for(31, synth.STREAM_SIGNS))
    cs = ops.rope_cos_sin_table(table_rows(S) + 64, D)       # a longer table is fine
    codes, scale = ops.rope_hadamard_rotate_quant_fp8(x.cuda(), cs, torch.from_numpy(s).cuda())
    ops.check()
    ref = rope.rope_quantise_blocks(to64(x), s.astype(np.float64))
    np.testing.assert_allclose(scale.cpu().double().numpy(), ref["scale"], rtol=SCALE_RTOL, atol=0)
    check_codes(codes.cpu().numpy(), ref, TIE_RTOL, TIE_ATOL)


@pytest.mark.parametrize("causal", [False, True])
def test_rope_then_fp8_attention_matches_oracle(causal):
    # End to end: rotary Q and K through the fused quantiser, V through the plain one, then FP8
    # attention; element by element against exact attention on the oracle's quantisation of the
    # oracle's rotary Q and K (tests/fp8_bound.py), widened by the codes the fused quantiser's
    # fp32 rotary arithmetic may put on the other side of a rounding midpoint (TIE_ATOL) and by
    # its scales (SCALE_RTOL)
    from oracle import quantise
    from tests import fp8_bound
    B, S, H, D = 1, 640, 2, 128
    q, k, v = inputs(B, S, H, D, case=32, dist="outliers")
    s = synth.signs(D, synth.seed_for(32, synth.STREAM_SIGNS))
    sd = torch.from_numpy(s).cuda()
    cs = ops.rope_cos_sin_table(table_rows(S), D)
    q8, sq = ops.rope_hadamard_rotate_quant_fp8(q.cuda(), cs, sd)
    k8, sk = ops.rope_hadamard_rotate_quant_fp8(k.cuda(), cs, sd)
    v8, sv = ops.hadamard_rotate_quant_fp8(v.cuda(), None)
    o, lse = ops.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, causal=causal)
    ops.check()
    s64 = s.astype(np.float64)
    res = [rope.rope_quantise_blocks(to64(q), s64), rope.rope_quantise_blocks(to64(k), s64),
           quantise.quantise_blocks(to64(v), None)]
    for r, g in zip(res, (q8, k8, v8)):
        check_codes(g.cpu().numpy(), r, TIE_RTOL, TIE_ATOL)
    deq = [quantise.dequantise(r["q"], r["scale"]) for r in res]
    widths = [fp8_bound.tie_widths_blocks(r, TIE_RTOL, TIE_ATOL, SCALE_RTOL) for r in res]
    ref = fp8_bound.reference(*deq, res[2]["scale"], 1 / np.sqrt(D), causal, dq=widths[0], dk=widths[1], dv=widths[2])
    fp8_bound.check(to64(o), to64(lse), ref)
