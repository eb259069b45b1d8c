"""The FP8 path on packed variable-length batches vs the fp64 oracle, through the C ABI (GPU).

Quantiser: codes and scales as in the fixed-length quantiser tests (ties aside, bit-identical
codes; scales to 2e-6), over length mixes with empty sequences, single tokens and every
remainder mod 128; one sequence is the fixed-length quantiser bit for bit; bad offsets write
nothing.  Attention: the kernel gets the oracle's own codes and scales, and every output
element lies within the FP8 bounds of tests/fp8_bound.py against exact attention on the
de-quantised values (V's block ratios taken over the sequence's own blocks); lse within 1e-3.
End to end from the GPU's packed quantiser, the bounds widen by the codes that may sit on the
other side of a rounding midpoint.  Equal lengths are attn_fwd_fp8 bit for bit.
"""

import numpy as np
import pytest
import torch

from exact_attention_46_gb300 import _lib, ops, synth
from oracle import varlen as oracle_varlen
from oracle import varlen_fp8 as VF
from tests import fp8_bound, helpers
from tests.helpers import to64

pytestmark = pytest.mark.gpu

MIXES = {
    "edges": [0, 5, 5, 133, 134, 390, 391, 600],
    "tiles": np.concatenate([[0], np.cumsum([127, 128, 129, 255, 256, 257, 511, 512, 513, 1])]),
    "empty_ends": [0, 0, 0, 300, 300, 300],
}


def packed(total, H, D, case):
    q, k, v = synth.make_qkv(1, total, H, D, case)
    return q[0], k[0], v[0]


def signs(case, D):
    return synth.signs(D, synth.seed_for(case, synth.STREAM_SIGNS))



@pytest.mark.parametrize("rotate", [False, True])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("mix", sorted(MIXES))
def test_quantiser_matches_oracle(mix, D, rotate):
    cu = np.asarray(MIXES[mix], dtype=np.int32)
    x = packed(int(cu[-1]), 3, D, case=90)[0]
    s = signs(90, D) if rotate else None
    dev = torch.device("cuda")
    codes, scale = ops.hadamard_rotate_quant_fp8_varlen(x.to(dev), torch.from_numpy(cu).to(dev),
                                                        torch.from_numpy(s).to(dev) if rotate else None)
    ops.check()
    ref = VF.quantise_varlen(to64(x), cu, None if s is None else s.astype(np.float64))
    live = ~np.isnan(ref["scale"])
    np.testing.assert_allclose(scale.cpu().double().numpy()[live], ref["scale"][live], rtol=2e-6, atol=0)
    helpers.check_codes(codes.cpu().numpy(), ref, 1e-5, 1e-12)


def test_one_sequence_is_the_fixed_length_quantiser():
    S, H, D = 700, 2, 128
    x = packed(S, H, D, case=91)[0].cuda()
    sg = torch.from_numpy(signs(91, D)).cuda()
    c1, s1 = ops.hadamard_rotate_quant_fp8_varlen(x, torch.tensor([0, S], dtype=torch.int32).cuda(), sg)
    c2, s2 = ops.hadamard_rotate_quant_fp8(x[None].contiguous(), sg)
    ops.check()
    assert torch.equal(c1, c2[0])
    assert torch.equal(s1[:, :s2.shape[2]], s2[0])


def test_bad_offsets_write_nothing():
    dev = torch.device("cuda")
    x = packed(300, 2, 128, case=92)[0].to(dev)
    for cu in ([0, 200, 100, 300], [1, 150, 300], [0, 150, 299], [0, 150, 301]):
        out = torch.full((300, 2, 128), 7, dtype=torch.uint8, device=dev)
        sc = torch.full((2, ops.varlen_scale_blocks(300, len(cu) - 1)), 7.0, device=dev)
        ops.hadamard_rotate_quant_fp8_varlen(x, torch.tensor(cu, dtype=torch.int32, device=dev), None, out=out,
                                             scale=sc)
        with pytest.raises(_lib.AttnError) as e:
            ops.check()
        assert e.value.status == 1
        assert bool((out == 7).all()) and bool((sc == 7.0).all())
    ops.hadamard_rotate_quant_fp8_varlen(x, torch.tensor([0, 150, 300], dtype=torch.int32, device=dev))
    ops.check()


def per_scale(r, cu, total, D):
    """Each element's block scale (fp32 values widened), [total, H, D], and the fp32 scales."""
    sc32 = np.nan_to_num(r["scale"], nan=1.0).astype(np.float32).astype(np.float64)
    out = np.ones((total, sc32.shape[0], D))
    base = VF.block_base(cu)
    for si, (s0, n) in enumerate(oracle_varlen.segments(cu)):
        if n:
            blk = base[si] + np.arange(n) // 128
            out[s0:s0 + n] = sc32.T[blk][:, :, None]
    return out, sc32


def run_attention(cu, H, D, causal, case):
    cu = np.asarray(cu, dtype=np.int32)
    total = int(cu[-1])
    q, k, v = packed(total, H, D, case)
    s = signs(case, D).astype(np.float64)
    rq, rk, rv = VF.quantise_varlen(to64(q), cu, s), VF.quantise_varlen(to64(k), cu, s), VF.quantise_varlen(to64(v), cu)
    dev = torch.device("cuda")
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    sc = [per_scale(r, cu, total, D) for r in (rq, rk, rv)]
    o, lse = ops.attn_fwd_varlen_fp8(up(rq["codes"]), up(rk["codes"]), up(rv["codes"]),
                                     *(up(c[1].astype(np.float32)) for c in sc), up(cu),
                                     max(1, int(np.diff(cu).max())), causal=causal)
    ops.check()
    qd, kd, vd = (r["q"] * c[0] for r, c in zip((rq, rk, rv), sc))
    ref = fp8_bound.reference_varlen(qd, kd, vd, sc[2][1], cu, 1 / np.sqrt(D), causal)
    return to64(o)[None], to64(lse)[None], ref


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mix", sorted(MIXES))
def test_attention_matches_oracle(mix, causal, D):
    o, lse, ref = run_attention(MIXES[mix], 2, D, causal, case=93)
    fp8_bound.check(o, lse, ref)


def test_equal_lengths_are_attn_fwd_fp8():
    B, S, H, D = 4, 256, 2, 128
    q, k, v = synth.make_qkv(B, S, H, D, case=94)
    dev = torch.device("cuda")
    cu = torch.arange(0, B * S + 1, S, dtype=torch.int32, device=dev)
    sg = torch.from_numpy(signs(94, D)).to(dev)
    fixed = [ops.hadamard_rotate_quant_fp8(t.to(dev), sg if i < 2 else None) for i, t in enumerate((q, k, v))]
    packed_q = [ops.hadamard_rotate_quant_fp8_varlen(t.to(dev).reshape(B * S, H, D), cu, sg if i < 2 else None)
                for i, t in enumerate((q, k, v))]
    for causal in (False, True):
        a, la = ops.attn_fwd_fp8(*(f[0] for f in fixed), *(f[1] for f in fixed), causal=causal)
        b, lb = ops.attn_fwd_varlen_fp8(*(t[0] for t in packed_q), *(t[1] for t in packed_q), cu, S, causal=causal)
        ops.check()
        assert torch.equal(a.reshape(B * S, H, D), b)
        assert torch.equal(la.permute(1, 0, 2).reshape(H, B * S), lb)


def test_end_to_end_from_the_quantiser():
    # GPU packed quantiser -> GPU attention, element by element against exact attention on the
    # oracle's de-quantised values, the bounds widened by the tie widths of the codes
    cu = np.asarray(MIXES["tiles"], dtype=np.int32)
    H, D = 2, 128
    total = int(cu[-1])
    q, k, v = packed(total, H, D, case=95)
    s = signs(95, D)
    dev = torch.device("cuda")
    cud, sg = torch.from_numpy(cu).to(dev), torch.from_numpy(s).to(dev)
    q8, sq = ops.hadamard_rotate_quant_fp8_varlen(q.to(dev), cud, sg)
    k8, sk = ops.hadamard_rotate_quant_fp8_varlen(k.to(dev), cud, sg)
    v8, sv = ops.hadamard_rotate_quant_fp8_varlen(v.to(dev), cud, None)
    o, lse = ops.attn_fwd_varlen_fp8(q8, k8, v8, sq, sk, sv, cud, causal=True)
    ops.check()
    s64 = s.astype(np.float64)
    res = [VF.quantise_varlen(to64(q), cu, s64), VF.quantise_varlen(to64(k), cu, s64), VF.quantise_varlen(to64(v), cu)]
    for r, g in zip(res, (q8, k8, v8)):
        helpers.check_codes(g.cpu().numpy(), r, 1e-5, 1e-12)
    sc = [per_scale(r, cu, total, D) for r in res]
    deq = [r["q"] * c[0] for r, c in zip(res, sc)]
    widths = [fp8_bound.tie_widths(r["pre"], c[0]) for r, c in zip(res, sc)]
    ref = fp8_bound.reference_varlen(*deq, sc[2][1], cu, 1 / np.sqrt(D), True,
                                     dq=widths[0], dk=widths[1], dv=widths[2])
    fp8_bound.check(to64(o)[None], to64(lse)[None], ref)


@pytest.mark.parametrize("rotate", [False, True])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("mix", sorted(MIXES))
def test_rope_quantiser_matches_oracle(mix, D, rotate):
    # RoPE in front, positions restarting at every sequence; codes within the fused RoPE
    # quantiser's tie rule (its fp32 rotary arithmetic is a few ulps from fp64)
    cu = np.asarray(MIXES[mix], dtype=np.int32)
    x = packed(int(cu[-1]), 3, D, case=96)[0]
    s = signs(96, D) if rotate else None
    dev = torch.device("cuda")
    max_len = int(np.diff(cu).max())
    cs = ops.rope_cos_sin_table(128 * ((max_len + 127) // 128), D)
    codes, scale = ops.rope_hadamard_rotate_quant_fp8_varlen(x.to(dev), cs, torch.from_numpy(cu).to(dev),
                                                             torch.from_numpy(s).to(dev) if rotate else None)
    ops.check()
    ref = VF.quantise_varlen(to64(x), cu, None if s is None else s.astype(np.float64), rope_base=10000.0)
    live = ~np.isnan(ref["scale"])
    np.testing.assert_allclose(scale.cpu().double().numpy()[live], ref["scale"][live], rtol=1e-5, atol=0)
    helpers.check_codes(codes.cpu().numpy(), ref, 1e-5, 5e-4)


def test_rope_table_too_short_writes_nothing():
    dev = torch.device("cuda")
    x = packed(400, 2, 128, case=97)[0].to(dev)
    cu = torch.tensor([0, 100, 400], dtype=torch.int32, device=dev)    # 300 tokens need 384 rows
    cs = ops.rope_cos_sin_table(256, 128)
    out = torch.full((400, 2, 128), 7, dtype=torch.uint8, device=dev)
    sc = torch.full((2, ops.varlen_scale_blocks(400, 2)), 7.0, device=dev)
    ops.rope_hadamard_rotate_quant_fp8_varlen(x, cs, cu, None, out=out, scale=sc)
    with pytest.raises(_lib.AttnError) as e:
        ops.check()
    assert e.value.status == 1
    assert bool((out == 7).all()) and bool((sc == 7.0).all())
    ops.rope_hadamard_rotate_quant_fp8_varlen(x, ops.rope_cos_sin_table(384, 128), cu)
    ops.check()
