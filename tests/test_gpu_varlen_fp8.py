"""The FP8 path on packed variable-length batches vs the fp64 oracle, through the C ABI (GPU).

Quantiser: codes and scales as in the fixed-length quantiser tests (ties aside, bit-identical
codes; scales to 2e-6), over length mixes with empty sequences, single tokens and every
remainder mod 128; one sequence is the fixed-length quantiser bit for bit; bad offsets write
nothing.  Attention: the kernel gets the oracle's own codes and scales, and
RMS(O - O_deq) <= 2 * RMS(O_emul - O_deq) + RMS(half a bf16 ulp of O_deq) + 1e-4 with O_deq
exact attention on the de-quantised values and O_emul the oracle's FP8 reading (numerators
rounded with V's block ratios over the sequence's blocks); lse within 1e-3.  Equal lengths are
attn_fwd_fp8 bit for bit.
"""

import numpy as np
import pytest
import torch

from exact_attention_46_gb300 import _lib, ops, synth
from oracle import varlen as oracle_varlen
from oracle import varlen_fp8 as VF
from tests import helpers
from tests.helpers import half_ulp_bf16, to64

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


def rms(x):
    return float(np.sqrt(np.mean(np.square(x))))


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
    helpers.check_codes(codes.cpu().numpy(), ref, 1e-5, 1e-12, 1e-5)


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


def deq32(r, cu):
    """The oracle's E4M3 values times their block scales rounded to fp32 (what the kernel sees)."""
    sc32 = r["scale"].astype(np.float32).astype(np.float64)
    out = np.zeros_like(r["q"])
    base = VF.block_base(cu)
    for si, (s0, n) in enumerate(oracle_varlen.segments(cu)):
        if n:
            blk = base[si] + np.arange(n) // 128
            out[s0:s0 + n] = r["q"][s0:s0 + n] * sc32.T[blk][:, :, None]
    return out, sc32


def run_attention(cu, H, D, causal, case):
    cu = np.asarray(cu, dtype=np.int32)
    q, k, v = packed(int(cu[-1]), H, D, case)
    s = signs(case, D).astype(np.float64)
    rq, rk, rv = VF.quantise_varlen(to64(q), cu, s), VF.quantise_varlen(to64(k), cu, s), VF.quantise_varlen(to64(v), cu)
    dev = torch.device("cuda")
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    scales = [up(np.nan_to_num(r["scale"], nan=1.0).astype(np.float32)) for r in (rq, rk, rv)]
    o, lse = ops.attn_fwd_varlen_fp8(up(rq["codes"]), up(rk["codes"]), up(rv["codes"]), *scales, up(cu),
                                     max(1, int(np.diff(cu).max())), causal=causal)
    ops.check()
    (qd, _), (kd, _), (vd, vs32) = deq32(rq, cu), deq32(rk, cu), deq32(rv, cu)
    sc = 1 / np.sqrt(D)
    O_deq, lse_deq = VF.fp8_attention_varlen(qd, kd, vd, vs32, cu, sc, causal, round_p=False)
    O_emul, _ = VF.fp8_attention_varlen(qd, kd, vd, vs32, cu, sc, causal)
    return to64(o), to64(lse), O_deq, O_emul, lse_deq


def check(o, lse, O_deq, O_emul, lse_deq):
    assert np.isfinite(o).all()
    e_gpu, e_emul = rms(o - O_deq), rms(O_emul - O_deq)
    bound = 2 * e_emul + rms(half_ulp_bf16(O_deq)) + 1e-4
    assert e_gpu <= bound, (e_gpu, e_emul, bound)
    assert float(np.abs(lse - lse_deq).max()) <= 1e-3


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mix", sorted(MIXES))
def test_attention_matches_oracle(mix, causal, D):
    check(*run_attention(MIXES[mix], 2, D, causal, case=93))


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
    # GPU quantiser -> GPU attention against exact attention on the bf16 inputs: the error of the
    # E4M3 inputs (e_in, exact attention on the oracle's quantisation) plus the bound above
    cu = np.asarray(MIXES["tiles"], dtype=np.int32)
    H, D = 2, 128
    q, k, v = packed(int(cu[-1]), H, D, case=95)
    s = signs(95, D)
    dev = torch.device("cuda")
    cud, sg = torch.from_numpy(cu).to(dev), torch.from_numpy(s).to(dev)
    q8, sq = ops.hadamard_rotate_quant_fp8_varlen(q.to(dev), cud, sg)
    k8, sk = ops.hadamard_rotate_quant_fp8_varlen(k.to(dev), cud, sg)
    v8, sv = ops.hadamard_rotate_quant_fp8_varlen(v.to(dev), cud, None)
    o, lse = ops.attn_fwd_varlen_fp8(q8, k8, v8, sq, sk, sv, cud, causal=True)
    ops.check()
    O_ref, lse_ref = oracle_varlen.attention_varlen(to64(q), to64(k), to64(v), cu, causal=True)
    s64 = s.astype(np.float64)
    rq, rk, rv = VF.quantise_varlen(to64(q), cu, s64), VF.quantise_varlen(to64(k), cu, s64), VF.quantise_varlen(to64(v), cu)
    (qd, _), (kd, _), (vd, vs32) = deq32(rq, cu), deq32(rk, cu), deq32(rv, cu)
    O_deq, lse_deq = VF.fp8_attention_varlen(qd, kd, vd, vs32, cu, 1 / np.sqrt(D), True, round_p=False)
    O_emul, _ = VF.fp8_attention_varlen(qd, kd, vd, vs32, cu, 1 / np.sqrt(D), True)
    e_in, e_p = rms(O_deq - O_ref), rms(O_emul - O_deq)
    bound = e_in + 2 * e_p + rms(half_ulp_bf16(O_deq)) + 1e-4
    assert rms(to64(o) - O_ref) <= bound, (rms(to64(o) - O_ref), e_in, e_p)
    assert float(np.abs(to64(lse) - lse_ref).max()) <= float(np.abs(lse_deq - lse_ref).max()) + 1e-3


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
    helpers.check_codes(codes.cpu().numpy(), ref, 1e-5, 5e-4, 1e-4)


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
