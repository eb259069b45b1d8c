"""FP8 grouped-query attention -- prefill (attn_fwd_gqa_fp8) and decoding (attn_decode_fp8) --
vs the fp64 oracle, through the C ABI (GPU).

The kernels get the oracle's own E4M3 codes and block scales (Q and K rotated by the same
random signs, V not rotated), so both sides see the same inputs.  O_deq is exact grouped
attention on the de-quantised values and O_emul the oracle's FP8 reading, which also rounds
the softmax numerators to E4M3 (relative to the exact row max; the kernel rounds relative to
its running max, split by split -- independent roundings of the same size).  The check:

    RMS(O_gpu - O_deq) <= 2 * RMS(O_emul - O_deq) + RMS(half a bf16 ulp of O_deq) + 1e-4

(the middle term is the bf16 rounding of the output, which is all there is for one key),
and lse, which the numerator rounding does not touch, within 1e-3 of the exact one.
"""

import numpy as np
import pytest
import torch

from exact_attention_46_gb300 import ops, synth
from oracle import gqa as oracle_gqa
from oracle import quantise
from tests.helpers import half_ulp_bf16, to64

pytestmark = pytest.mark.gpu

LSE_TOL = 1e-3


def raw_inputs(B, Sq, Sk, Hq, Hkv, D, case, block_gain=False):
    """fp32 Q [B, Sq, Hq, D], K, V [B, Sk, Hkv, D]; block_gain multiplies each 128-key block of
    K and V by its own power of two (2^-3 .. 2^3) so that the block scales differ."""
    q = synth.normal((B, Sq, Hq, D), synth.seed_for(case, synth.STREAM_Q))
    k = synth.normal((B, Sk, Hkv, D), synth.seed_for(case, synth.STREAM_K))
    v = synth.normal((B, Sk, Hkv, D), synth.seed_for(case, synth.STREAM_V))
    if block_gain:
        g = np.exp2((np.arange(Sk) // 128) % 7 - 3.0).astype(np.float32)[None, :, None, None]
        k = k * np.float32(0.5) * g
        v = v * g[:, ::-1] if Sk > 1 else v
    return q.astype(np.float32), np.ascontiguousarray(k, np.float32), np.ascontiguousarray(v, np.float32)


def quantised(x, signs):
    """The oracle's codes (uint8) and fp32 block scales of x, and their de-quantised values."""
    r = quantise.quantise_blocks(np.asarray(x, np.float64), signs)
    sc32 = r["scale"].astype(np.float32)
    return r["codes"], sc32, quantise.dequantise(r["q"], sc32.astype(np.float64))


def run(B, Sq, Sk, Hq, Hkv, D, causal, case, block_gain=False, rotate=True, fn=None):
    q, k, v = raw_inputs(B, Sq, Sk, Hq, Hkv, D, case, block_gain)
    s = synth.signs(D, synth.seed_for(case, synth.STREAM_SIGNS)).astype(np.float64) if rotate else None
    (q8, sq, qd), (k8, sk, kd), (v8, sv, vd) = quantised(q, s), quantised(k, s), quantised(v, None)
    dev = torch.device("cuda")
    t = [torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in (q8, k8, v8, sq, sk, sv)]
    o, lse = (fn or ops.attn_decode_fp8)(*t, causal=causal)
    ops.check()
    O_deq, lse_deq = oracle_gqa.attention_gqa(qd, kd, vd, causal=causal)
    O_emul, _ = oracle_gqa.attention_gqa(qd, kd, vd, causal=causal, round_p=True)
    return to64(o), to64(lse), O_deq, O_emul, lse_deq


def rms(x):
    return float(np.sqrt(np.mean(np.square(x))))


def check(o, lse, O_deq, O_emul, lse_deq):
    assert np.isfinite(o).all()
    e_gpu, e_emul = rms(o - O_deq), rms(O_emul - O_deq)
    bound = 2 * e_emul + rms(half_ulp_bf16(O_deq)) + 1e-4
    assert e_gpu <= bound, (e_gpu, e_emul, bound)
    lse_err = float(np.abs(lse - lse_deq).max())
    assert lse_err <= LSE_TOL, lse_err


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S,Hkv", [(1, 1), (100, 1), (300, 2), (513, 8)])
def test_gqa_fp8_prefill_matches_oracle(S, Hkv, D, causal):
    check(*run(2, S, S, 8, Hkv, D, causal, case=85, fn=ops.attn_fwd_gqa_fp8))


def test_gqa_fp8_prefill_block_scales_that_differ():
    check(*run(1, 1000, 1000, 8, 2, 128, True, case=86, block_gain=True, fn=ops.attn_fwd_gqa_fp8))


def test_gqa_fp8_with_one_group_per_head_is_attn_fwd_fp8():
    B, S, H, D = 2, 700, 4, 128
    q, k, v = raw_inputs(B, S, S, H, H, D, case=87)
    dev = torch.device("cuda")
    t = [torch.from_numpy(np.ascontiguousarray(a)).to(dev)
         for r in (quantised(q, None), quantised(k, None), quantised(v, None)) for a in r[:2]]
    q8, sq, k8, sk, v8, sv = t
    a, la = ops.attn_fwd_gqa_fp8(q8, k8, v8, sq, sk, sv, causal=True)
    b, lb = ops.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, causal=True)
    ops.check()
    assert torch.equal(a, b) and torch.equal(la, lb)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Sq,Sk,Hq,Hkv", [
    (1, 1, 1, 8, 8), (2, 1, 100, 8, 2), (2, 1, 129, 32, 8), (1, 4, 1000, 16, 2), (3, 16, 300, 8, 1),
    (2, 8, 4097, 16, 1), (1, 1, 65536, 4, 1), (4, 2, 20000, 32, 4), (1, 128, 2000, 1, 1),
    (2, 6, 3000, 8, 1), (1, 2, 700, 32, 1), (1, 33, 500, 1, 1),
    (1, 17, 900, 1, 1), (2, 1, 3000, 16, 1)])
def test_decode_fp8_matches_oracle(B, Sq, Sk, Hq, Hkv, D, causal):
    check(*run(B, Sq, Sk, Hq, Hkv, D, causal, case=80))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Sk", [1000, 30000])
def test_decode_fp8_block_scales_that_differ(Sk, D):
    # per-block gains of 2^-3 .. 2^3: the value scale of each tile enters the exponent
    # as log2(sv_j / max sv) and the key scale the logit multiplier
    check(*run(2, 2, Sk, 16, 2, D, True, case=81, block_gain=True))


def test_decode_fp8_without_rotation():
    check(*run(2, 1, 3000, 8, 1, 128, False, case=82, rotate=False))


def test_decode_fp8_from_the_quantiser():
    # the GPU quantiser feeds the decoding kernel.  Rotated Q and K give the logits of the
    # unrotated inputs, so against exact attention on the original bf16 values the error is
    # that of the E4M3 inputs (e_in: exact attention on the oracle's quantisation of the same
    # values) plus the kernel's own bound above (triangle inequality); the GPU quantiser's
    # codes are the oracle's but for rounding ties
    B, Sq, Sk, Hq, Hkv, D = 2, 1, 5000, 16, 2, 128
    q, k, v = raw_inputs(B, Sq, Sk, Hq, Hkv, D, case=83)
    qb, kb, vb = (torch.from_numpy(a).to(torch.bfloat16) for a in (q, k, v))
    s = synth.signs(D, synth.seed_for(83, synth.STREAM_SIGNS))
    dev = torch.device("cuda")
    sg = torch.from_numpy(s).to(dev)
    q8, sq = ops.hadamard_rotate_quant_fp8(qb.to(dev), sg)
    k8, sk = ops.hadamard_rotate_quant_fp8(kb.to(dev), sg)
    v8, sv = ops.hadamard_rotate_quant_fp8(vb.to(dev), None)
    o, lse = ops.attn_decode_fp8(q8, k8, v8, sq, sk, sv, causal=True)
    ops.check()
    O_ref, lse_ref = oracle_gqa.attention_gqa(to64(qb), to64(kb), to64(vb), causal=True)
    s64 = s.astype(np.float64)
    qd, kd, vd = quantised(to64(qb), s64)[2], quantised(to64(kb), s64)[2], quantised(to64(vb), None)[2]
    O_deq, lse_deq = oracle_gqa.attention_gqa(qd, kd, vd, causal=True)
    O_emul, _ = oracle_gqa.attention_gqa(qd, kd, vd, causal=True, round_p=True)
    e_in, e_p = rms(O_deq - O_ref), rms(O_emul - O_deq)
    bound = e_in + 2 * e_p + rms(half_ulp_bf16(O_deq)) + 1e-4
    assert rms(to64(o) - O_ref) <= bound, (rms(to64(o) - O_ref), e_in, e_p)
    assert float(np.abs(to64(lse) - lse_ref).max()) <= float(np.abs(lse_deq - lse_ref).max()) + LSE_TOL


def test_decode_fp8_without_lse_and_repeatable():
    B, Sq, Sk, Hq, Hkv, D = 2, 3, 5000, 16, 4, 128
    q, k, v = raw_inputs(B, Sq, Sk, Hq, Hkv, D, case=84)
    dev = torch.device("cuda")
    t = [torch.from_numpy(np.ascontiguousarray(a)).to(dev)
         for r in (quantised(q, None), quantised(k, None), quantised(v, None)) for a in r[:2]]
    q8, sq, k8, sk, v8, sv = t
    a, la = ops.attn_decode_fp8(q8, k8, v8, sq, sk, sv, causal=True)
    b, lb = ops.attn_decode_fp8(q8, k8, v8, sq, sk, sv, causal=True, want_lse=False)
    ops.check()
    assert lb is None and torch.equal(a, b)


def test_decode_fp8_zero_value_scales():
    # one V block with scale 0 and one key/value head whose V scales are all 0
    B, Sq, Sk, Hq, Hkv, D = 2, 1, 3000, 8, 2, 128
    q, k, v = raw_inputs(B, Sq, Sk, Hq, Hkv, D, case=88)
    (q8, sq, qd), (k8, sk, kd), (v8, sv, _) = quantised(q, None), quantised(k, None), quantised(v, None)
    sv = sv.copy()
    sv[0, 0, 5] = 0.0
    sv[1, 1, :] = 0.0
    rv = quantise.quantise_blocks(np.asarray(v, np.float64))
    vd = quantise.dequantise(rv["q"], sv.astype(np.float64))
    dev = torch.device("cuda")
    t = [torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in (q8, k8, v8, sq, sk, sv)]
    o, lse = ops.attn_decode_fp8(*t, causal=True)
    ops.check()
    O_deq, lse_deq = oracle_gqa.attention_gqa(qd, kd, vd, causal=True)
    O_emul, _ = oracle_gqa.attention_gqa(qd, kd, vd, causal=True, round_p=True)
    og = to64(o)
    assert np.all(og[1, :, 4:8] == 0.0)                     # query heads of key/value head 1, batch 1
    check(og, to64(lse), O_deq, O_emul, lse_deq)
