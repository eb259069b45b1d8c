"""FP8 grouped-query attention -- prefill (attn_fwd_gqa_fp8) and decoding (attn_decode_fp8) --
vs the fp64 oracle, through the C ABI (GPU).

The kernels get the oracle's own E4M3 codes and block scales (Q and K rotated by the same
random signs, V not rotated), so both sides see the same inputs.  Every output element must
lie within the FP8 bounds of tests/fp8_bound.py against exact grouped attention on the
de-quantised values (the decoding kernel takes V's largest block scale per key split, which
only raises the ratios r_j the bound divides by); lse within 1e-3 of the exact one.  The
bounds' reference is checked against the oracle's grouped attention (oracle/gqa.py, pinned
against torch in the CPU tests) on every case.
"""

import numpy as np
import pytest
import torch

from exact_attention_46_gb300 import ops, synth
from oracle import gqa as oracle_gqa
from oracle import quantise
from tests import fp8_bound
from tests.helpers import check_codes, to64

pytestmark = pytest.mark.gpu


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
    return to64(o), to64(lse), reference(qd, kd, vd, sv, D, causal)


def reference(qd, kd, vd, sv, D, causal):
    ref = fp8_bound.reference(qd, kd, vd, sv, 1 / np.sqrt(D), causal)
    O_gqa, lse_gqa = oracle_gqa.attention_gqa(qd, kd, vd, causal=causal)
    np.testing.assert_allclose(ref["O"], O_gqa, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(ref["lse"], lse_gqa, rtol=1e-10, atol=1e-12)
    return ref


def check(o, lse, ref):
    fp8_bound.check(o, lse, ref)


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
    # the GPU quantiser feeds the decoding kernel; element by element against exact grouped
    # attention on the oracle's de-quantised values, the bounds widened by the tie widths of
    # the codes (the GPU quantiser's codes are the oracle's but for rounding midpoints)
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
    s64 = s.astype(np.float64)
    res = [quantise.quantise_blocks(to64(qb), s64), quantise.quantise_blocks(to64(kb), s64),
           quantise.quantise_blocks(to64(vb), None)]
    for r, g in zip(res, (q8, k8, v8)):
        check_codes(g.cpu().numpy(), r, 1e-5, 1e-12)
    deq = [quantise.dequantise(r["q"], r["scale"]) for r in res]
    widths = [fp8_bound.tie_widths_blocks(r) for r in res]
    ref = fp8_bound.reference(*deq, res[2]["scale"], 1 / np.sqrt(D), True, dq=widths[0], dk=widths[1], dv=widths[2])
    fp8_bound.check(to64(o), to64(lse), ref)


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
    og = to64(o)
    assert np.all(og[1, :, 4:8] == 0.0)                     # query heads of key/value head 1, batch 1
    check(og, to64(lse), reference(qd, kd, vd, sv, D, True))
