"""FP8 path vs the fp64 oracle, through the C ABI (GPU).

Quantiser: block scales agree to 2e-6 relative; E4M3 codes are bit-identical except where
the oracle's exact pre-rounding value lies within 1e-5 (relative) of a rounding midpoint --
there the kernel's fp32 transform may land on either side, and the test checks that the two
codes are the neighbouring grid values around that midpoint.

FP8 attention: the only rounding the oracle's FP8 path has beyond the quantised inputs is the
E4M3 rounding of the softmax numerators, with V's block ratios sv_j / max sv folded in as the
kernel folds them (``fold_v``); the kernel rounds relative to its running max rather than the
exact row max, so the two roundings are independent draws of the same size.
The check: RMS(O_gpu - O_deq) <= 2 * RMS(O_emul - O_deq) + 1e-4, where O_deq is exact
attention on the de-quantised inputs and O_emul the oracle's FP8 path; lse (which the
rounding does not touch) within 1e-3 of the oracle's.
"""

import numpy as np
import pytest
import torch

from exact_attention_46_gb300 import ops, synth
from oracle import attention as oracle_attention
from oracle import e4m3, fp8_path, quantise
from tests import helpers
from tests.helpers import inputs, sample_rows, stats, to64

pytestmark = pytest.mark.gpu

SCALE_RTOL = 2e-6
TIE_RTOL = 1e-5


def signs_for(case, D):
    return synth.signs(D, synth.seed_for(case, synth.STREAM_SIGNS))


def check_codes(gpu_codes, ref):
    return helpers.check_codes(gpu_codes, ref, TIE_RTOL, 1e-12, 1e-5)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("rotate", [False, True])
@pytest.mark.parametrize("S", [1, 128, 300, 1024])
def test_quantiser_matches_oracle(S, D, rotate):
    B, H = 2, 3
    x = inputs(B, S, H, D, case=20, dist="outliers")[0]
    s = signs_for(20, D) if rotate else None
    codes, scale = ops.hadamard_rotate_quant_fp8(x.cuda(), torch.from_numpy(s).cuda() if rotate else None)
    ops.check()
    ref = quantise.quantise_blocks(to64(x), None if s is None else s.astype(np.float64))
    np.testing.assert_allclose(scale.cpu().double().numpy(), ref["scale"], rtol=SCALE_RTOL, atol=0)
    check_codes(codes.cpu().numpy(), ref)


def test_quantiser_zero_block_and_benchmark_size():
    B, S, H, D = 16, 1024, 16, 128
    x = inputs(B, S, H, D, case=21, dist="outliers")[0]
    x[0, 0:128, 3] = 0
    s = signs_for(21, D)
    codes, scale = ops.hadamard_rotate_quant_fp8(x.cuda(), torch.from_numpy(s).cuda())
    ops.check()
    assert scale[0, 3, 0].item() == 1.0 and int(codes[0, 0:128, 3].max()) == 0
    ref = quantise.quantise_blocks(to64(x), s.astype(np.float64))
    np.testing.assert_allclose(scale.cpu().double().numpy(), ref["scale"], rtol=SCALE_RTOL)
    check_codes(codes.cpu().numpy(), ref)


def run_fp8_path(q, k, v, s, causal):
    dev = torch.device("cuda")
    sd = torch.from_numpy(s).to(dev) if s is not None else None
    q8, sq = ops.hadamard_rotate_quant_fp8(q.to(dev), sd)
    k8, sk = ops.hadamard_rotate_quant_fp8(k.to(dev), sd)
    v8, sv = ops.hadamard_rotate_quant_fp8(v.to(dev), None)
    o, lse = ops.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, causal=causal)
    ops.check()
    return o, lse


def oracle_fp8(q, k, v, s, causal, rows):
    s64 = None if s is None else s.astype(np.float64)
    O_emul, lse_emul, (Qq, Kq, Vq) = fp8_path.fp8_attention(to64(q), to64(k), to64(v), s64,
                                                            causal=causal, rows=rows, fold_v=True)
    qd = quantise.dequantise(Qq["q"], Qq["scale"])
    kd = quantise.dequantise(Kq["q"], Kq["scale"])
    vd = quantise.dequantise(Vq["q"], Vq["scale"])
    O_deq, lse_deq = oracle_attention.attention(qd, kd, vd, causal=causal, rows=rows)
    return O_emul, O_deq, lse_deq


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("rotate", [False, True])
@pytest.mark.parametrize("B,S,H,D", [(2, 300, 3, 128), (1, 1024, 4, 128), (2, 513, 2, 64), (1, 640, 2, 256)])
def test_fp8_attention_matches_oracle(B, S, H, D, rotate, causal):
    q, k, v = inputs(B, S, H, D, case=22, dist="outliers")
    s = signs_for(22, D) if rotate else None
    o, lse = run_fp8_path(q, k, v, s, causal)
    O_emul, O_deq, lse_deq = oracle_fp8(q, k, v, s, causal, None)
    _, e_gpu = stats(to64(o), O_deq)
    _, e_emul = stats(O_emul, O_deq)
    assert np.isfinite(to64(o)).all()
    assert e_gpu <= 2 * e_emul + 1e-4, (e_gpu, e_emul)
    assert np.abs(to64(lse) - lse_deq).max() <= 1e-3


@pytest.mark.parametrize("S", [32768, 65536])
def test_fp8_long_context(S):
    # the long-context workload (B=1, H=16, D=128), non-causal and causal, checked on sampled
    # query rows; each side quantises once and both masks use the result
    B, H, D = 1, 16, 128
    q, k, v = inputs(B, S, H, D, case=24)
    s = signs_for(24, D)
    dev = torch.device("cuda")
    sd = torch.from_numpy(s).to(dev)
    q8, sq = ops.hadamard_rotate_quant_fp8(q.to(dev), sd)
    k8, sk = ops.hadamard_rotate_quant_fp8(k.to(dev), sd)
    v8, sv = ops.hadamard_rotate_quant_fp8(v.to(dev), None)
    Qq, Kq, Vq = fp8_path.quantise_qkv(to64(q), to64(k), to64(v), s.astype(np.float64))
    qd = quantise.dequantise(Qq["q"], Qq["scale"])
    kd = quantise.dequantise(Kq["q"], Kq["scale"])
    vd = quantise.dequantise(Vq["q"], Vq["scale"])
    rows = sample_rows(S, n_random=8)
    ratio = fp8_path.v_block_ratio(Vq["scale"], S)
    for causal in (False, True):
        o, lse = ops.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, causal=causal)
        ops.check()
        O_emul, _ = fp8_path.attention_rounded_p(qd, kd, vd, 1 / np.sqrt(D), causal, rows, v_ratio=ratio)
        O_deq, lse_deq = fp8_path.attention_rounded_p(qd, kd, vd, 1 / np.sqrt(D), causal, rows, round_p=False)
        og = to64(o)[:, rows]
        _, e_gpu = stats(og, O_deq)
        _, e_emul = stats(O_emul, O_deq)
        assert np.isfinite(og).all()
        assert e_gpu <= 2 * e_emul + 1e-4, (causal, e_gpu, e_emul)
        assert np.abs(to64(lse)[:, :, rows] - lse_deq).max() <= 1e-3, causal


def test_fp8_unit_scales_through_attn_fwd():
    # E4M3 codes drawn directly (magnitudes <= 2, random signs): no quantiser involved.
    B, S, H, D = 2, 400, 2, 128
    u = synth.uniform((3, B, S, H, D), synth.seed_for(23, 0))
    codes = (np.floor(u * 0x41).astype(np.uint8) | np.where(synth.uniform((3, B, S, H, D), 77) < 0.5, 0x80, 0).astype(np.uint8))
    vals = e4m3.decode(codes)
    dev = torch.device("cuda")
    t = [torch.from_numpy(codes[i].copy()).to(dev) for i in range(3)]
    for causal in (False, True):
        o, lse = ops.attn_fwd(t[0], t[1], t[2], causal=causal)
        ops.check()
        O_emul, lse_emul = fp8_path.attention_rounded_p(vals[0], vals[1], vals[2], 1 / np.sqrt(D), causal)
        O_deq, _ = fp8_path.attention_rounded_p(vals[0], vals[1], vals[2], 1 / np.sqrt(D), causal, round_p=False)
        _, e_gpu = stats(to64(o), O_deq)
        _, e_emul = stats(O_emul, O_deq)
        assert e_gpu <= 2 * e_emul + 1e-4, (e_gpu, e_emul)
        assert np.abs(to64(lse) - lse_emul).max() <= 1e-3


def _experiment(S, case):
    B, H, D = 16384 // S, 16, 128
    q, k, v = inputs(B, S, H, D, case=case, dist="outliers")
    s = signs_for(case, D)
    rows = sample_rows(S, n_random=16)
    O_ref, _ = oracle_attention.attention(to64(q), to64(k), to64(v), rows=rows)
    out = {}
    for name, sg in (("none", None), ("hadamard", s)):
        o, _ = run_fp8_path(q, k, v, sg, False)
        O_emul, _, _ = oracle_fp8(q, k, v, sg, False, rows)
        out[name] = (stats(to64(o)[:, rows], O_ref)[1], stats(O_emul, O_ref)[1])
    r_gpu = out["hadamard"][0] / out["none"][0]
    r_emul = out["hadamard"][1] / out["none"][1]
    print(f"S={S}: RMS none gpu/emul {out['none']}, hadamard gpu/emul {out['hadamard']}, "
          f"ratio gpu {r_gpu:.3f} emul {r_emul:.3f}")
    return r_gpu, r_emul


@pytest.mark.parametrize("S", [1024, 8192])
def test_incoherent_processing_ratio_matches_emulation(S):
    r_gpu, r_emul = _experiment(S, case=40)
    assert r_gpu < 1.0
    assert abs(r_gpu - r_emul) <= 0.1


@pytest.mark.xfail(strict=False, reason="the rotation's error reduction under these readings is "
                   "about 0.6-0.8x, not the <= 0.5x target (the pages report 2.6x)")
def test_incoherent_processing_halves_error():
    r_gpu, _ = _experiment(1024, case=41)
    assert r_gpu <= 0.5


def test_zero_value_scales():
    # A V block with scale 0 holds zeros (value = code * scale), and one head's V scales are all
    # 0: O and lse stay finite, the zero block contributes nothing, the all-zero head gives O = 0.
    B, S, H, D = 1, 700, 2, 128
    q, k, v = inputs(B, S, H, D, case=25)
    Qq, Kq, Vq = fp8_path.quantise_qkv(to64(q), to64(k), to64(v), None)
    vs = Vq["scale"].astype(np.float32)
    vs[0, 0, 2] = 0.0
    vs[0, 1, :] = 0.0
    sc32 = [Qq["scale"].astype(np.float32), Kq["scale"].astype(np.float32), vs]
    dev = torch.device("cuda")
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    qd, kd, vd = (quantise.dequantise(r["q"], s.astype(np.float64)) for r, s in zip((Qq, Kq, Vq), sc32))
    ratio = fp8_path.v_block_ratio(sc32[2], S)
    for causal in (False, True):
        o, lse = ops.attn_fwd_fp8(up(Qq["codes"]), up(Kq["codes"]), up(Vq["codes"]), *(up(s) for s in sc32),
                                  causal=causal)
        ops.check()
        O_deq, lse_deq = fp8_path.attention_rounded_p(qd, kd, vd, 1 / np.sqrt(D), causal, round_p=False)
        O_emul, _ = fp8_path.attention_rounded_p(qd, kd, vd, 1 / np.sqrt(D), causal, v_ratio=ratio)
        og = to64(o)
        assert np.isfinite(og).all() and np.isfinite(to64(lse)).all()
        assert np.all(og[:, :, 1] == 0.0)
        _, e_gpu = stats(og, O_deq)
        _, e_emul = stats(O_emul, O_deq)
        assert e_gpu <= 2 * e_emul + 1e-4, (causal, e_gpu, e_emul)
        assert np.abs(to64(lse) - lse_deq).max() <= 1e-3
