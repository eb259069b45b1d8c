"""Grouped-query backward (dQ; dK, dV summed over each group) vs the fp64 oracle, through the
C ABI (GPU).

The forward runs on the GPU (attn_fwd_gqa's bf16 O and fp32 lse feed attn_bwd_gqa); the
oracle differentiates multi-head attention with each key/value head repeated over its group
and sums dK, dV over the group, in fp64 from the same bf16 inputs.

Tolerance.  Per repeated head the kernel makes the roundings the multi-head backward makes
(one bf16 operand per gradient GEMM, the bf16 O in Delta), so the element bound of that
backward holds head by head; dK and dV of a key/value head add G such heads in fp32 and round
to bf16 once, so their bound is half a bf16 ulp plus the SUM of the G heads' operand bounds.
The RMS bound is the multi-head one (the G heads' rounding errors are independent, so their
sum grows like sqrt(G) while the sum of the gradients grows like G or sqrt(G)).
"""

import numpy as np
import pytest
import torch

from exact_attention_46_gb300 import ops, synth
from oracle import backward as oracle_backward
from tests.helpers import half_ulp_bf16, to64
from tests.test_gpu_backward import EPS, RMS_REL, error_bounds

pytestmark = pytest.mark.gpu


def inputs(B, S, Hq, Hkv, D, case):
    sd = synth.seed_for
    q = torch.from_numpy(synth.normal((B, S, Hq, D), sd(case, synth.STREAM_Q))).to(torch.bfloat16)
    k = torch.from_numpy(synth.normal((B, S, Hkv, D), sd(case, synth.STREAM_K))).to(torch.bfloat16)
    v = torch.from_numpy(synth.normal((B, S, Hkv, D), sd(case, synth.STREAM_V))).to(torch.bfloat16)
    do = torch.from_numpy(synth.normal((B, S, Hq, D), sd(case, synth.STREAM_OUT_VAL))).to(torch.bfloat16)
    return q, k, v, do


def gpu_grads(q, k, v, do, causal):
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = ops.attn_fwd_gqa(qd, kd, vd, causal=causal)
    g = ops.attn_bwd_gqa(qd, kd, vd, o, lse, dod, causal=causal)
    ops.check()
    return g


def group_bounds(q, k, v, do, causal):
    """Element bounds: the multi-head bounds of the repeated heads, dK and dV summed per group."""
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    bq, bk, bv = error_bounds(q, np.repeat(k, G, axis=2), np.repeat(v, G, axis=2), do, causal)
    return (bq, bk.reshape(B, S, Hkv, G, D).sum(axis=3), bv.reshape(B, S, Hkv, G, D).sum(axis=3))


def check(gpu, ref, bounds):
    for name, g, r, bnd in zip(("dq", "dk", "dv"), gpu, ref, bounds):
        g64 = to64(g)
        assert g64.shape == r.shape, (name, g64.shape, r.shape)
        assert np.isfinite(g64).all(), name
        err = np.abs(g64 - r)
        excess = err - (half_ulp_bf16(r) + 1.05 * EPS * bnd + 1e-7)
        assert excess.max() <= 0, (name, float(excess.max()), float((err / (EPS * bnd + 1e-30)).max()))
        rms = float(np.sqrt(np.mean(err ** 2)))
        scale = max(float(np.sqrt(np.mean(r ** 2))), 1e-3)
        assert rms <= RMS_REL * scale, (name, rms / scale)


def run(B, S, Hq, Hkv, D, causal, case):
    q, k, v, do = inputs(B, S, Hq, Hkv, D, case)
    gpu = gpu_grads(q, k, v, do, causal)
    args = (to64(q), to64(k), to64(v), to64(do))
    ref = oracle_backward.attention_backward_gqa(*args, causal=causal)
    check(gpu, ref, group_bounds(*args, causal))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S,Hq,Hkv", [(1, 4, 1), (100, 4, 2), (129, 8, 2), (300, 6, 3), (513, 8, 1)])
def test_gqa_backward_small(S, Hq, Hkv, D, causal):
    run(2, S, Hq, Hkv, D, causal, case=70)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_backward_long_group(causal):
    # G = 8 over 16 query tiles: the dK/dV CTA streams 128 tiles (causal: fewer) into one sum
    run(1, 2048, 8, 1, 128, causal, case=71)


@pytest.mark.parametrize("causal", [False, True])
def test_one_head_per_group_is_the_multi_head_backward(causal):
    q, k, v, do = inputs(2, 300, 3, 3, 128, case=72)
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = ops.attn_fwd(qd, kd, vd, causal=causal)
    a = ops.attn_bwd_gqa(qd, kd, vd, o, lse, dod, causal=causal)
    b = ops.attn_bwd(qd, kd, vd, o, lse, dod, causal=causal)
    ops.check()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_gqa_backward_deterministic():
    q, k, v, do = inputs(1, 640, 8, 2, 128, case=73)
    a, b = gpu_grads(q, k, v, do, True), gpu_grads(q, k, v, do, True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
