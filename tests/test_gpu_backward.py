"""Backward pass (dQ, dK, dV) vs the fp64 oracle, through the C ABI (GPU).

The forward runs on the GPU (its bf16 O and fp32 lse are what attn_bwd consumes, as in
training); the oracle computes the exact gradients from the same bf16 Q, K, V, dO in fp64.

Tolerance, from the arithmetic.  The kernel's products are exact and its sums fp32; what it
rounds is one bf16 operand per gradient GEMM (P for dV, dS for dQ and dK), the bf16 O that
enters Delta, and the bf16 result.  bf16 has 8 significant bits, so each rounding has
relative error at most eps = 2^-8.  Element-wise, with |.| taken entry by entry:
    |dV - dV*| <= ulp/2 + eps * P^T |dO|
    |dQ - dQ*| <= ulp/2 + eps * scale * (|dS| |K| + diag(E) P |K|),   E_i = sum_d |dO_id O_id|
    |dK - dK*| <= ulp/2 + eps * scale * (|dS|^T |Q| + P^T diag(E) |Q|)
(ulp/2 = half a bf16 ulp of the exact value; a 5 % margin covers the fp32 terms).  With
independent rounding errors the RMS error is far below these worst cases: about
2^-8 / sqrt(3) = 2.3e-3 of RMS(ref) from the operand plus ~1.5e-3 from the output rounding;
the test also bounds RMS(err) <= 4e-3 * max(RMS(ref), 1e-3) (the floor covers one visible key,
where the exact dQ = dK = 0 and the kernel returns the fp32 residue of dP - Delta, ~1e-8).
"""

import numpy as np
import pytest
import torch

from exact_attention_46_gb300 import ops, synth
from oracle import attention as oracle_attention
from oracle import backward as oracle_backward
from tests.helpers import half_ulp_bf16, to64

pytestmark = pytest.mark.gpu

EPS = 2.0 ** -8
RMS_REL = 4e-3


def error_bounds(q, k, v, do, causal):
    """Worst-case rounding bounds (see the module docstring), [B, S, H, D] each."""
    B, S, H, D = q.shape
    scale = 1.0 / np.sqrt(D)
    bq, bk, bv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            P, _, _ = oracle_attention.attention_weights(q[b, :, h], k[b, :, h], scale, causal)
            o = P @ v[b, :, h]
            g = do[b, :, h]
            dS = P * (g @ v[b, :, h].T - (g * o).sum(axis=1)[:, None])
            E = np.abs(g * o).sum(axis=1)
            aq, ak = np.abs(q[b, :, h]), np.abs(k[b, :, h])
            bv[b, :, h] = P.T @ np.abs(g)
            bq[b, :, h] = scale * (np.abs(dS) @ ak + E[:, None] * (P @ ak))
            bk[b, :, h] = scale * (np.abs(dS).T @ aq + P.T @ (E[:, None] * aq))
    return bq, bk, bv


def grads(B, S, H, D, causal, case):
    q, k, v = synth.make_qkv(B, S, H, D, case)
    do = torch.from_numpy(synth.normal((B, S, H, D), synth.seed_for(case, synth.STREAM_OUT_VAL))).to(torch.bfloat16)
    dev = torch.device("cuda")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = ops.attn_fwd(qd, kd, vd, causal=causal)
    dq, dk, dv = ops.attn_bwd(qd, kd, vd, o, lse, dod, causal=causal)
    ops.check()
    args = (to64(q), to64(k), to64(v), to64(do))
    ref = oracle_backward.attention_backward(*args, causal=causal)
    return (dq, dk, dv), ref, error_bounds(*args, causal)


def check(gpu, ref, bounds):
    for name, g, r, bnd in zip(("dq", "dk", "dv"), gpu, ref, bounds):
        g64 = to64(g)
        assert np.isfinite(g64).all(), name
        err = np.abs(g64 - r)
        excess = err - (half_ulp_bf16(r) + 1.05 * EPS * bnd + 1e-7)
        assert excess.max() <= 0, (name, float(excess.max()), float((err / (EPS * bnd + 1e-30)).max()))
        rms = float(np.sqrt(np.mean(err ** 2)))
        scale = max(float(np.sqrt(np.mean(r ** 2))), 1e-3)
        assert rms <= RMS_REL * scale, (name, rms / scale)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [1, 100, 128, 129, 256, 300, 513])
def test_full_small(S, D, causal):
    check(*grads(2, S, 3, D, causal, case=50))


@pytest.mark.parametrize("causal", [False, True])
def test_longer_sequence(causal):
    check(*grads(1, 2048, 4, 128, causal, case=51))


@pytest.mark.parametrize("causal", [False, True])
def test_more_ctas_than_sms(causal):
    check(*grads(4, 700, 16, 64, causal, case=52))


def test_deterministic():
    (a, _, _), (b, _, _) = grads(1, 640, 2, 128, True, case=53), grads(1, 640, 2, 128, True, case=53)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
