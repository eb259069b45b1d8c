"""BF16 fused attention vs the fp64 oracle, through the C ABI (GPU).

Bounds (N(0,1) inputs): max |O - O_ref| <= 1e-2 beyond half a bf16 ulp of O_ref (the rounding
of the exact result to the bf16 output, which alone reaches 0.0078 at |O| >= 2), RMS <= 2e-3,
max |lse - lse_ref| <= 1e-3.
Full rows at small sizes spanning several 128-tiles and a ragged tail; sampled rows at the
benchmark sizes (D = 128, H = 16, B = 16384 / S), the causal head-dimension sweep and the
long-context sizes.
"""

import numpy as np
import pytest
import torch

from exact_attention_46_gb300 import ops
from oracle import attention as oracle_attention
from tests.helpers import BF16_MAX_ABS, BF16_RMS, LSE_MAX_ABS, bf16_stats, inputs, sample_rows, stats, to64

pytestmark = pytest.mark.gpu


def run_and_check(B, S, H, D, causal, case, rows=None, dist="normal", tol=None):
    q, k, v = inputs(B, S, H, D, case, dist)
    dev = torch.device("cuda")
    o, lse = ops.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal)
    ops.check()
    O_ref, lse_ref = oracle_attention.attention(to64(q), to64(k), to64(v), causal=causal, rows=rows)
    o64, lse64 = to64(o), to64(lse)
    if rows is not None:
        o64, lse64 = o64[:, rows], lse64[:, :, rows]
    max_abs, rms, _ = bf16_stats(o64, O_ref)
    lse_err = float(np.abs(lse64 - lse_ref).max())
    mx, rm, le = tol or (BF16_MAX_ABS, BF16_RMS, LSE_MAX_ABS)
    assert np.isfinite(o64).all() and np.isfinite(lse64).all()
    assert max_abs <= mx and rms <= rm and lse_err <= le, (max_abs, rms, lse_err)
    return max_abs, rms, lse_err


def test_tiny_config():
    run_and_check(1, 128, 2, 64, False, case=0)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [1, 100, 128, 129, 255, 256, 300, 513])
def test_full_rows_small(S, D, causal):
    run_and_check(2, S, 3, D, causal, case=1)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_full_rows_more_items_than_sms(D, causal):
    # 8 * 24 heads * ceil(300 / rows per CTA) items > 152 CTAs: every CTA of the persistent
    # kernel walks several items, and the ragged tail sits in the last query block.
    run_and_check(8, 300, 24, D, causal, case=11)


@pytest.mark.parametrize("S", [512, 1024, 2048, 4096, 8192, 16384])
def test_benchmark_sizes_d128(S):
    run_and_check(16384 // S, S, 16, 128, False, case=2, rows=sample_rows(S))


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("S", [1024, 2048, 4096, 8192, 16384])
def test_causal_head_dims(S, D):
    run_and_check(16384 // S, S, 2048 // D, D, True, case=3, rows=sample_rows(S))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [32768, 65536])
def test_long_context(S, causal):
    run_and_check(1, S, 16, 128, causal, case=5, rows=sample_rows(S, n_random=8))


def test_uniform_value_rows_and_zero_queries():
    B, S, H, D = 1, 700, 2, 128
    dev = torch.device("cuda")
    q, k, v = inputs(B, S, H, D, case=6)
    u = v[:, :1].expand(B, S, H, D).contiguous()
    o, _ = ops.attn_fwd(q.to(dev), k.to(dev), u.to(dev), causal=True)
    ops.check()
    np.testing.assert_allclose(to64(o), np.broadcast_to(to64(u[:, :1]), (B, S, H, D)), atol=1e-2)
    z = torch.zeros_like(q)
    o, lse = ops.attn_fwd(z.to(dev), k.to(dev), v.to(dev), causal=True)
    ops.check()
    cum = np.cumsum(to64(v), axis=1) / np.arange(1, S + 1)[None, :, None, None]
    np.testing.assert_allclose(to64(o), cum, atol=1e-2)
    np.testing.assert_allclose(to64(lse), np.broadcast_to(np.log(np.arange(1, S + 1)), (B, H, S)), atol=1e-3)


def test_large_logits_exercise_rescaling():
    # Scores spread over many binades force the running max to be raised repeatedly.
    B, S, H, D = 1, 1024, 2, 64
    q, k, v = inputs(B, S, H, D, case=7)
    ramp = torch.linspace(0.2, 6.0, S).to(torch.bfloat16).view(1, S, 1, 1)
    k = (k * ramp).to(torch.bfloat16)
    dev = torch.device("cuda")
    o, lse = ops.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=True, scale=0.5)
    ops.check()
    O_ref, lse_ref = oracle_attention.attention(to64(q), to64(k), to64(v), scale=0.5, causal=True)
    max_abs, rms, _ = bf16_stats(to64(o), O_ref)
    assert max_abs <= BF16_MAX_ABS and rms <= BF16_RMS
    assert np.abs(to64(lse) - lse_ref).max() <= 1e-3 * max(1.0, np.abs(lse_ref).max() / 16)


def test_deterministic_replay():
    B, S, H, D = 2, 1000, 4, 128
    q, k, v = (t.cuda() for t in inputs(B, S, H, D, case=8))
    o1, l1 = ops.attn_fwd(q, k, v, causal=True)
    o2, l2 = ops.attn_fwd(q, k, v, causal=True)
    ops.check()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_lse_optional_and_explicit_scale():
    B, S, H, D = 1, 384, 2, 128
    q, k, v = inputs(B, S, H, D, case=9)
    dev = torch.device("cuda")
    o, lse = ops.attn_fwd(q.to(dev), k.to(dev), v.to(dev), scale=0.05, want_lse=False)
    ops.check()
    assert lse is None
    O_ref, _ = oracle_attention.attention(to64(q), to64(k), to64(v), scale=0.05)
    assert bf16_stats(to64(o), O_ref)[0] <= BF16_MAX_ABS
