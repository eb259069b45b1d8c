"""Grouped-query attention (prefill) and decoding vs the fp64 oracle, through the C ABI (GPU).

Same bounds as the BF16 forward tests (max error beyond half a bf16 ulp <= 1e-2, RMS <= 2e-3,
lse <= 1e-3).  Decoding shapes cover one and several query tokens, group sizes 1 .. 32
(G * Sq up to the 128-row tile; the kernel keeps 4, 2 or 1 copies of the packed rows for
G * Sq <= 32, <= 64 and above, and 33 and 64 rows sit on those edges), key counts below, at and
above a tile, ragged tails, and enough keys for many key splits (the partial results then go
through the merge kernel).
"""

import numpy as np
import pytest
import torch

from exact_attention_46_gb300 import ops, synth
from oracle import gqa as oracle_gqa
from tests.helpers import BF16_MAX_ABS, BF16_RMS, LSE_MAX_ABS, bf16_stats, to64

pytestmark = pytest.mark.gpu


def qkv(B, Sq, Sk, Hq, Hkv, D, case):
    q = torch.from_numpy(synth.normal((B, Sq, Hq, D), synth.seed_for(case, synth.STREAM_Q))).to(torch.bfloat16)
    k = torch.from_numpy(synth.normal((B, Sk, Hkv, D), synth.seed_for(case, synth.STREAM_K))).to(torch.bfloat16)
    v = torch.from_numpy(synth.normal((B, Sk, Hkv, D), synth.seed_for(case, synth.STREAM_V))).to(torch.bfloat16)
    return q, k, v


def check(o, lse, q, k, v, causal):
    O_ref, lse_ref = oracle_gqa.attention_gqa(to64(q), to64(k), to64(v), causal=causal)
    max_abs, rms, _ = bf16_stats(to64(o), O_ref)
    lse_err = float(np.abs(to64(lse) - lse_ref).max())
    assert np.isfinite(to64(o)).all()
    assert max_abs <= BF16_MAX_ABS and rms <= BF16_RMS and lse_err <= LSE_MAX_ABS, (max_abs, rms, lse_err)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S,Hkv", [(100, 1), (300, 2), (513, 8)])
def test_gqa_prefill(S, Hkv, D, causal):
    q, k, v = qkv(2, S, S, 8, Hkv, D, case=70)
    dev = torch.device("cuda")
    o, lse = ops.attn_fwd_gqa(q.to(dev), k.to(dev), v.to(dev), causal=causal)
    ops.check()
    check(o, lse, q, k, v, causal)


def test_gqa_with_one_group_per_head_is_attn_fwd():
    q, k, v = (t.cuda() for t in synth.make_qkv(2, 700, 4, 128, case=71))
    a, la = ops.attn_fwd_gqa(q, k, v, causal=True)
    b, lb = ops.attn_fwd(q, k, v, causal=True)
    ops.check()
    assert torch.equal(a, b) and torch.equal(la, lb)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Sq,Sk,Hq,Hkv", [
    (1, 1, 1, 8, 8), (2, 1, 100, 8, 2), (2, 1, 129, 32, 8), (1, 4, 1000, 16, 2), (3, 16, 300, 8, 1),
    (2, 8, 4097, 16, 1), (1, 1, 65536, 4, 1), (4, 2, 20000, 32, 4), (1, 128, 2000, 1, 1),
    (2, 6, 3000, 8, 1), (1, 2, 700, 32, 1), (1, 33, 500, 1, 1),
    (1, 17, 900, 1, 1), (2, 1, 3000, 16, 1)])
def test_decode(B, Sq, Sk, Hq, Hkv, D, causal):
    q, k, v = qkv(B, Sq, Sk, Hq, Hkv, D, case=72)
    dev = torch.device("cuda")
    o, lse = ops.attn_decode(q.to(dev), k.to(dev), v.to(dev), causal=causal)
    ops.check()
    check(o, lse, q, k, v, causal)


def test_decode_without_lse_and_repeatable():
    q, k, v = (t.cuda() for t in qkv(2, 3, 5000, 16, 4, 128, case=73))
    a, la = ops.attn_decode(q, k, v, causal=True)
    b, lb = ops.attn_decode(q, k, v, causal=True, want_lse=False)
    ops.check()
    assert lb is None and torch.equal(a, b)
