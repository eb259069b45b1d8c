"""Many back-to-back forward launches on one stream (GPU): every bounded wait completes and every
launch returns the same bits.

The forward's roles hand tiles to each other through mbarriers whose waits test a phase parity,
so a barrier that ran two phases ahead of its waiter would make that wait time out
(ATTN_ERR_TIMEOUT) only under some interleavings of the roles.  Hundreds of launches of shapes
with many short items (S = 512, causal S = 1024) and with long ones exercise those interleavings;
the outputs must be bitwise those of the first launch, since the kernels' results do not depend
on timing.
"""

import pytest
import torch

from exact_attention_46_gb300 import ops, synth

pytestmark = pytest.mark.gpu

SHAPES = [(32, 512, 16, 128, False), (16, 1024, 16, 128, True), (2, 8192, 32, 64, True), (4, 2048, 16, 64, False)]


def _inputs(B, S, H, D, case):
    return [t.cuda() for t in synth.make_qkv(B, S, H, D, case)]


@pytest.mark.parametrize("B,S,H,D,causal", SHAPES)
def test_fp8_forward_repeated(B, S, H, D, causal):
    q, k, v = _inputs(B, S, H, D, case=401)
    s = torch.from_numpy(synth.signs(D, 17)).cuda()
    q8, sq = ops.hadamard_rotate_quant_fp8(q, s)
    k8, sk = ops.hadamard_rotate_quant_fp8(k, s)
    v8, sv = ops.hadamard_rotate_quant_fp8(v, None)
    o0, l0 = ops.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, causal=causal)
    ops.check()
    for _ in range(300):
        o, lse = ops.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, causal=causal)
    ops.check()
    assert torch.equal(o, o0) and torch.equal(lse, l0)


@pytest.mark.parametrize("B,S,H,D,causal", SHAPES)
def test_bf16_forward_repeated(B, S, H, D, causal):
    q, k, v = _inputs(B, S, H, D, case=402)
    o0, l0 = ops.attn_fwd(q, k, v, causal=causal)
    ops.check()
    for _ in range(300):
        o, lse = ops.attn_fwd(q, k, v, causal=causal)
    ops.check()
    assert torch.equal(o, o0) and torch.equal(lse, l0)
