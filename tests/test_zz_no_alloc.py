"""attn_bwd_noalloc against attn_bwd, through the C ABI (GPU).

attn_bwd_noalloc is the backward pass for callers that cannot allocate device memory where they
run it (an engine that gave the GPU's memory to its own pool, a host that forbids allocation
inside per-step calls): it uses a fixed scratch array built into the library instead of a
caller workspace.  Two calls in a row, on different inputs, so that the second finds the
first's contents in the shared scratch; each must give what attn_bwd gives with a fresh
workspace.  Both run the same deterministic kernels, so the comparison is bit for bit, stricter
than the backward tests' rounding bound.  The file name sorts last, so a run that stops at the
first failure has run every other test before this one.
"""

import ctypes

import pytest
import torch

from exact_attention_46_gb300 import _lib, ops, synth

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("first,second", [((2, 700, 4, 128, False), (1, 1000, 3, 64, True))])
def test_two_calls_in_a_row_match_attn_bwd(first, second):
    lib = _lib.load()
    dev = torch.device("cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for case, (B, S, H, D, causal) in enumerate((first, second), start=60):
        q, k, v = (t.to(dev) for t in synth.make_qkv(B, S, H, D, case))
        do = torch.from_numpy(synth.normal((B, S, H, D), synth.seed_for(case, synth.STREAM_OUT_VAL))).to(torch.bfloat16).to(dev)
        o, lse = ops.attn_fwd(q, k, v, causal=causal)
        ref = ops.attn_bwd(q, k, v, o, lse, do, causal=causal)
        ops.check()
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        rc = lib.attn_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv),
                                  B, H, S, D, int(causal), 0.0, stream)
        assert rc == 0, lib.attn_get_last_error()
        ops.check()
        for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            assert torch.equal(got, want), name


def test_the_largest_problem_that_fits():
    # B * H * (S rounded up to 128) = 8 * 16 * 16384 = 2,097,152 rows: exactly the 16 MiB the
    # built-in scratch holds; the last padded rows land on its last bytes
    lib = _lib.load()
    B, S, H, D, causal = 8, 16384, 16, 64, False
    assert lib.attn_bwd_workspace_bytes(B, H, S) == 16 * 1024 * 1024
    dev = torch.device("cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    q, k, v = (t.to(dev) for t in synth.make_qkv(B, S, H, D, 62))
    do = torch.from_numpy(synth.normal((B, S, H, D), synth.seed_for(62, synth.STREAM_OUT_VAL))).to(torch.bfloat16).to(dev)
    o, lse = ops.attn_fwd(q, k, v, causal=causal)
    ref = ops.attn_bwd(q, k, v, o, lse, do, causal=causal)
    ops.check()
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    rc = lib.attn_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv),
                              B, H, S, D, int(causal), 0.0, stream)
    assert rc == 0, lib.attn_get_last_error()
    ops.check()
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert torch.equal(got, want), name
    # one more 128-row block does not fit, and is refused before anything runs
    assert lib.attn_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv),
                                B, H, S + 1, D, int(causal), 0.0, stream) == 1
