"""Boundary behaviour on the GPU: bad arguments launch nothing, the bounded-wait timeout
path reports ATTN_ERR_TIMEOUT without hanging or faulting, and the context stays usable."""

import numpy as np
import pytest
import torch

from exact_attention_46_gb300 import _lib, ops
from oracle import attention as oracle_attention
from tests.helpers import inputs, stats, to64

pytestmark = pytest.mark.gpu


def test_bounded_wait_timeout_is_reported_and_context_survives():
    ops.check()                                    # clean state
    ops.selftest_bounded_wait(2_000_000)           # ~1 ms of spinning, then gives up
    with pytest.raises(_lib.AttnError) as ei:
        ops.check()
    assert ei.value.status == 4
    ops.check()                                    # the error word was cleared
    q, k, v = inputs(1, 256, 2, 64, case=30)
    o, _ = ops.attn_fwd(q.cuda(), k.cuda(), v.cuda())
    ops.check()
    O_ref, _ = oracle_attention.attention(to64(q), to64(k), to64(v))
    assert stats(to64(o), O_ref)[0] <= 1e-2


def test_invalid_arguments_raise_and_launch_nothing():
    q = torch.zeros((1, 128, 1, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(_lib.AttnError) as ei:
        ops.attn_fwd(q, q.clone(), q.clone())
    assert ei.value.status == 2
    q = torch.zeros((1, 128, 1, 128), dtype=torch.bfloat16, device="cuda")
    o = torch.full_like(q, 7.0)
    with pytest.raises(_lib.AttnError):
        ops.attn_fwd(q, q.clone(), q.clone(), out=o, scale=-1.0)
    assert bool((o == 7.0).all())                  # untouched
    with pytest.raises(_lib.AttnError):
        ops.attn_fwd(q, q, q, out=q)               # output aliases input
    ops.check()


def test_binding_rejects_malformed_tensors_before_the_library():
    import torch
    from exact_attention_46_gb300 import ops
    dev = torch.device("cuda")
    q = torch.zeros((1, 256, 2, 128), dtype=torch.bfloat16, device=dev)
    codes = torch.zeros((1, 256, 2, 128), dtype=torch.uint8, device=dev)
    sc = torch.ones((1, 2, 2), dtype=torch.float32, device=dev)
    with pytest.raises(ValueError, match="shape"):
        ops.attn_fwd_fp8(codes, codes, codes, sc, sc, sc[:, :, :1].contiguous())     # one block short
    with pytest.raises(ValueError, match="dtype"):
        ops.attn_fwd_fp8(codes, codes, codes, sc, sc.double(), sc)
    with pytest.raises(ValueError, match="dtype"):
        ops.attn_fwd(q, codes, codes)                                             # mixed families
    with pytest.raises(ValueError, match="dtype"):
        ops.attn_fwd(q, q, q, out=torch.empty_like(q, dtype=torch.float32))
    with pytest.raises(ValueError, match="shape"):
        ops.attn_decode(q[:, :1].contiguous(), q, q[:, :128].contiguous())
    with pytest.raises(ValueError, match="shape"):
        ops.hadamard_rotate_quant_fp8(q, torch.ones(64, device=dev))               # signs of D values
