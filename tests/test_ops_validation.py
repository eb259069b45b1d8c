"""The Python binding rejects malformed tensors before it calls the library (CPU only: the
checks on the first argument -- type, dtype, rank, then device -- come before any CUDA use)."""

import pytest
import torch

from exact_attention_46_gb300 import ops


def test_first_argument_checks():
    x32 = torch.zeros((1, 4, 1, 64), dtype=torch.float32)
    with pytest.raises(ValueError, match="dtype"):
        ops.attn_fwd(x32, x32, x32)
    bf = torch.zeros((1, 4, 1, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="dtype"):
        ops.attn_fwd_fp8(bf, bf, bf, None, None, None)               # codes must be 1-byte
    with pytest.raises(ValueError, match="dimensions"):
        ops.attn_fwd(bf[0], bf[0], bf[0])
    with pytest.raises(ValueError, match="dimensions"):
        ops.attn_fwd_varlen(bf, bf, bf, torch.zeros(2, dtype=torch.int32))
    with pytest.raises(TypeError):
        ops.hadamard_rotate_quant_fp8([1, 2, 3])
    with pytest.raises(ValueError, match="contiguous"):
        ops.attn_fwd(bf.transpose(1, 3), bf, bf)
    with pytest.raises(ValueError, match="CUDA"):
        ops.attn_fwd(bf, bf, bf)
    with pytest.raises(ValueError, match="dtype"):
        ops.attn_bwd_gqa(x32, bf, bf, bf, None, bf)                   # q must be bf16
