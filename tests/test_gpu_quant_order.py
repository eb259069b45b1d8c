"""Stream order across consecutive quantiser launches (GPU).

A quantiser launch may start while the grid before it on the stream is finishing (programmatic
dependent launch), but it reads no input before that grid has completed.  So a launch whose
input bytes are the output of the quantiser launch just before it must see that output.  Here
the E4M3 codes of the second batch of a B = 2, D = 128 tensor, read back as a bf16 tensor of
D = 64, are quantised again (without rotation: the reinterpreted values are only scaled, and no
code byte makes a bf16 infinity or NaN, since a code's magnitude byte is at most 0x7E) directly
after the launch that writes them, with new contents every iteration.  The blocks the second
launch's CTAs read first include the last ones the first launch writes (its CTAs take every
152nd block, and the second batch holds the first launch's last round).  Each result must be
bitwise the second quantisation of the same codes run after a synchronisation.  The window in
which an early read could see the previous iteration's codes is short (about one block's time),
so a pass states the guarantee rather than proving that no ordering could break it.
"""

import pytest
import torch

from exact_attention_46_gb300 import ops
from tests.helpers import inputs
from tests.test_gpu_fp8 import signs_for

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("qkv", [False, True])
def test_launch_reads_the_output_of_the_launch_before(qkv):
    B, S, H, D = 2, 4096, 8, 128
    xs = [inputs(B, S, H, D, case=60 + i, dist="outliers")[0].cuda() for i in range(4)]
    s = torch.from_numpy(signs_for(60, D)).cuda()
    nb = S // 128
    c8 = torch.empty((B, S, H, D), dtype=torch.uint8, device="cuda")
    sc = torch.empty((B, H, nb), dtype=torch.float32, device="cuda")
    e8 = [torch.empty((1, S, H, D // 2), dtype=torch.uint8, device="cuda") for _ in range(3)]
    se = [torch.empty((1, H, nb), dtype=torch.float32, device="cuda") for _ in range(3)]
    kept = []
    for it in range(24):
        ops.hadamard_rotate_quant_fp8(xs[it % 4], s, out=c8, scale=sc)
        y = c8[1:].view(torch.bfloat16)                    # [1, S, H, 64] bf16 over batch 1's codes
        if qkv:
            ops.hadamard_rotate_quant_fp8_qkv(y, y, y, None, out=tuple(e8), scale=tuple(se))
        else:
            ops.hadamard_rotate_quant_fp8(y, None, out=e8[0], scale=se[0])
        kept.append((c8.clone(), e8[0].clone(), se[0].clone()))
    ops.check()
    torch.cuda.synchronize()
    for it, (codes, got, got_scale) in enumerate(kept):
        c_ref, _ = ops.hadamard_rotate_quant_fp8(xs[it % 4], s)
        ops.check()
        assert torch.equal(codes, c_ref), f"iteration {it}: first launch"
        e_ref, s_ref = ops.hadamard_rotate_quant_fp8(codes[1:].view(torch.bfloat16), None)
        ops.check()
        assert torch.equal(got, e_ref) and torch.equal(got_scale, s_ref), f"iteration {it}: second launch"
