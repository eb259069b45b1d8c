"""The three-tensor quantiser (hadamard_rotate_quant_fp8_qkv) through the C ABI (GPU).

One launch quantises Q and K (rotated by the same random signs) and V (not rotated).  Each
output must be bitwise what hadamard_rotate_quant_fp8 writes for its tensor alone, since the
arithmetic is the same, over D = 64, 128, 256, ragged S, with and without signs; one case is also
compared with the oracle's codes and scales directly.
"""

import numpy as np
import pytest
import torch

from exact_attention_46_gb300 import ops
from oracle import quantise
from tests.helpers import inputs, to64
from tests.test_gpu_fp8 import SCALE_RTOL, check_codes, signs_for

pytestmark = pytest.mark.gpu


def _qkv(B, S, H, D, case):
    q, k, v = inputs(B, S, H, D, case=case, dist="outliers")
    return q.cuda(), k.cuda(), v.cuda()


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("rotate", [False, True])
@pytest.mark.parametrize("B,S,H", [(1, 1, 1), (2, 100, 3), (2, 300, 5), (1, 1024, 4), (3, 129, 2)])
def test_qkv_form_is_three_single_launches(B, S, H, D, rotate):
    q, k, v = _qkv(B, S, H, D, case=30)
    s = torch.from_numpy(signs_for(30, D)).cuda() if rotate else None
    q8, sq, k8, sk, v8, sv = ops.hadamard_rotate_quant_fp8_qkv(q, k, v, s)
    ops.check()
    for x, sg, c, sc in ((q, s, q8, sq), (k, s, k8, sk), (v, None, v8, sv)):
        c1, sc1 = ops.hadamard_rotate_quant_fp8(x, sg)
        ops.check()
        assert torch.equal(c, c1) and torch.equal(sc, sc1)


def test_qkv_form_matches_oracle_at_the_benchmark_width():
    B, S, H, D = 2, 1000, 16, 128
    q, k, v = _qkv(B, S, H, D, case=31)
    s = signs_for(31, D)
    q8, sq, k8, sk, v8, sv = ops.hadamard_rotate_quant_fp8_qkv(q, k, v, torch.from_numpy(s).cuda())
    ops.check()
    for x, sg, c, sc in ((q, s, q8, sq), (k, s, k8, sk), (v, None, v8, sv)):
        ref = quantise.quantise_blocks(to64(x.cpu()), None if sg is None else sg.astype(np.float64))
        np.testing.assert_allclose(sc.cpu().double().numpy(), ref["scale"], rtol=SCALE_RTOL, atol=0)
        check_codes(c.cpu().numpy(), ref)


def test_qkv_form_rejects_overlapping_outputs():
    B, S, H, D = 1, 256, 2, 64
    q, k, v = _qkv(B, S, H, D, case=32)
    codes = torch.empty((B, S, H, D), dtype=torch.uint8, device="cuda")
    scales = [torch.empty((B, H, 2), dtype=torch.float32, device="cuda") for _ in range(3)]
    from exact_attention_46_gb300 import _lib
    with pytest.raises(_lib.AttnError):
        _lib.call("hadamard_rotate_quant_fp8_qkv", q.data_ptr(), k.data_ptr(), v.data_ptr(), codes.data_ptr(),
                  codes.data_ptr(), codes.data_ptr(), *[t.data_ptr() for t in scales], None, B, H, S, D, None)
