"""Key-split tail of the non-causal forward vs the fp64 oracle, through the C ABI (GPU).

When the query blocks do not fill the last round of persistent CTAs, the blocks of that round
may be cut into key ranges whose partial (O, lse) a second kernel merges.  The shapes here have
more blocks than SMs and a short last round, so the plan (checked first) splits them, into 2,
3 or 4 ranges.  Checks:
  - full rows against the oracle with the BF16 forward bounds (FP8: the RMS criterion of the
    FP8 tests), over ragged S and D = 64, 128, 256;
  - rows of blocks that run whole are bitwise equal with and without the split; rows of cut
    blocks differ by at most twice the kernel's own error bounds (each key range rounds its
    softmax numerators to bf16 against its own running max, an independent rounding draw),
    and lse, formed from the unrounded numerators, within 1e-5;
  - grouped-query attention with repeated K/V heads is bitwise multi-head attention, split the
    same way; runs are bitwise repeatable; the launch without lse gives the same O.
"""

import numpy as np
import pytest
import torch

from exact_attention_46_gb300 import ops
from oracle import attention as oracle_attention
from oracle import fp8_path, quantise
from tests.helpers import BF16_MAX_ABS, BF16_RMS, LSE_MAX_ABS, bf16_stats, half_ulp_bf16, inputs, stats, to64
from tests.test_gpu_fp8 import signs_for

pytestmark = pytest.mark.gpu


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def plan(B, S, H, D, max_parts=4):
    nt = 1 if D == 256 else 2
    n_items = B * H * (-(-S // (128 * nt)))
    return ops.key_split_plan(n_items, sms(), -(-S // 128), max_parts)


def cut_rows(B, S, H, D, p):
    """Boolean [B, S, H]: rows of the query blocks that were cut."""
    nt = 1 if D == 256 else 2
    nqb = -(-S // (128 * nt))
    mask = np.zeros((B, S, H), dtype=bool)
    n_whole, n_tail, _ = p
    for item in range(n_whole, n_whole + n_tail):
        hb, qb = divmod(item, nqb)
        b, h = divmod(hb, H)
        mask[b, 128 * nt * qb: 128 * nt * (qb + 1), h] = True
    return mask


def with_split(max_parts, fn):
    ops.set_key_split(max_parts)
    try:
        return fn()
    finally:
        ops.set_key_split(4)


@pytest.mark.parametrize("B,S,H,D,parts", [(2, 2000, 11, 128, 4), (2, 2048, 11, 64, 4), (2, 2048, 11, 256, 3),
                                           (2, 1920, 11, 128, 3), (2, 2432, 11, 128, 2)])
def test_split_matches_oracle_and_unsplit(B, S, H, D, parts):
    p = plan(B, S, H, D)
    assert p[2] == parts and p[1] > 0, p
    q, k, v = inputs(B, S, H, D, case=80)
    dev = torch.device("cuda")
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    o, lse = ops.attn_fwd(qd, kd, vd)
    o1, lse1 = with_split(1, lambda: ops.attn_fwd(qd, kd, vd))
    ops.check()
    O_ref, lse_ref = oracle_attention.attention(to64(q), to64(k), to64(v))
    o64 = to64(o)
    max_abs, rms, _ = bf16_stats(o64, O_ref)
    lse_err = float(np.abs(to64(lse) - lse_ref).max())
    assert np.isfinite(o64).all()
    assert max_abs <= BF16_MAX_ABS and rms <= BF16_RMS and lse_err <= LSE_MAX_ABS, (max_abs, rms, lse_err)
    cut = cut_rows(B, S, H, D, p)
    a, b = o.cpu(), o1.cpu()
    assert torch.equal(a[torch.from_numpy(~cut)], b[torch.from_numpy(~cut)])
    # a key range rounds its numerators to bf16 against its own running max, so cut rows differ
    # from the unsplit ones by two independent draws of the kernel's rounding error
    d = np.abs(to64(a) - to64(b))[cut]
    excess = d - 2 * half_ulp_bf16(np.maximum(np.abs(to64(a)), np.abs(to64(b)))[cut])
    assert excess.max() <= 2 * BF16_MAX_ABS and np.sqrt(np.mean(d ** 2)) <= 2 * BF16_RMS
    # the row sums take the unrounded numerators: lse differs by fp32 arithmetic alone
    assert float(np.abs(to64(lse) - to64(lse1)).max()) <= 1e-5


def test_split_fp8_matches_oracle():
    B, S, H, D = 2, 2048, 11, 128
    assert plan(B, S, H, D)[2] == 4
    q, k, v = inputs(B, S, H, D, case=81, dist="outliers")
    s = signs_for(81, D)
    dev = torch.device("cuda")
    sd = torch.from_numpy(s).to(dev)
    q8, sq = ops.hadamard_rotate_quant_fp8(q.to(dev), sd)
    k8, sk = ops.hadamard_rotate_quant_fp8(k.to(dev), sd)
    v8, sv = ops.hadamard_rotate_quant_fp8(v.to(dev), None)
    o, lse = ops.attn_fwd_fp8(q8, k8, v8, sq, sk, sv)
    o1, _ = with_split(1, lambda: ops.attn_fwd_fp8(q8, k8, v8, sq, sk, sv))
    ops.check()
    O_emul, _, (Qq, Kq, Vq) = fp8_path.fp8_attention(to64(q), to64(k), to64(v), s.astype(np.float64), fold_v=True)
    qd, kd, vd = (quantise.dequantise(X["q"], X["scale"]) for X in (Qq, Kq, Vq))
    O_deq, lse_deq = oracle_attention.attention(qd, kd, vd)
    _, e_gpu = stats(to64(o), O_deq)
    _, e_emul = stats(O_emul, O_deq)
    assert np.isfinite(to64(o)).all()
    assert e_gpu <= 2 * e_emul + 1e-4, (e_gpu, e_emul)
    assert np.abs(to64(lse) - lse_deq).max() <= 1e-3
    keep = torch.from_numpy(~cut_rows(B, S, H, D, plan(B, S, H, D)))
    assert torch.equal(o.cpu()[keep], o1.cpu()[keep])


def test_split_grouped_query_is_repeated_multi_head():
    B, S, Hq, Hkv, D = 2, 2048, 12, 4, 128
    assert plan(B, S, Hq, D)[2] == 3
    q, k, v = inputs(B, S, Hq, D, case=82)
    dev = torch.device("cuda")
    qd = q.to(dev)
    kd, vd = k[:, :, :Hkv].contiguous().to(dev), v[:, :, :Hkv].contiguous().to(dev)
    a, la = ops.attn_fwd_gqa(qd, kd, vd)
    rep = Hq // Hkv
    b, lb = ops.attn_fwd(qd, kd.repeat_interleave(rep, dim=2).contiguous(), vd.repeat_interleave(rep, dim=2).contiguous())
    ops.check()
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_split_repeatable_and_without_lse():
    B, S, H, D = 2, 2048, 11, 128
    assert plan(B, S, H, D)[2] == 4
    q, k, v = (t.cuda() for t in inputs(B, S, H, D, case=83))
    o1, l1 = ops.attn_fwd(q, k, v)
    o2, l2 = ops.attn_fwd(q, k, v)
    o3, l3 = ops.attn_fwd(q, k, v, want_lse=False)
    ops.check()
    assert l3 is None
    assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(o1, o3)


def test_split_fp8_grouped_query_is_repeated_multi_head():
    # E4M3 codes and block scales of repeated K/V heads are repeated too, so the grouped launch
    # and the multi-head launch on the repeated codes do the same arithmetic, split the same way
    B, S, Hq, Hkv, D = 2, 2048, 12, 4, 128
    assert plan(B, S, Hq, D)[2] == 3
    q, k, v = inputs(B, S, Hq, D, case=84)
    s = signs_for(84, D)
    dev = torch.device("cuda")
    sd = torch.from_numpy(s).to(dev)
    q8, sq = ops.hadamard_rotate_quant_fp8(q.to(dev), sd)
    k8, sk = ops.hadamard_rotate_quant_fp8(k[:, :, :Hkv].contiguous().to(dev), sd)
    v8, sv = ops.hadamard_rotate_quant_fp8(v[:, :, :Hkv].contiguous().to(dev), None)
    a, la = ops.attn_fwd_gqa_fp8(q8, k8, v8, sq, sk, sv)
    rep = Hq // Hkv
    rk8, rv8 = (t.repeat_interleave(rep, dim=2).contiguous() for t in (k8, v8))
    rsk, rsv = (t.repeat_interleave(rep, dim=1).contiguous() for t in (sk, sv))
    b, lb = ops.attn_fwd_fp8(q8, rk8, rv8, sq, rsk, rsv)
    ops.check()
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_split_unit_scale_fp8_is_attn_fwd_fp8_with_unit_scales():
    # attn_fwd on E4M3 codes (scales taken as 1) against attn_fwd_fp8 with all-one scale arrays
    B, S, H, D = 2, 2048, 11, 128
    assert plan(B, S, H, D)[2] == 4
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(85)
    codes = [(torch.randint(0, 0x41, (B, S, H, D), generator=g, dtype=torch.int32)
              | (torch.randint(0, 2, (B, S, H, D), generator=g, dtype=torch.int32) << 7)).to(torch.uint8).to(dev)
             for _ in range(3)]
    ones = torch.ones((B, H, -(-S // 128)), dtype=torch.float32, device=dev)
    a, la = ops.attn_fwd(*codes)
    b, lb = ops.attn_fwd_fp8(*codes, ones, ones, ones)
    ops.check()
    assert torch.isfinite(a.float()).all()
    assert torch.equal(a, b) and torch.equal(la, lb)
