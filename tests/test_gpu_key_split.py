"""Key-split tail of the non-causal forward (attn_fwd_split) vs the fp64 oracle, through the C ABI (GPU).

When the query blocks do not fill the last round of persistent CTAs, attn_fwd_split may cut the
blocks of that round into key ranges whose partial (O, lse) go to the caller's workspace and a
second kernel merges.  The shapes here have more blocks than SMs and a short last round, so the
plan (checked first) splits them, into 2, 3 or 4 ranges.  attn_fwd never splits.  Checks:
  - full rows against the oracle with the BF16 forward bounds (FP8: the element-wise bounds of
    the FP8 tests), over ragged S and D = 64, 128, 256;
  - rows of blocks that run whole are bitwise equal to attn_fwd's; rows of cut blocks differ by
    at most twice the kernel's own error bounds (each key range rounds its softmax numerators
    to bf16 against its own running max, an independent rounding draw), and lse, formed from
    the unrounded numerators, within 1e-5;
  - the same arguments and workspace give the same bits on every call, whatever the workspace
    held before; a workspace smaller than attn_fwd_split_workspace_bytes is an error and
    writes nothing; no workspace runs unsplit;
  - grouped-query attention with repeated K/V heads is bitwise multi-head attention, split the
    same way; runs are bitwise repeatable; the launch without lse gives the same O.
"""

import numpy as np
import pytest
import torch

from exact_attention_46_gb300 import _lib, ops
from oracle import attention as oracle_attention
from oracle import fp8_path, quantise
from tests import fp8_bound
from tests.helpers import BF16_MAX_ABS, BF16_RMS, LSE_MAX_ABS, bf16_stats, half_ulp_bf16, inputs, to64
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


def workspace_bytes(B, S, H, D, p):
    nt = 1 if D == 256 else 2
    return p[1] * p[2] * 128 * nt * (D + 1) * 4


@pytest.mark.parametrize("B,S,H,D,parts", [(2, 2000, 11, 128, 4), (2, 2048, 11, 64, 4), (2, 2048, 11, 256, 3),
                                           (2, 1920, 11, 128, 3), (2, 2432, 11, 128, 2)])
def test_split_matches_oracle_and_unsplit(B, S, H, D, parts):
    p = plan(B, S, H, D)
    assert p[2] == parts and p[1] > 0, p
    q, k, v = inputs(B, S, H, D, case=80)
    dev = torch.device("cuda")
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    assert ops.split_workspace_bytes(B, H, S, D) == workspace_bytes(B, S, H, D, p)
    o, lse = ops.attn_fwd_split(qd, kd, vd)
    o1, lse1 = ops.attn_fwd(qd, kd, vd)
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
    # the oracle's codes and scales (Q, K rotated), split into 4 key ranges; every element
    # within the FP8 bounds of tests/fp8_bound.py (each range folds V's block scales against its
    # own largest one, which only raises the ratios the bound divides by)
    B, S, H, D = 2, 2048, 11, 128
    assert plan(B, S, H, D)[2] == 4
    q, k, v = inputs(B, S, H, D, case=81, dist="outliers")
    s = signs_for(81, D).astype(np.float64)
    res = fp8_path.quantise_qkv(to64(q), to64(k), to64(v), s)
    sc32 = [r["scale"].astype(np.float32) for r in res]
    dev = torch.device("cuda")
    t = [torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in [r["codes"] for r in res] + sc32]
    o, lse = ops.attn_fwd_split(*t)
    o1, _ = ops.attn_fwd_fp8(*t)
    ops.check()
    qd, kd, vd = (quantise.dequantise(r["q"], sc.astype(np.float64)) for r, sc in zip(res, sc32))
    ref = fp8_bound.reference(qd, kd, vd, sc32[2], 1 / np.sqrt(D), False)
    fp8_bound.check(to64(o), to64(lse), ref)
    keep = torch.from_numpy(~cut_rows(B, S, H, D, plan(B, S, H, D)))
    assert torch.equal(o.cpu()[keep], o1.cpu()[keep])


def test_split_grouped_query_is_repeated_multi_head():
    B, S, Hq, Hkv, D = 2, 2048, 12, 4, 128
    assert plan(B, S, Hq, D)[2] == 3
    q, k, v = inputs(B, S, Hq, D, case=82)
    dev = torch.device("cuda")
    qd = q.to(dev)
    kd, vd = k[:, :, :Hkv].contiguous().to(dev), v[:, :, :Hkv].contiguous().to(dev)
    a, la = ops.attn_fwd_split(qd, kd, vd)
    rep = Hq // Hkv
    b, lb = ops.attn_fwd_split(qd, kd.repeat_interleave(rep, dim=2).contiguous(),
                               vd.repeat_interleave(rep, dim=2).contiguous())
    ops.check()
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_split_repeatable_and_without_lse():
    B, S, H, D = 2, 2048, 11, 128
    assert plan(B, S, H, D)[2] == 4
    q, k, v = (t.cuda() for t in inputs(B, S, H, D, case=83))
    o1, l1 = ops.attn_fwd_split(q, k, v)
    o2, l2 = ops.attn_fwd_split(q, k, v)
    o3, l3 = ops.attn_fwd_split(q, k, v, want_lse=False)
    ops.check()
    assert l3 is None
    assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(o1, o3)


@pytest.mark.parametrize("fp8", [False, True])
def test_same_arguments_and_workspace_give_the_same_bits_whatever_it_held(fp8):
    # the library allocates nothing: the split's scratch is the caller's workspace, so the result
    # is a function of the arguments alone -- not of the workspace's previous contents, nor of
    # what else the process has allocated
    B, S, H, D = 2, 2048, 11, 128
    p = plan(B, S, H, D)
    assert p[2] == 4
    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in inputs(B, S, H, D, case=86))
    if fp8:
        sd = torch.from_numpy(signs_for(86, D)).to(dev)
        (q, sq), (k, sk), (v, sv) = (ops.hadamard_rotate_quant_fp8(t, s) for t, s in ((q, sd), (k, sd), (v, None)))
        scales = (sq, sk, sv)
    else:
        scales = (None, None, None)
    need = ops.split_workspace_bytes(B, H, S, D)
    assert need == workspace_bytes(B, S, H, D, p) and need > 0
    outs = []
    for fill in (0x00, 0xFF, 0x7F, None):
        ws = torch.empty((need + 4096,), dtype=torch.uint8, device=dev)
        if fill is None:
            ws.copy_(torch.randint(0, 256, ws.shape, dtype=torch.uint8, device=dev))
        else:
            ws.fill_(fill)
        hog = torch.empty((int(64e6),), dtype=torch.uint8, device=dev)   # other allocations around it
        outs.append(ops.attn_fwd_split(q, k, v, *scales, workspace=ws[:need]))
        outs.append(ops.attn_fwd_split(q, k, v, *scales, workspace=ws[4096 - 16 * (fill or 1):][:need]))
        del hog
    ops.check()
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])
    # rows of whole blocks are the unsplit launch's, bit for bit
    o1, _ = (ops.attn_fwd_fp8(q, k, v, *scales) if fp8 else ops.attn_fwd(q, k, v))
    ops.check()
    keep = torch.from_numpy(~cut_rows(B, S, H, D, p))
    assert torch.equal(outs[0][0].cpu()[keep], o1.cpu()[keep])
    assert not torch.equal(outs[0][0], o1)            # and the cut rows did run split


def test_workspace_too_small_or_absent():
    B, S, H, D = 2, 2048, 11, 128
    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in inputs(B, S, H, D, case=87))
    need = ops.split_workspace_bytes(B, H, S, D)
    out = torch.full((B, S, H, D), 7.0, dtype=torch.bfloat16, device=dev)
    with pytest.raises(_lib.AttnError) as e:
        ops.attn_fwd_split(q, k, v, out=out, workspace=torch.empty((need - 16,), dtype=torch.uint8, device=dev))
    assert e.value.status == 1
    ops.check()
    assert bool((out == 7.0).all())
    # an empty workspace runs every block whole: attn_fwd's result
    a, la = ops.attn_fwd_split(q, k, v, workspace=torch.empty((0,), dtype=torch.uint8, device=dev))
    b, lb = ops.attn_fwd(q, k, v)
    ops.check()
    assert torch.equal(a, b) and torch.equal(la, lb)
    # shapes the plan does not split need no workspace
    assert ops.split_workspace_bytes(B, H, S, D, causal=True) == 0
    assert ops.split_workspace_bytes(1, 16, 8192, 128) == 0 or plan(1, 8192, 16, 128)[2] > 1


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
    a, la = ops.attn_fwd_split(q8, k8, v8, sq, sk, sv)
    rep = Hq // Hkv
    rk8, rv8 = (t.repeat_interleave(rep, dim=2).contiguous() for t in (k8, v8))
    rsk, rsv = (t.repeat_interleave(rep, dim=1).contiguous() for t in (sk, sv))
    b, lb = ops.attn_fwd_split(q8, rk8, rv8, sq, rsk, rsv)
    ops.check()
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_split_unit_scale_fp8_is_attn_fwd_fp8_with_unit_scales():
    # E4M3 codes without scales (taken as 1) against the same codes with all-one scale arrays
    B, S, H, D = 2, 2048, 11, 128
    assert plan(B, S, H, D)[2] == 4
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(85)
    codes = [(torch.randint(0, 0x41, (B, S, H, D), generator=g, dtype=torch.int32)
              | (torch.randint(0, 2, (B, S, H, D), generator=g, dtype=torch.int32) << 7)).to(torch.uint8).to(dev)
             for _ in range(3)]
    ones = torch.ones((B, H, -(-S // 128)), dtype=torch.float32, device=dev)
    a, la = ops.attn_fwd_split(*codes)
    b, lb = ops.attn_fwd_split(*codes, ones, ones, ones)
    ops.check()
    assert torch.isfinite(a.float()).all()
    assert torch.equal(a, b) and torch.equal(la, lb)
