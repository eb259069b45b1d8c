"""BF16 attention over packed variable-length batches vs the fp64 oracle, through the C ABI (GPU).

Same bounds as the fixed-length BF16 tests (max error beyond half a bf16 ulp <= 1e-2,
RMS <= 2e-3, lse <= 1e-3).  Length mixes cover empty sequences, single tokens, every
remainder modulo the 128-row tile and the 256-row CTA block, sequences shorter and longer
than a block, more work items than SMs, 4096 sequences (the limit) and a 32K-token
sequence.  Equal lengths must give attn_fwd's output bit for bit: masked keys contribute
exact zeros whether the tile ran into the next sequence or past the tensor.  Offsets that
break the rules, or a sequence longer than max_seqlen, are rejected by the kernel without
writing anything.
"""

import numpy as np
import pytest
import torch

from exact_attention_46_gb300 import _lib, ops, synth
from oracle import varlen as oracle_varlen
from tests.helpers import BF16_MAX_ABS, BF16_RMS, LSE_MAX_ABS, bf16_stats, to64

pytestmark = pytest.mark.gpu


def packed(total, H, D, case):
    q, k, v = synth.make_qkv(1, total, H, D, case)
    return q[0], k[0], v[0]


def run_and_check(cu, H, D, causal, case, rows=None):
    cu = np.asarray(cu, dtype=np.int32)
    q, k, v = packed(int(cu[-1]), H, D, case)
    dev = torch.device("cuda")
    max_len = max(1, int(np.diff(cu).max()))
    o, lse = ops.attn_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), torch.from_numpy(cu).to(dev), max_len,
                                 causal=causal)
    ops.check()
    O_ref, lse_ref = oracle_varlen.attention_varlen(to64(q), to64(k), to64(v), cu, causal=causal, rows=rows)
    o64, lse64 = to64(o), to64(lse)
    if rows is not None:
        o64, lse64 = o64[rows], lse64[:, rows]
    max_abs, rms, _ = bf16_stats(o64, O_ref)
    lse_err = float(np.abs(lse64 - lse_ref).max())
    assert np.isfinite(o64).all() and np.isfinite(lse64).all()
    assert max_abs <= BF16_MAX_ABS and rms <= BF16_RMS and lse_err <= LSE_MAX_ABS, (max_abs, rms, lse_err)


MIXES = {
    "edges": [0, 5, 5, 133, 134, 390, 391, 600],                        # 5, 0, 128, 1, 256, 1, 209
    "tiles": np.concatenate([[0], np.cumsum([127, 128, 129, 255, 256, 257, 511, 512, 513, 1])]),
    "empty_ends": [0, 0, 0, 300, 300, 300],
}


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mix", sorted(MIXES))
def test_full_rows_length_mixes(mix, D, causal):
    run_and_check(MIXES[mix], 2, D, causal, case=40)


@pytest.mark.parametrize("causal", [False, True])
def test_more_items_than_sms(causal):
    _, cu = synth.seqlens(6000, 1, 700, synth.seed_for(41, synth.STREAM_LENGTHS))
    run_and_check(cu, 12, 128, causal, case=41)


def test_4096_sequences():
    lens = (synth.uniform((4096,), synth.seed_for(42, synth.STREAM_LENGTHS)) * 12).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    run_and_check(cu, 2, 64, True, case=42)


@pytest.mark.parametrize("causal", [False, True])
def test_long_sequence_in_a_mix(causal):
    cu = [0, 1000, 1000 + 32768, 1000 + 32768 + 77]
    rows = np.array(sorted({0, 999, 1000, 1001, 1127, 1128, 1255, 1256, 17000, 33766, 33767, 33768, 33844}), dtype=np.int64)
    run_and_check(cu, 4, 128, causal, case=43, rows=rows)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_equal_lengths_match_attn_fwd_bitwise(D, causal):
    B, S, H = 3, 1000, 4
    q, k, v = synth.make_qkv(B, S, H, D, case=44)
    dev = torch.device("cuda")
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    o_ref, lse_ref = ops.attn_fwd(qd, kd, vd, causal=causal)
    cu = torch.arange(0, (B + 1) * S, S, dtype=torch.int32, device=dev)
    o, lse = ops.attn_fwd_varlen(qd.reshape(B * S, H, D), kd.reshape(B * S, H, D), vd.reshape(B * S, H, D), cu,
                                 S, causal=causal)
    ops.check()
    assert torch.equal(o.reshape(B, S, H, D), o_ref)
    assert torch.equal(lse.reshape(H, B, S).permute(1, 0, 2), lse_ref)


def test_bad_offsets_are_rejected_on_the_device_and_nothing_is_written():
    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in packed(300, 2, 128, case=45))
    for cu, max_len in (([0, 200, 100, 300], 200), ([1, 150, 300], 150), ([0, 150, 299], 150),
                        ([0, 150, 301], 151), ([0, 100, 300], 150)):
        o = torch.full_like(q, 7.0)
        lse = torch.full((2, 300), 7.0, device=dev)
        ops.attn_fwd_varlen(q, k, v, torch.tensor(cu, dtype=torch.int32, device=dev), max_len, out=o, lse=lse)
        with pytest.raises(_lib.AttnError) as e:
            ops.check()
        assert e.value.status == 1
        assert bool((o == 7.0).all()) and bool((lse == 7.0).all())
    # the context stays usable
    o, _ = ops.attn_fwd_varlen(q, k, v, torch.tensor([0, 150, 300], dtype=torch.int32, device=dev), 150)
    ops.check()
    assert torch.isfinite(o.float()).all()


def test_max_seqlen_at_the_level_limit():
    # one sequence of exactly 1024 levels (262144 tokens at D = 128): the top level is used
    dev = torch.device("cuda")
    total = 262144 + 300
    cu = np.array([0, 300, total], dtype=np.int32)
    rows = np.array([0, 299, 300, 301, 555, 131372, total - 2, total - 1], dtype=np.int64)
    q, k, v = packed(total, 1, 128, case=47)
    o, lse = ops.attn_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), torch.from_numpy(cu).to(dev), 262144, causal=True)
    ops.check()
    O_ref, lse_ref = oracle_varlen.attention_varlen(to64(q), to64(k), to64(v), cu, causal=True, rows=rows)
    max_abs, rms, _ = bf16_stats(to64(o)[rows], O_ref)
    assert max_abs <= BF16_MAX_ABS and rms <= BF16_RMS
    assert float(np.abs(to64(lse)[:, rows] - lse_ref).max()) <= LSE_MAX_ABS


def test_without_lse():
    dev = torch.device("cuda")
    cu = np.array([0, 130, 300], dtype=np.int32)
    q, k, v = (t.to(dev) for t in packed(300, 2, 128, case=46))
    o, lse = ops.attn_fwd_varlen(q, k, v, torch.from_numpy(cu).to(dev), want_lse=False)
    ops.check()
    assert lse is None
    o_ref, _ = ops.attn_fwd_varlen(q, k, v, torch.from_numpy(cu).to(dev))
    ops.check()
    assert torch.equal(o, o_ref)
