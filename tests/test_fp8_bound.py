"""Pins for the FP8 attention error bounds of tests/fp8_bound.py (CPU only).

The bounds must hold for every rounding of the softmax numerators that the FP8 attention step
allows -- the oracle's plain reading (numerators relative to the exact row max, no V fold) and
the reading the library's kernels take (numerators relative to a running reference up to
2^8 below the max, V's block ratio folded in) -- and must reject plausible mistakes: a wrong V
block scale, a dropped key, a wrong output scale, a wrong lse.
"""

import numpy as np
import pytest
import torch

from exact_attention_46_gb300 import synth
from oracle import e4m3, fp8_path, quantise
from tests import fp8_bound

RNG = np.random.default_rng(5)


def _inputs(B, S, H, D, case, gains=False):
    q, k, v = (t.to(torch.float64).numpy() for t in synth.make_qkv(B, S, H, D, case, "outliers"))
    if gains:                                     # block scales that differ by up to 2^6
        g = np.exp2((np.arange(S) // 128) % 7 - 3.0)[None, :, None, None]
        v = v * g
    return q, k, v


def _quantised(q, k, v, signs):
    Qq, Kq, Vq = fp8_path.quantise_qkv(q, k, v, signs)
    deq = [quantise.dequantise(r["q"], r["scale"]) for r in (Qq, Kq, Vq)]
    return deq, Vq["scale"], (Qq, Kq, Vq)


def _bf16(x):
    return torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()


def _lazy_fold_emulation(qd, kd, vd, v_scale, scale, causal, seed):
    """Numerators p * 2^delta * r_j rounded to E4M3, delta drawn in [0, 8] per (row, 128-key
    tile), r_j the V block ratio; O = sum_j E4M3(p') / (2^delta r_j) v_j / l."""
    rng = np.random.default_rng(seed)
    B, S, H, D = qd.shape
    O = np.empty_like(qd)
    r_blk = fp8_bound.v_ratio(v_scale)
    vis = np.tril(np.ones((S, S), dtype=bool)) if causal else np.ones((S, S), dtype=bool)
    for b in range(B):
        for h in range(H):
            s = np.where(vis, scale * qd[b, :, h] @ kd[b, :, h].T, -np.inf)
            m = s.max(axis=1, keepdims=True)
            p = np.exp(s - m)
            l = p.sum(axis=1, keepdims=True)
            delta = rng.uniform(0, 8, size=(S, (S + 127) // 128))[:, np.arange(S) // 128]
            r = r_blk[b, h][np.arange(S) // 128][None, :]
            fac = np.exp2(delta) * r
            pt = e4m3.round_e4m3(p * fac) / fac
            O[b, :, h] = (pt @ vd[b, :, h]) / l
    return O


@pytest.mark.parametrize("rotate", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_oracle_reading_lies_within_the_bounds(rotate, causal):
    B, S, H, D = 1, 600, 2, 64
    q, k, v = _inputs(B, S, H, D, case=301)
    s = synth.signs(D, 11).astype(np.float64) if rotate else None
    (qd, kd, vd), sv, _ = _quantised(q, k, v, s)
    O_emul, _ = fp8_path.attention_rounded_p(qd, kd, vd, 1 / np.sqrt(D), causal)
    ref = fp8_bound.reference(qd, kd, vd, sv, 1 / np.sqrt(D), causal)
    r = fp8_bound.check(_bf16(O_emul), ref["lse"], ref)
    print(r)


@pytest.mark.parametrize("causal", [False, True])
def test_running_reference_and_folded_v_ratio_lie_within_the_bounds(causal):
    B, S, H, D = 1, 700, 2, 64
    q, k, v = _inputs(B, S, H, D, case=302, gains=True)
    (qd, kd, vd), sv, _ = _quantised(q, k, v, synth.signs(D, 12).astype(np.float64))
    assert fp8_bound.v_ratio(sv).min() < 0.05            # the subnormal term matters here
    O = _lazy_fold_emulation(qd, kd, vd, sv, 1 / np.sqrt(D), causal, seed=3)
    ref = fp8_bound.reference(qd, kd, vd, sv, 1 / np.sqrt(D), causal)
    fp8_bound.check(_bf16(O), ref["lse"], ref)


def _base_case():
    B, S, H, D = 1, 2048, 2, 64
    q, k, v = _inputs(B, S, H, D, case=303)
    (qd, kd, vd), sv, _ = _quantised(q, k, v, synth.signs(D, 13).astype(np.float64))
    rows = np.arange(0, S, 16)
    O_emul, _ = fp8_path.attention_rounded_p(qd, kd, vd, 1 / np.sqrt(D), False, rows)
    ref = fp8_bound.reference(qd, kd, vd, sv, 1 / np.sqrt(D), False, rows)
    return qd, kd, vd, sv, rows, _bf16(O_emul), ref


def test_planted_mistakes_fail_the_check():
    qd, kd, vd, sv, rows, O, ref = _base_case()
    D = qd.shape[-1]
    fp8_bound.check(O, ref["lse"], ref)                  # the unplanted result passes
    # (1) one V block read with twice its scale
    v2 = vd.copy()
    v2[:, 512:640] *= 2
    O1, _ = fp8_path.attention_rounded_p(qd, kd, v2, 1 / np.sqrt(D), False, rows)
    with pytest.raises(AssertionError):
        fp8_bound.check(_bf16(O1), ref["lse"], ref)
    # (2) a causal mask that hides the diagonal key (query i sees keys j < i)
    S2, D2 = 256, qd.shape[-1]
    q2, k2, v2_ = (t[:, :S2] for t in (qd, kd, vd))
    rows2 = np.arange(1, S2)
    ref2 = fp8_bound.reference(q2, k2, v2_, sv[:, :, :2], 1 / np.sqrt(D2), True, rows2)
    shifted = fp8_bound.reference(q2[:, 1:], k2[:, :-1], v2_[:, :-1], sv[:, :, :2], 1 / np.sqrt(D2), True)
    fp8_bound.check(ref2["O"], ref2["lse"], ref2)
    with pytest.raises(AssertionError):
        fp8_bound.check(_bf16(shifted["O"]), ref2["lse"], ref2)
    # (3) the output scaled by 1.5 (a wrong descale; forgetting the V scale would be far larger)
    with pytest.raises(AssertionError):
        fp8_bound.check(_bf16(O * 1.5), ref["lse"], ref)
    # (4) lse off by 2e-3
    with pytest.raises(AssertionError):
        fp8_bound.check(O, ref["lse"] + 2e-3, ref)
    # (5) two query rows exchanged
    O5 = O.copy()
    O5[:, [3, 4]] = O5[:, [4, 3]]
    with pytest.raises(AssertionError):
        fp8_bound.check(O5, ref["lse"], ref)


def test_tie_widths_cover_codes_that_take_the_other_neighbour():
    # inputs whose quotients often sit on E4M3 midpoints (bf16 values, no rotation); flip every
    # near-tie code to its other neighbour, as a quantiser deciding ties in fp32 may
    B, S, H, D = 1, 300, 2, 64
    q, k, v = _inputs(B, S, H, D, case=304)
    (qd, kd, vd), sv, res = _quantised(q, k, v, None)
    flipped = []
    n_flip = 0
    for r in res:
        pre, qv = r["pre"], r["q"].copy()
        step = quantise.grid_step(pre)
        t = np.abs(pre) / step
        tie = np.abs(t - np.floor(t) - 0.5) * step <= 1e-12
        n_flip += int(tie.sum())
        other = np.sign(pre) * (2 * np.abs(pre) - np.abs(qv))       # the other side of the midpoint
        qv[tie] = other[tie]
        flipped.append(quantise.dequantise(qv, r["scale"] * (1 + 1e-6)))
    assert n_flip > 50
    dq, dk, dv = (fp8_bound.tie_widths_blocks(r) for r in res)
    ref = fp8_bound.reference(qd, kd, vd, sv, 1 / np.sqrt(D), True, dq=dq, dk=dk, dv=dv)
    O, lse = fp8_path.attention_rounded_p(*flipped, 1 / np.sqrt(D), True)
    fp8_bound.check(_bf16(O), lse, ref)
