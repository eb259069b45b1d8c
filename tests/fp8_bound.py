"""Element-wise error bounds for FP8 attention against exact attention on the de-quantised inputs.

Test infrastructure.  The reference values come from the fp64 definition (softmax of the scaled
logits of the de-quantised Q and K, times the de-quantised V); the bounds are derived from the
E4M3 format's rounding error and fp32 arithmetic, not from any kernel's order of operations.

What the FP8 attention step computes ("FlashAttention-3 (NL)", "Technische innovaties", item 3;
hada.io FA3 summary, "Niedrige FP8-Präzision und incoherent processing"): both GEMMs in FP8, so
the softmax numerators are rounded to E4M3 before the P-V product, while the row sum uses the
unrounded numerators.  The library's kernels (a) form each numerator relative to a running
reference m_run <= m_i, the row maximum, and (b) fold V's block scale into it: the E4M3 operand
is p'_ij = p_ij * 2^delta_ij * r_j with p_ij = exp(s_ij - m_i), delta_ij >= 0 and
r_j = sv_j / (largest V block scale of the head, sequence or key range) <= 1; the product with
V's codes is scaled back by that largest scale and divided by the row sum of p'_ij / r_j.  In
real arithmetic this is exactly O = sum_j P_ij v_j; the rounding of p' to E4M3 (nearest) errs by
at most max(2^-4 p', min(p', 2^-10)): half a grid step, which is at most 2^-4 of the value in
the normal range and 2^-10 below 2^-6, and never more than p' itself (a value below 2^-10
rounds to 0).  Carried to the output, with l_i = sum_j p_ij,

    |dO_id| <= sum_j h_ij |v_jd| / l_i,    h_ij = max(2^-4 p_ij, min(p_ij, 2^-10 / r_j))   (worst case)

because 2^delta >= 1 only shrinks the subnormal term.  A key whose V block scale is 0 has
v_j = 0 and contributes nothing.  The same per-key sizes give

* a statistical bound: the rounding errors of different keys meet V entries of random sign,
  so by Hoeffding's inequality |dO_id| <= 7 sqrt(sum_j h_ij^2 v_jd^2) / l_i except with
  probability below 2 exp(-24.5) ~ 5e-11 per element;
* an expected square error: an error spread evenly over [-h, h] has mean square h^2 / 3, so the
  RMS over many elements stays below sqrt(mean(sum_j h_ij^2 v_jd^2 / (3 l_i^2))).

fp32 terms, added to each bound: the logit of a key is a D-term fp32 sum of products of codes
(each addition errs by at most 2^-23 of sum_d |q_d k_d|), times the multiplier, minus the
reference, with exp2 approximated to 2^-21 relative (|d exp| <= ln 2 |dx| + 2^-21 relative);
the P-V and row-sum accumulations make at most n + 2 ceil(n / 128) + 16 roundings of 2^-23 of
the accumulated magnitude (n visible keys; worst case n of them, statistically 7 sqrt(n)).  The
output's bf16 rounding adds half a bf16 ulp.

Inputs that differ from the oracle's (an end-to-end test feeds the GPU quantiser's codes, which
may take the other neighbour at an exact rounding midpoint, and fp32 scales) are covered by
perturbation widths dq, dk, dv: each logit then moves by at most
eps_ij = scale * sum_d (dq_id (|k_jd| + dk_jd) + |q_id| dk_jd), so every P_ij moves by a factor
within exp(+-2 eps_i) and O by at most (exp(2 eps_i) - 1) sum_j P_ij |v_jd| + e^{2 eps_i} sum_j
P_ij dv_jd, and the lse by at most eps_i.
"""

import numpy as np

from tests.helpers import half_ulp_bf16

LN2 = np.log(2.0)
LOG2E = 1.0 / LN2
LSE_TOL = 1e-3


def _rows(q, k, v, vis, scale, r, dq=None, dk=None, dv=None):
    """Reference and bounds for R query rows against N keys (one head).

    q [R, D], k, v [N, D] fp64 de-quantised values; vis [R, N] bool (every row sees a key);
    r [N] the V block-scale ratio of every key (0 where the block's scale is 0)."""
    D = q.shape[1]
    s = scale * (q @ k.T)
    s = np.where(vis, s, -np.inf)
    m = s.max(axis=1)
    p = np.where(vis, np.exp(s - m[:, None]), 0.0)
    l = p.sum(axis=1)
    P = p / l[:, None]
    O = P @ v
    lse = m + np.log(l)
    av = np.abs(v)
    # fp32 error of the exponent argument, and the relative error of each numerator
    A = np.abs(q) @ np.abs(k).T
    x = np.where(vis, s * LOG2E, 0.0)
    dx = D * 2.0 ** -23 * scale * LOG2E * A + 2.0 ** -21 * (np.abs(x) + np.abs(m * LOG2E)[:, None]) + 2.0 ** -20
    gam = np.where(vis, LN2 * dx + 2.0 ** -21, 0.0)
    live = vis & (r > 0)[None, :]
    rr = np.where(r > 0, r, 1.0)[None, :]
    sub = np.where(live, 2.0 ** -10 / rr, 0.0)
    h = np.where(live, np.maximum(2.0 ** -4 * (1.0 + gam) * p, np.minimum((1.0 + gam) * p, sub)) + gam * p, 0.0)
    E_w = (h @ av) / l[:, None]
    E_s2 = ((h * h) @ (v * v)) / (l * l)[:, None]
    n = vis.sum(axis=1).astype(np.float64)
    W = ((1.07 * p + sub) @ av) / l[:, None]
    nacc = n + 2 * np.ceil(n / 128) + 16
    gmax = gam.max(axis=1)
    worst = E_w + (nacc * 2.0 ** -23 + gmax)[:, None] * W
    stat = 7.0 * np.sqrt(E_s2) + (7.0 * np.sqrt(nacc) * 2.0 ** -23 + gmax)[:, None] * W
    var = E_s2 / 3.0
    eps = np.zeros_like(m)
    if dq is not None:
        e = scale * (dq @ (np.abs(k) + dk).T + np.abs(q) @ dk.T)
        eps = np.where(vis, e, 0.0).max(axis=1)
        g = np.exp(2 * eps)[:, None]
        pv = P @ av
        worst = g * worst + (g - 1) * pv + g * (P @ dv)
        stat = g * stat + (g - 1) * pv + g * (P @ dv)
    return O, lse, worst, stat, var, n, eps


def v_ratio(v_scale):
    """r per block: the block's V scale over the largest of the given blocks (0 if all are 0)."""
    v_scale = np.asarray(v_scale, dtype=np.float64)
    mx = v_scale.max(axis=-1, keepdims=True)
    return np.where(mx > 0, v_scale / np.where(mx > 0, mx, 1.0), 0.0)


def reference(qd, kd, vd, v_scale, scale, causal, rows=None, dq=None, dk=None, dv=None):
    """Exact attention on de-quantised inputs with the FP8 bounds, for [B, S, H, D] layouts.

    qd [B, Sq, Hq, D]; kd, vd [B, Sk, Hkv, D] (Hq a multiple of Hkv: query head h reads key/value
    head h // (Hq / Hkv)); v_scale [B, Hkv, ceil(Sk / 128)], the V block scales the kernel gets;
    causal: query i sees keys j <= Sk - Sq + i.  rows: query rows to compute (default all).
    dq, dk, dv: optional perturbation widths of the inputs (same shapes).
    Returns a dict of O [B, R, Hq, D], lse [B, Hq, R], worst / stat / var [B, R, Hq, D],
    n [B, R, Hq] (visible keys) and eps [B, Hq, R]."""
    B, Sq, Hq, D = qd.shape
    Sk, Hkv = kd.shape[1], kd.shape[2]
    G = Hq // Hkv
    rows = np.arange(Sq) if rows is None else np.asarray(rows, dtype=np.int64)
    R = len(rows)
    keys = np.arange(Sk)
    vis = (keys[None, :] <= (Sk - Sq + rows)[:, None]) if causal else np.ones((R, Sk), dtype=bool)
    out = {k_: np.zeros((B, R, Hq, D)) for k_ in ("O", "worst", "stat", "var")}
    out["lse"] = np.zeros((B, Hq, R))
    out["eps"] = np.zeros((B, Hq, R))
    out["n"] = np.zeros((B, R, Hq))
    ratio = v_ratio(v_scale)
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            r = ratio[b, hk][keys // 128]
            pert = () if dq is None else (dq[b, rows, h], dk[b, :, hk], dv[b, :, hk])
            O, lse, w, st, var, n, eps = _rows(qd[b, rows, h], kd[b, :, hk], vd[b, :, hk], vis, scale, r, *pert)
            out["O"][b, :, h], out["worst"][b, :, h], out["stat"][b, :, h], out["var"][b, :, h] = O, w, st, var
            out["lse"][b, h], out["n"][b, :, h], out["eps"][b, h] = lse, n, eps
    return out


def reference_varlen(qd, kd, vd, v_scale, cu_seqlens, scale, causal, dq=None, dk=None, dv=None):
    """The same for a packed batch: qd, kd, vd [total, H, D]; v_scale [H, NB] with sequence s's
    blocks at cu[s] // 128 + s + (0, 1, ...).  Returns the dict with a leading batch axis of 1."""
    total, H, D = qd.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    out = {k_: np.zeros((1, total, H, D)) for k_ in ("O", "worst", "stat", "var")}
    out["lse"] = np.zeros((1, H, total))
    out["eps"] = np.zeros((1, H, total))
    out["n"] = np.zeros((1, total, H))
    for s in range(len(cu) - 1):
        s0, n = int(cu[s]), int(cu[s + 1] - cu[s])
        if n == 0:
            continue
        nblk = (n + 127) // 128
        base = s0 // 128 + s
        sl = slice(s0, s0 + n)
        pert = {} if dq is None else {"dq": dq[None, sl], "dk": dk[None, sl], "dv": dv[None, sl]}
        o = reference(qd[None, sl], kd[None, sl], vd[None, sl], v_scale[None, :, base:base + nblk], scale, causal,
                      **pert)
        for k_ in ("O", "worst", "stat", "var", "n"):
            out[k_][:, sl] = o[k_]
        out["lse"][:, :, sl] = o["lse"]
        out["eps"][:, :, sl] = o["eps"]
    return out


def rms(x):
    return float(np.sqrt(np.mean(np.square(x)))) if np.size(x) else 0.0


def check(o, lse, ref, lse_tol=LSE_TOL, rms_min_keys=128):
    """Assert the three FP8 bounds element by element (o [B, R, H, D] fp64 from the GPU) and the
    lse within lse_tol (+ the perturbation eps).  Returns the largest error/bound ratios."""
    O = ref["O"]
    assert np.isfinite(o).all(), "non-finite output"
    err = np.abs(o - O)
    worst = ref["worst"] + half_ulp_bf16(np.abs(O) + ref["worst"])
    stat = ref["stat"] + half_ulp_bf16(np.abs(O) + ref["stat"])
    def ratio(bound):
        # an exact zero (a zero value, or no error possible) must be met exactly
        safe = np.where(bound > 0, bound, 1.0)
        return float(np.where(bound > 0, err / safe, np.where(err > 0, np.inf, 0.0)).max())

    r_w, r_s = ratio(worst), ratio(stat)
    assert r_w <= 1.0, f"worst-case bound exceeded: {int((err > worst).sum())} elements, max ratio {r_w:.3f}"
    assert r_s <= 1.0, f"statistical bound exceeded: {int((err > stat).sum())} elements, max ratio {r_s:.3f}"
    many = np.broadcast_to((ref["n"] >= rms_min_keys)[..., None], err.shape)
    r_rms = 0.0
    if many.any():
        e_rms = rms(err[many])
        allowed = 1.5 * np.sqrt(np.mean(ref["var"][many])) + rms(half_ulp_bf16(O[many])) + 1e-7
        r_rms = e_rms / allowed
        assert r_rms <= 1.0, f"RMS {e_rms:.3e} above the expected {allowed:.3e}"
    if lse is not None:
        lerr = np.abs(lse - ref["lse"]) - ref["eps"]
        assert float(lerr.max()) <= lse_tol, float(lerr.max())
    return {"worst": r_w, "stat": r_s, "rms": r_rms}


def tie_widths(pre, per_scale, tie_rtol=1e-5, tie_atol=1e-12, scale_rtol=2e-6):
    """Perturbation widths of de-quantised inputs whose codes may take the other neighbour at a
    rounding midpoint (where the oracle's pre-rounding quotient ``pre`` lies within
    tie_rtol * |pre| + tie_atol of one) and whose scales may differ by scale_rtol: one grid step
    times the element's block scale ``per_scale`` there, plus scale_rtol of every value."""
    from oracle import quantise
    step = quantise.grid_step(pre)
    t = np.abs(pre) / step
    near = np.abs(t - np.floor(t) - 0.5) * step <= tie_rtol * np.abs(pre) + tie_atol
    return np.where(near, step * per_scale, 0.0) + scale_rtol * (np.abs(pre) + step) * per_scale


def tie_widths_blocks(qres, tie_rtol=1e-5, tie_atol=1e-12, scale_rtol=2e-6):
    """tie_widths for the oracle quantiser's dict of a [B, S, H, D] tensor."""
    from oracle import quantise
    per_scale = quantise.dequantise(np.ones_like(qres["pre"]), qres["scale"])
    return tie_widths(qres["pre"], per_scale, tie_rtol, tie_atol, scale_rtol)
