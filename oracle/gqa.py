"""Grouped-query attention and decoding (fewer query rows than keys), fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: hada.io FA3 summary, "Weitere Optimierungen und künftige Integration": optimising LLM
inference is named as future work; the pages define neither grouped-query attention nor
decoding.  Readings (the common ones):

* grouped-query attention: Hq query heads share Hkv key/value heads, G = Hq / Hkv; query head h
  reads key/value head h // G (contiguous groups);
* decoding: S_q query tokens are the last S_q positions of a sequence whose S_k >= S_q keys
  include them, so under the causal mask query i (0-based) sees keys j <= S_k - S_q + i (the
  mask is aligned at the bottom-right); without the mask every query sees all S_k keys.

Per query head this is the definition in ``attention`` with that key/value head and mask.

For the FP8 path (inputs already de-quantised from E4M3) ``round_p`` rounds the softmax
numerators exp(s - m) to E4M3 before the product with V, as in ``fp8_path``: relative to the
exact row max, with the row sum taken over the unrounded numerators.
"""

import numpy as np

from .attention import default_scale
from .e4m3 import round_e4m3

__all__ = ["attention_gqa"]


def attention_gqa(q, k, v, scale=None, causal=False, round_p=False):
    """q [B, Sq, Hq, D], k and v [B, Sk, Hkv, D] -> (O [B, Sq, Hq, D], lse [B, Hq, Sq])."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    if Hq % Hkv or Sk < Sq:
        raise ValueError("need Hq a multiple of Hkv and Sk >= Sq")
    G = Hq // Hkv
    if scale is None:
        scale = default_scale(D)
    visible = np.ones((Sq, Sk), dtype=bool)
    if causal:
        visible = np.arange(Sk)[None, :] <= (Sk - Sq + np.arange(Sq))[:, None]
    O = np.empty_like(q)
    lse = np.empty((B, Hq, Sq))
    for b in range(B):
        for h in range(Hq):
            s = scale * (q[b, :, h] @ k[b, :, h // G].T)
            s = np.where(visible, s, -np.inf)
            m = s.max(axis=1)
            e = np.exp(s - m[:, None])
            l = e.sum(axis=1)
            num = round_e4m3(e) if round_p else e
            O[b, :, h] = (num / l[:, None]) @ v[b, :, h // G]
            lse[b, h] = m + np.log(l)
    return O, lse
