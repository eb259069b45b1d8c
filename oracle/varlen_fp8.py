"""The FP8 path over a packed batch of variable-length sequences, fp64 with E4M3 rounding
emulated.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources: the FP8 path of "FlashAttention-3 (NL)", "Technische innovaties", item 3, and of the
hada.io FA3 summary, "Niedrige FP8-Präzision und incoherent processing" (rotate Q and K,
quantise per 128-token block, attend in FP8), applied to the packed batches of the same
summary's "Weitere Optimierungen und künftige Integration".  The pages define neither the
combination nor the block layout.

Readings:
* a scale block never straddles two sequences: sequence s is cut into blocks of 128 tokens
  from its own first token (the last one may be shorter), and each (block, head) gets one
  scale, amax / 448, exactly as ``quantise.quantise_blocks`` does for a single sequence;
* the scales of all sequences share one array [H, NB] with NB = total // 128 + n_seq + 1;
  block k of sequence s sits at index cu[s] // 128 + s + k.  These indices never collide
  (a sequence of length L starting at a covers ceil(L / 128) <= (a + L) // 128 - a // 128 + 1
  indices) and stay below NB; unused indices carry no meaning;
* the attention of every sequence is the FP8 path of ``fp8_path`` on its own de-quantised
  values;
* with rotary embedding in front (``rope_base``), positions restart at every sequence's first
  token: each sequence is embedded as ``rope.rope`` embeds a tensor of its own.
"""

import numpy as np

from . import fp8_path
from .quantise import quantise_blocks, dequantise
from .rope import rope
from .varlen import segments

__all__ = ["scale_blocks", "block_base", "quantise_varlen", "fp8_attention_varlen"]


def scale_blocks(total, n_seq):
    """NB, the number of scale entries per head."""
    return total // 128 + n_seq + 1


def block_base(cu_seqlens):
    """Index of the first scale block of every sequence: cu[s] // 128 + s."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    return cu[:-1] // 128 + np.arange(cu.size - 1)


def quantise_varlen(x, cu_seqlens, signs=None, rope_base=None):
    """Quantise packed x [total, H, D] (fp64 values) sequence by sequence (after rotary
    embedding with positions 0 .. len-1 of each sequence when ``rope_base`` is given).

    Returns a dict with ``q`` (E4M3 values), ``codes`` and ``pre`` (the value rounded, as in
    ``quantise_blocks``) [total, H, D], ``scale`` [H, NB] (NaN where no block lives), and
    ``deq``, the de-quantised values [total, H, D].
    """
    x = np.asarray(x, dtype=np.float64)
    total, H, D = x.shape
    segs = segments(cu_seqlens)
    base = block_base(cu_seqlens)
    scale = np.full((H, scale_blocks(total, len(segs))), np.nan)
    q = np.zeros_like(x)
    pre = np.zeros_like(x)
    codes = np.zeros(x.shape, dtype=np.uint8)
    deq = np.zeros_like(x)
    for s, (s0, n) in enumerate(segs):
        if n == 0:
            continue
        xs = x[None, s0:s0 + n] if rope_base is None else rope(x[None, s0:s0 + n], rope_base)
        r = quantise_blocks(xs, signs)
        nblk = r["scale"].shape[2]
        scale[:, base[s]:base[s] + nblk] = r["scale"][0]
        q[s0:s0 + n] = r["q"][0]
        pre[s0:s0 + n] = r["pre"][0]
        codes[s0:s0 + n] = r["codes"][0]
        deq[s0:s0 + n] = dequantise(r["q"], r["scale"])[0]
    return {"q": q, "pre": pre, "codes": codes, "scale": scale, "deq": deq}


def fp8_attention_varlen(qd, kd, vd, cu_seqlens, scale, causal=False, round_p=True):
    """Attention of every packed sequence on de-quantised qd, kd, vd [total, H, D], with the
    softmax numerators rounded to E4M3 (``round_p``).  Returns (O [total, H, D], lse [H, total])."""
    total, H, D = qd.shape
    O = np.zeros((total, H, D))
    lse = np.zeros((H, total))
    for s, (s0, n) in enumerate(segments(cu_seqlens)):
        if n == 0:
            continue
        o, l = fp8_path.attention_rounded_p(qd[None, s0:s0 + n], kd[None, s0:s0 + n], vd[None, s0:s0 + n], scale,
                                            causal, None, round_p)
        O[s0:s0 + n] = o[0]
        lse[:, s0:s0 + n] = l[0]
    return O, lse
