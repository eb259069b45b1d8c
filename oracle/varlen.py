"""Attention over a packed batch of variable-length sequences, fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: hada.io FA3 summary, "Weitere Optimierungen und künftige Integration":
beyond the blog's content the paper adds variable-length sequences (and a
persistent kernel).  The pages define neither.

Reading: the sequences of a batch are packed along one token axis,
q, k, v [total, H, D], with offsets cu_seqlens[0..n] (cu_seqlens[0] = 0,
non-decreasing, cu_seqlens[n] = total; a sequence may be empty).  Sequence s
owns tokens cu_seqlens[s] .. cu_seqlens[s+1]-1 and attends to its own keys
only, under the causal mask to its own keys j <= i (positions counted from the
sequence's first token).  Per sequence this is exactly the definition in
``attention``; lse is laid out [H, total].
"""

import numpy as np

from .attention import attention, default_scale

__all__ = ["attention_varlen", "segments"]


def segments(cu_seqlens):
    """(start, length) of every sequence, empty ones included."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    if cu.ndim != 1 or cu.size < 1 or cu[0] != 0 or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must start at 0 and be non-decreasing")
    return [(int(cu[s]), int(cu[s + 1] - cu[s])) for s in range(cu.size - 1)]


def attention_varlen(q, k, v, cu_seqlens, scale=None, causal=False, rows=None):
    """Exact attention of every packed sequence.

    q, k, v: [total, H, D].  ``rows``: optional sorted global token indices to
    compute (default: all).  Returns (O [R, H, D], lse [H, R]).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    total, H, D = q.shape
    if scale is None:
        scale = default_scale(D)
    segs = segments(cu_seqlens)
    if segs and segs[-1][0] + segs[-1][1] != total:
        raise ValueError("cu_seqlens[-1] must equal the number of tokens")
    rows = np.arange(total) if rows is None else np.asarray(rows, dtype=np.int64)
    O = np.empty((len(rows), H, D))
    lse = np.empty((H, len(rows)))
    for s0, n in segs:
        if n == 0:
            continue
        sel = np.nonzero((rows >= s0) & (rows < s0 + n))[0]
        if sel.size == 0:
            continue
        o, l = attention(q[None, s0:s0 + n], k[None, s0:s0 + n], v[None, s0:s0 + n], scale, causal,
                         rows[sel] - s0)
        O[sel] = o[0]
        lse[:, sel] = l[0]
    return O, lse
