"""fp64 CPU oracle for the fused exact-attention forward and its FP8 path.

TEST INFRASTRUCTURE ONLY.  The product (the CUDA library and its Python
binding) never imports, calls or executes anything in this package; only the
tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference leg of
``bench.py`` may.  It shares no code with the CUDA path.

Sources (web pages, cited by title and section):

* "FlashAttention-3 (NL)" (systems-analysis.info), its Greek twin
  "FlashAttention-3 (EL)" (a sentence-for-sentence translation), and
* "FlashAttention-3: Schnellere und präzisere Attention durch Asynchronität
  und geringe Präzision" (hada.io summary of the FA3 announcement).

Modules:

* ``attention``  -- materialised-softmax attention (the definition) and a
  blockwise online-softmax recomputation used only to pin it.
* ``hadamard``   -- explicit Sylvester Hadamard matrix and the random-sign
  rotation (incoherent processing).
* ``e4m3``       -- the FP8 E4M3 number format: round-to-nearest-even,
  saturating, written from the format's definition.
* ``quantise``   -- per (b, h, 128-token block) scale + E4M3 quantiser with
  optional rotation.
* ``fp8_path``   -- the FP8 path end to end: rotate, quantise, attend on
  the de-quantised values, with P rounded to E4M3.
* ``backward``   -- gradients dQ, dK, dV of exact attention.
* ``gqa``        -- grouped-query attention and decoding (S_q <= S_k, mask
  aligned at the last key).
* ``varlen``     -- attention over a packed batch of variable-length
  sequences (cu_seqlens offsets).
* ``rope``       -- rotary position embedding (the pages' example of a
  memory-bound op to fuse the rotation with) and its fusion with the
  quantiser.

Every array is numpy float64 unless stated; inputs are the exact values the
GPU sees (bf16 or E4M3 values widened to fp64).
"""

from . import attention, backward, gqa, hadamard, e4m3, quantise, fp8_path, rope, varlen  # noqa: F401
