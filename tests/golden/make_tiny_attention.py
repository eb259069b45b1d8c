"""Writes tiny_attention.json: a small regression fixture produced by the oracle only.

Run from the repository root:  python tests/golden/make_tiny_attention.py
The inputs are small fixed rational numbers written here; the expected
outputs come from oracle.attention (fp64).  The fixture guards the oracle
against unnoticed changes; it is not one of its independent pins.
"""

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
from oracle import attention as A  # noqa: E402


def inputs():
    B, S, H, D = 1, 6, 2, 4
    idx = np.arange(B * S * H * D).reshape(B, S, H, D)
    q = ((idx * 7) % 11 - 5) / 4.0
    k = ((idx * 5) % 13 - 6) / 4.0
    v = ((idx * 3) % 17 - 8) / 8.0
    return q, k, v


def main():
    q, k, v = inputs()
    out = {"shape": list(q.shape), "scale": 0.5, "q": q.ravel().tolist(), "k": k.ravel().tolist(),
           "v": v.ravel().tolist()}
    for causal in (False, True):
        O, lse = A.attention(q, k, v, scale=0.5, causal=causal)
        out["causal" if causal else "full"] = {"O": O.ravel().tolist(), "lse": lse.ravel().tolist()}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_attention.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
