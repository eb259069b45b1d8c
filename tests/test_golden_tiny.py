"""The oracle still reproduces its stored tiny fixture (regression guard, CPU only).

tests/golden/tiny_attention.json is written by tests/golden/make_tiny_attention.py,
which calls only the oracle.  A change to the oracle's arithmetic that moves
these numbers must regenerate the fixture and say why in its commit.
"""

import json
import os

import numpy as np

from oracle import attention as A

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_fixture_reproduces():
    with open(os.path.join(HERE, "golden", "tiny_attention.json")) as f:
        g = json.load(f)
    shape = g["shape"]
    q, k, v = (np.array(g[n]).reshape(shape) for n in ("q", "k", "v"))
    for key, causal in (("full", False), ("causal", True)):
        O, lse = A.attention(q, k, v, scale=g["scale"], causal=causal)
        np.testing.assert_allclose(O.ravel(), g[key]["O"], atol=1e-15)
        np.testing.assert_allclose(lse.ravel(), g[key]["lse"], atol=1e-15)
