"""Random-sign Hadamard rotation (incoherent processing), explicit matrix, fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources:

* "FlashAttention-3 (NL)", "Technische innovaties", item 3 (Lage precisie
  (FP8)): before attention, queries Q and keys K are multiplied by a random
  orthogonal matrix (for example a Hadamard matrix); because the matrix is
  orthogonal, the product QK^T is unchanged.
* hada.io FA3 summary, "Niedrige FP8-Präzision und incoherent processing":
  the implementation uses a Hadamard transform with random signs, O(d log d)
  per head instead of O(d^2).

Readings where the pages are silent: the Hadamard matrix is Sylvester's
(H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]], natural order); the rotation of
one D-element row x is  x' = (x * s) @ H_D / sqrt(D)  with s a vector of +-1
signs, i.e. R = diag(s) H_D / sqrt(D), which is orthogonal.  Q and K use the
same s (needed for QK^T to be unchanged); V is not rotated.  This oracle
builds H_D explicitly and multiplies -- it never uses a fast transform.
"""

import numpy as np

__all__ = ["sylvester", "rotation_matrix", "rotate"]


def sylvester(D):
    """Explicit D x D Sylvester Hadamard matrix (entries +-1), D a power of two."""
    if D < 1 or (D & (D - 1)) != 0:
        raise ValueError("D must be a power of two")
    H = np.ones((1, 1))
    while H.shape[0] < D:
        H = np.block([[H, H], [H, -H]])
    return H


def rotation_matrix(signs):
    """R = diag(signs) @ H_D / sqrt(D) for a +-1 sign vector of length D."""
    s = np.asarray(signs, dtype=np.float64)
    D = s.shape[0]
    return (s[:, None] * sylvester(D)) / np.sqrt(float(D))


def rotate(x, signs):
    """Rotate every length-D row of x (last axis): x' = x @ diag(s) H_D / sqrt(D)."""
    x = np.asarray(x, dtype=np.float64)
    return x @ rotation_matrix(signs)
