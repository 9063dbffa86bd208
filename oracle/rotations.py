"""fp64 application of disjoint Givens rotations along one mode (TEST
INFRASTRUCTURE ONLY: only tests/ and bench.py's CPU leg import it).

"An HPC Approach to Accelerate Tensor Decompositions" (the page on the Jacobi
method, §2 and §4.3, "Application of Rotations"): one step multiplies the tensor
in mode n by R^T, where R differs from the identity only in 2 x 2 blocks
[[c, -s], [s, c]] at rows and columns (p, q) of a group of disjoint pivot pairs.
Written out, for every fibre along mode n and every pair g:

    new[p_g] = c_g * old[p_g] + s_g * old[q_g]
    new[q_g] = c_g * old[q_g] - s_g * old[p_g]

and entries whose mode-n index is in no pair stay as they are.

Pins (tests/test_rotations_oracle.py): the explicit mode-n product with the
dense matrix R^T, norm preservation, the inverse rotation, independence of
disjoint pairs.
"""
from __future__ import annotations

import numpy as np


def apply_rotations(Y, mode: int, pairs, c, s) -> np.ndarray:
    """Y x_mode R^T for the disjoint pivot pairs `pairs` (G x 2) with cosines `c`
    and sines `s` (G each); fp64 result, Y unchanged."""
    Y = np.asarray(Y, dtype=np.float64)
    out = np.moveaxis(Y.copy(), mode, 0)
    src = np.moveaxis(Y, mode, 0)
    for (p, q), cg, sg in zip(np.asarray(pairs), np.asarray(c, dtype=np.float64), np.asarray(s, dtype=np.float64)):
        out[p] = cg * src[p] + sg * src[q]
        out[q] = cg * src[q] - sg * src[p]
    return np.moveaxis(out, 0, mode)


def rotation_matrix(N: int, pairs, c, s) -> np.ndarray:
    """R (N x N): the identity with the blocks [[c, -s], [s, c]] at (p, q)."""
    R = np.eye(N)
    for (p, q), cg, sg in zip(np.asarray(pairs), c, s):
        R[p, p] = cg
        R[p, q] = -sg
        R[q, p] = sg
        R[q, q] = cg
    return R
