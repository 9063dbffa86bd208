"""fp64 dense mode-n product, TTM (TEST INFRASTRUCTURE ONLY: only tests/ and
bench.py's CPU leg import it).

"An HPC Approach to Accelerate Tensor Decompositions", §2, eq. (1): for a
tensor X of size I_1 x ... x I_D and a matrix M of size J x I_n, the mode-n
product T = X x_n M has size I_1 x ... x I_{n-1} x J x I_{n+1} x ... x I_D and

    t[i_1 .. i_{n-1}, j, i_{n+1} .. i_D] = sum over i_n of x[i_1 .. i_n .. i_D] * m[j, i_n].

Modes are numbered from 0 here.  `ttm` is that sum with the contracted index
moved last and one matrix product as the library step; `ttm_loops` is the same
sum as plain Python loops, for tiny inputs.

Pins (tests/test_ttm_oracle.py): the loops on tiny inputs for every mode, the
d = 2 cases as matrix products, the identity matrix, composition in one mode,
commutation across two modes, the rank-one closed form, the 2-way MTTKRP
oracle on the permuted tensor, and planted mistakes.
"""
from __future__ import annotations

import itertools

import numpy as np


def ttm(X, mode: int, M) -> np.ndarray:
    """X x_mode M in fp64 (X unchanged)."""
    X = np.asarray(X, dtype=np.float64)
    M = np.asarray(M, dtype=np.float64)
    if M.ndim != 2 or M.shape[1] != X.shape[mode]:
        raise ValueError("M must be J x I_mode")
    Xm = np.moveaxis(X, mode, -1)             # [..., I_mode]
    T = Xm @ M.T                              # [..., J]: sum over i of x[..., i] m[j, i]
    return np.moveaxis(T, -1, mode)


def ttm_loops(X, mode: int, M) -> np.ndarray:
    """The same sum, one output entry at a time (tiny inputs only)."""
    X = np.asarray(X, dtype=np.float64)
    M = np.asarray(M, dtype=np.float64)
    J, In = M.shape
    shape = list(X.shape)
    shape[mode] = J
    T = np.zeros(shape)
    for idx in itertools.product(*[range(n) for n in shape]):
        j = idx[mode]
        acc = 0.0
        for i in range(In):
            src = idx[:mode] + (i,) + idx[mode + 1:]
            acc += X[src] * M[j, i]
        T[idx] = acc
    return T
