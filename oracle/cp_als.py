"""fp64 CP-ALS sweep around the MTTKRP oracle (TEST INFRASTRUCTURE ONLY).

Only ``tests/`` and ``bench.py``'s CPU leg may import this module.

CP-ALS is the end-to-end workload of "A Performance Portable Matrix Free Dense
MTTKRP in GenTen" (Fig. 5: per iteration an MTTKRP per mode plus the "other
CP-ALS operations", an inner product and a Cholesky solve among them).  The page
does not print the iteration; this is the standard alternating least squares
sweep it names, in its plainest form:

for every mode n = 0 .. d-1 in turn (each update uses the newest factors):
    V   = Hadamard product over m != n of the Gram matrices A_m^T A_m   (R x R)
    M   = MTTKRP(Y, A, n)                                              (I_n x R)
    A_n = M V^{-1}          (least squares; V is symmetric positive definite and
                             is solved through its Cholesky factor)
    lambda_r = ||A_n(:, r)||_2,  A_n(:, r) /= lambda_r  (a zero column stays zero)
after the sweep, with X = sum_r lambda_r a_r^(0) o ... o a_r^(d-1):
    ||X||^2  = lambda^T (Hadamard product of all Gram matrices) lambda
    <Y, X>   = sum_r lambda_r sum_i M(i, r) A_{d-1}(i, r)   (M of the last mode)
    fit      = 1 - sqrt(max(||Y||^2 + ||X||^2 - 2 <Y, X>, 0)) / ||Y||

Everything is fp64; the MTTKRP step is the fp64 oracle of this package.
Pins (tests/test_cp_als_oracle.py): one sweep started at the exact factors of a
rank-R tensor returns them with fit 1; the fit formula against an explicitly
formed X; the normal equations of the last update; fits that do not decrease.
"""
from __future__ import annotations

import numpy as np

from . import mttkrp


def gram(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a, dtype=np.float64)
    return a.T @ a


def cholesky_solve(V: np.ndarray, B: np.ndarray) -> np.ndarray:
    """X with V X = B for symmetric positive definite V (lower Cholesky factor)."""
    L = np.linalg.cholesky(V)
    Z = np.linalg.solve(L, B)          # forward substitution
    return np.linalg.solve(L.T, Z)     # back substitution


def cp_als_sweep(Y, factors, norm_y2: float | None = None):
    """One sweep.  Returns (factors (fp64, normalised columns), lambda, fit, M_last)."""
    Y = np.asarray(Y)
    d = Y.ndim
    A = [np.asarray(a, dtype=np.float64).copy() for a in factors]
    R = A[0].shape[1]
    G = [gram(a) for a in A]
    if norm_y2 is None:
        norm_y2 = float(np.sum(np.asarray(Y, dtype=np.float64) ** 2))
    lam = np.ones(R)
    M = None
    for n in range(d):
        V = np.ones((R, R))
        for m in range(d):
            if m != n:
                V *= G[m]
        M = mttkrp(Y, A, n)
        An = cholesky_solve(V, M.T).T
        lam = np.linalg.norm(An, axis=0)
        safe = np.where(lam > 0, lam, 1.0)
        An = An / safe
        A[n] = An
        G[n] = gram(An)
    H = np.ones((R, R))
    for m in range(d):
        H *= G[m]
    norm_x2 = float(lam @ H @ lam)
    inner = float(np.sum(lam * np.sum(M * A[d - 1], axis=0)))
    fit = 1.0 - np.sqrt(max(norm_y2 + norm_x2 - 2.0 * inner, 0.0)) / np.sqrt(norm_y2)
    return A, lam, fit, M


def reconstruct(factors, lam) -> np.ndarray:
    """X = sum_r lambda_r a_r^(0) o ... o a_r^(d-1) (small tensors only)."""
    d = len(factors)
    letters = "abcdefgh"[:d]
    spec = ",".join(f"{c}r" for c in letters) + ",r->" + letters
    return np.einsum(spec, *[np.asarray(a, dtype=np.float64) for a in factors], np.asarray(lam))
