"""Pins of the fp64 CP-ALS oracle (CPU).

Each pin is something the mathematics fixes, not a retyping of the oracle:
an exact rank-R tensor started at its own factors is a fixed point with fit 1;
the fit formula agrees with an explicitly formed model tensor; the last update
satisfies its normal equations; alternating least squares never increases the
residual.  A planted mistake (the Gram of the updated mode kept in V, or the
transposed solve) fails at least one pin.
"""
import numpy as np
import pytest

import oracle
from oracle import cp_als

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def rank_r_tensor(seed, dims, R):
    rng = np.random.default_rng(seed)
    A = [rng.standard_normal((n, R)) for n in dims]
    lam = rng.uniform(1.0, 3.0, R)
    Y = cp_als.reconstruct(A, lam)
    return Y, A, lam


def normalised(A):
    return [a / np.linalg.norm(a, axis=0) for a in A]


def test_exact_rank_r_is_a_fixed_point():
    dims, R = (6, 7, 8), 3
    Y, A, lam = rank_r_tensor(1, dims, R)
    A0 = normalised(A)
    A1, lam1, fit, _ = cp_als.cp_als_sweep(Y, A0)
    for a, b in zip(A1, A0):
        assert np.allclose(a, b, atol=1e-10)
    # lambda carries the scale of every column (product of the original norms)
    scale = lam * np.prod([np.linalg.norm(a, axis=0) for a in A], axis=0)
    assert np.allclose(lam1, scale, rtol=1e-10)
    assert abs(fit - 1.0) < 1e-10


def test_fit_formula_matches_explicit_model():
    rng = np.random.default_rng(2)
    dims, R = (5, 6, 4, 3), 4
    Y = rng.standard_normal(dims)
    A = [rng.standard_normal((n, R)) for n in dims]
    A1, lam, fit, _ = cp_als.cp_als_sweep(Y, A)
    X = cp_als.reconstruct(A1, lam)
    explicit = 1.0 - np.linalg.norm(Y - X) / np.linalg.norm(Y)
    assert abs(fit - explicit) < 1e-10


def test_last_update_satisfies_normal_equations():
    rng = np.random.default_rng(3)
    dims, R = (7, 5, 6), 3
    Y = rng.standard_normal(dims)
    A = [rng.standard_normal((n, R)) for n in dims]
    A1, lam, _, M = cp_als.cp_als_sweep(Y, A)
    n = len(dims) - 1
    V = np.ones((R, R))
    for m in range(len(dims)):
        if m != n:
            V *= A1[m].T @ A1[m]
    # (A_n diag(lambda)) V = M_n and M_n is the MTTKRP with the final other factors
    assert np.allclose((A1[n] * lam) @ V, M, rtol=1e-9, atol=1e-9)
    assert np.allclose(oracle.mttkrp(Y, A1, n), M, rtol=1e-12, atol=1e-12)


def test_residual_never_increases():
    rng = np.random.default_rng(4)
    dims, R = (8, 9, 7), 4
    Y = cp_als.reconstruct([rng.standard_normal((n, R)) for n in dims], np.ones(R))
    Y = Y + 0.05 * rng.standard_normal(dims)
    A = [rng.standard_normal((n, R)) for n in dims]
    fits = []
    for _ in range(8):
        A, lam, fit, _ = cp_als.cp_als_sweep(Y, A)
        fits.append(fit)
    assert all(b >= a - 1e-12 for a, b in zip(fits, fits[1:])), fits
    assert fits[-1] > 0.9


def test_planted_mistakes_are_caught():
    dims, R = (6, 7, 8), 3
    Y, A, lam = rank_r_tensor(5, dims, R)
    A0 = normalised(A)

    def sweep_keeping_own_gram(Y, A):
        A = [a.copy() for a in A]
        G = [a.T @ a for a in A]
        for n in range(len(A)):
            V = np.prod(G, axis=0)          # mistake: includes m == n
            An = cp_als.cholesky_solve(V, oracle.mttkrp(Y, A, n).T).T
            A[n] = An / np.linalg.norm(An, axis=0)
            G[n] = A[n].T @ A[n]
        return A

    def sweep_transposed_solve(Y, A):
        A = [a.copy() for a in A]
        for n in range(len(A)):
            V = np.ones((R, R))
            for m in range(len(A)):
                if m != n:
                    V *= A[m].T @ A[m]
            V = V + np.triu(np.ones((R, R)), 1) * 0.1   # mistake: a non-symmetric system
            An = np.linalg.solve(V.T, oracle.mttkrp(Y, A, n).T).T
            A[n] = An / np.linalg.norm(An, axis=0)
        return A

    for bad in (sweep_keeping_own_gram, sweep_transposed_solve):
        A1 = bad(Y, A0)
        assert not all(np.allclose(a, b, atol=1e-6) for a, b in zip(A1, A0)), bad.__name__
