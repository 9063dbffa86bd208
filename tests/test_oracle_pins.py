"""Pins of the fp64 oracle against facts fixed by the mathematics (CPU only).

The oracle computes the matricized tensor times Khatri-Rao product of "A
Performance Portable Matrix Free Dense MTTKRP in GenTen" (abstract).  None of
the checks here re-runs the oracle's own formula: each compares it with
something it was not derived from.

  * a hand-worked 2x2x2 example (tests/golden/hand_2x2x2.txt);
  * brute force: the Khatri-Rao matrix formed explicitly (the matrix-based
    MTTKRP the abstract contrasts with) and multiplied with the mode-k
    unfolding ("An HPC Approach to Accelerate Tensor Decompositions",
    section 2: matricization in a fixed, consistent ordering);
  * the closed form for exact rank-S tensors,
    M_k = B_k (*)_{n != k} (B_n^T A_n)   ((*) = Hadamard product);
  * invariance under a permutation of the modes;
  * special cases: d = 2 is a matrix product, all-ones factors with R = 1
    give marginal sums, one-hot factor columns give a fibre of Y, scaling a
    factor by a power of two scales the result exactly;
  * thread-count independence of the parallel loop nest.
"""
import itertools
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import synth
from conftest import rel_fro

HERE = os.path.dirname(os.path.abspath(__file__))


def brute_force_krp(Y, A, k):
    """Y_(k) @ KRP with the Khatri-Rao matrix formed explicitly (fp64).

    Unfolding: rows i_k, columns the other modes in C order (first other mode
    slowest).  KRP row for those indices = elementwise product of the factor
    rows, built here as column-wise Kronecker products in the same order.
    """
    Y = np.asarray(Y, dtype=np.float64)
    d = Y.ndim
    R = A[0].shape[1]
    others = [n for n in range(d) if n != k]
    unfold = np.moveaxis(Y, k, 0).reshape(Y.shape[k], -1)
    krp = np.empty((unfold.shape[1], R))
    for r in range(R):
        col = np.ones(1)
        for n in others:
            col = np.kron(col, np.asarray(A[n][:, r], dtype=np.float64))
        krp[:, r] = col
    # textbook triple loop would be identical; the matrix product is a library step
    return unfold @ krp


def closed_form(B, A, k):
    S = B[0].shape[1]
    R = A[0].shape[1]
    H = np.ones((S, R))
    for n in range(len(B)):
        if n != k:
            H *= B[n].T @ np.asarray(A[n], dtype=np.float64)
    return B[k] @ H


# ---------------------------------------------------------------------------


def test_hand_worked_example():
    Y = (1 + np.arange(8, dtype=np.float64)).reshape(2, 2, 2)
    A = [np.array([[1.0, 1.0], [1000.0, 1.0]]),
         np.array([[1.0, 1.0], [10.0, 1.0]]),
         np.array([[1.0, 1.0], [100.0, 1.0]])]
    rows = [l.split() for l in open(os.path.join(HERE, "golden", "hand_2x2x2.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 6
    for fn in (oracle.mttkrp, oracle.mttkrp_naive):
        for k in range(3):
            M = fn(Y, A, k)
            for mode, row, m0, m1 in rows:
                if int(mode) == k:
                    assert M[int(row), 0] == float(m0)
                    assert M[int(row), 1] == float(m1)


SHAPES = [
    ((3, 4), 2),
    ((5, 3), 4),
    ((2, 3, 4), 3),
    ((4, 1, 5), 2),
    ((3, 2, 2, 3), 5),
    ((2, 3, 2, 2, 3), 2),
    ((1, 2, 3, 2, 1, 2), 3),
]


@pytest.mark.parametrize("dims,R", SHAPES)
def test_brute_force_krp(dims, R):
    Y, A = synth.random_case(101 + len(dims) * 7 + R, dims, R, dtype=np.float64)
    for k in range(len(dims)):
        ref = brute_force_krp(Y, A, k)
        assert rel_fro(oracle.mttkrp(Y, A, k), ref) <= 1e-13
        assert rel_fro(oracle.mttkrp_naive(Y, A, k), ref) <= 1e-13


def test_brute_force_fp32_input():
    """fp32 Y is converted exactly: the result equals the fp64 run on the same values."""
    Y, A = synth.random_case(7, (4, 5, 3), 4, dtype=np.float32)
    for k in range(3):
        ref = brute_force_krp(Y.astype(np.float64), A, k)
        assert rel_fro(oracle.mttkrp(Y, A, k), ref) <= 1e-13


@pytest.mark.parametrize("dims,S,R", [((6, 5, 4), 3, 4), ((5, 4, 3, 6), 2, 7),
                                      ((3, 4, 2, 3, 2), 4, 3)])
def test_closed_form_rank_sum(dims, S, R):
    seed = 900 + S
    B = [synth.normal(seed, synth.stream_generating_factor(n), (dims[n], S), 0.0, 1.0,
                      dtype=np.float64) for n in range(len(dims))]
    A = [synth.normal(seed, synth.stream_factor(n), (dims[n], R), 0.0, 1.0, dtype=np.float64)
         for n in range(len(dims))]
    Y = synth.rank_sum(B, dtype=np.float64)
    for k in range(len(dims)):
        ref = closed_form(B, A, k)
        assert rel_fro(oracle.mttkrp(Y, A, k), ref) <= 1e-12


def test_closed_form_bump_field_small():
    """The Gaussian-bump workload is an exact rank-32 CP tensor (separable bumps)."""
    w = synth.Workload(4, "bumps_small", (24, 20, 16), 6, "small bump field")
    B = synth.generating_factors(w)
    assert len(B) == 3 and B[0].shape == (24, 32)
    # direct evaluation of one point of the field, sum_j exp(-|x - c_j|^2 / (2 sigma^2))
    centres = synth.uniform(w.seed, synth.STREAM_CENTRES, (32, 3), 0.0, 1.0, dtype=np.float64)
    x = np.array([(5 + 0.5) / 24, (7 + 0.5) / 20, (3 + 0.5) / 16])
    direct = np.exp(-((x[None, :] - centres) ** 2).sum(1) / (2 * 0.05 ** 2)).sum()
    Y = synth.rank_sum(B, dtype=np.float64)
    assert abs(Y[5, 7, 3] - direct) <= 1e-12 * max(1.0, abs(direct))
    A = [synth.normal(w.seed, synth.stream_factor(n), (w.dims[n], w.R), 0.0, 1.0,
                      dtype=np.float64) for n in range(3)]
    for k in range(3):
        assert rel_fro(oracle.mttkrp(Y, A, k), closed_form(B, A, k)) <= 1e-12


@pytest.mark.parametrize("dims,R", [((3, 4, 5), 3), ((2, 3, 4, 5), 2), ((3, 2, 4, 2, 3), 2)])
def test_mode_permutation_invariance(dims, R):
    Y, A = synth.random_case(55, dims, R, dtype=np.float64)
    d = len(dims)
    base = [oracle.mttkrp(Y, A, k) for k in range(d)]
    rng = np.random.default_rng(3)
    for _ in range(4):
        perm = rng.permutation(d)
        Yp = np.ascontiguousarray(np.transpose(Y, perm))
        Ap = [A[p] for p in perm]
        for t in range(d):
            assert rel_fro(oracle.mttkrp(Yp, Ap, t), base[perm[t]]) <= 1e-13


def test_order_two_is_matrix_product():
    Y, A = synth.random_case(11, (7, 9), 5, dtype=np.float64)
    assert rel_fro(oracle.mttkrp(Y, A, 0), Y @ A[1]) <= 1e-14
    assert rel_fro(oracle.mttkrp(Y, A, 1), Y.T @ A[0]) <= 1e-14


def test_all_ones_rank_one_gives_marginals():
    Y, _ = synth.random_case(12, (4, 3, 5, 2), 1, dtype=np.float64)
    ones = [np.ones((n, 1)) for n in Y.shape]
    for k in range(4):
        axes = tuple(n for n in range(4) if n != k)
        assert rel_fro(oracle.mttkrp(Y, ones, k)[:, 0], Y.sum(axis=axes)) <= 1e-14


def test_one_hot_columns_give_fibres():
    dims = (4, 5, 3, 2)
    Y, _ = synth.random_case(13, dims, 1, dtype=np.float64)
    rng = np.random.default_rng(0)
    R = 6
    picks = [rng.integers(0, n, size=R) for n in dims]
    A = []
    for n in range(4):
        a = np.zeros((dims[n], R))
        a[picks[n], np.arange(R)] = 1.0
        A.append(a)
    for k in range(4):
        M = oracle.mttkrp(Y, A, k)
        for r in range(R):
            idx = [picks[n][r] for n in range(4)]
            idx[k] = slice(None)
            np.testing.assert_array_equal(M[:, r], Y[tuple(idx)])


def test_power_of_two_scaling_is_exact():
    Y, A = synth.random_case(14, (3, 4, 5), 3, dtype=np.float64)
    for k in range(3):
        M = oracle.mttkrp(Y, A, k)
        for n in range(3):
            A2 = [a.copy() for a in A]
            A2[n] *= 8.0
            M2 = oracle.mttkrp(Y, A2, k)
            np.testing.assert_array_equal(M2, M if n == k else 8.0 * M)


def test_row_subset_matches_full():
    Y, A = synth.random_case(15, (6, 7, 5), 4, dtype=np.float32)
    for k in range(3):
        full = oracle.mttkrp(Y, A, k)
        rows = [Y.shape[k] - 1, 0, 2]
        assert rel_fro(oracle.mttkrp(Y, A, k, rows=rows), full[rows]) <= 1e-15


def test_thread_count_independence():
    code = (
        "import numpy as np, oracle, synth, sys;"
        "Y, A = synth.random_case(16, (40, 33, 21), 9);"
        "sys.stdout.write(np.concatenate([oracle.mttkrp(Y, A, k).ravel() for k in range(3)])"
        ".tobytes().hex())"
    )
    root = os.path.dirname(HERE)
    outs = []
    for nt in ("1", "3", "8"):
        env = dict(os.environ, OMP_NUM_THREADS=nt, PYTHONPATH=root)
        outs.append(subprocess.run([sys.executable, "-c", code], env=env, cwd=root,
                                   capture_output=True, text=True, check=True).stdout)
    assert outs[0] == outs[1] == outs[2]


def test_rejects_bad_arguments():
    Y, A = synth.random_case(17, (3, 4), 2)
    with pytest.raises(ValueError):
        oracle.mttkrp(Y, A, 2)
    with pytest.raises(ValueError):
        oracle.mttkrp(Y, A, 0, rows=[3])
    with pytest.raises(ValueError):
        oracle.mttkrp(Y, [A[0]], 0)


def test_regression_fixture():
    """Results written earlier by tests/golden/make_oracle_fixture.py (oracle only)."""
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "make_oracle_fixture", os.path.join(HERE, "golden", "make_oracle_fixture.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    Y, A = synth.random_case(mod.SEED, mod.DIMS, mod.R)
    Ms = [oracle.mttkrp(Y, A, k) for k in range(len(mod.DIMS))]
    n = 0
    for line in open(os.path.join(HERE, "golden", "oracle_small_5x4x3x2.txt")):
        if line.startswith("#") or not line.strip():
            continue
        k, i, r, v = line.split()
        assert abs(Ms[int(k)][int(i), int(r)] - float(v)) <= 1e-14 * max(1.0, abs(float(v)))
        n += 1
    assert n == sum(mod.DIMS) * mod.R
