"""Pins of the fp64 mode-n product oracle (CPU), each independent of the
oracle's own formula: plain loops, textbook matrix-product special cases and
algebraic identities of the mode-n product."""
import numpy as np
import pytest

from oracle import ttm as ottm


def rnd(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("dims,mode,J", [((3, 4, 5), 0, 2), ((3, 4, 5), 1, 6), ((3, 4, 5), 2, 3),
                                         ((2, 3, 2, 3), 3, 4), ((2, 3, 2, 3), 1, 1), ((5,), 0, 3)])
def test_equals_loops(dims, mode, J):
    X = rnd(1 + mode, *dims)
    M = rnd(2 + J, J, dims[mode])
    assert np.allclose(ottm.ttm(X, mode, M), ottm.ttm_loops(X, mode, M), rtol=1e-13, atol=1e-13)


def test_matrix_cases():
    X = rnd(3, 6, 7)
    A = rnd(4, 5, 6)
    B = rnd(5, 4, 7)
    assert np.allclose(ottm.ttm(X, 0, A), A @ X, rtol=1e-13)          # X x_1 A = A X
    assert np.allclose(ottm.ttm(X, 1, B), X @ B.T, rtol=1e-13)        # X x_2 B = X B^T


def test_identity_composition_and_commutation():
    X = rnd(6, 4, 5, 6)
    assert np.array_equal(ottm.ttm(X, 1, np.eye(5)), X)
    A = rnd(7, 3, 5)
    B = rnd(8, 7, 3)
    # (X x_n A) x_n B = X x_n (B A)
    assert np.allclose(ottm.ttm(ottm.ttm(X, 1, A), 1, B), ottm.ttm(X, 1, B @ A), rtol=1e-12, atol=1e-12)
    C = rnd(9, 2, 6)
    # products in different modes commute
    assert np.allclose(ottm.ttm(ottm.ttm(X, 1, A), 2, C), ottm.ttm(ottm.ttm(X, 2, C), 1, A), rtol=1e-12, atol=1e-12)


def test_rank_one_closed_form():
    a, b, c = rnd(10, 4), rnd(11, 5), rnd(12, 6)
    X = np.einsum("i,j,k->ijk", a, b, c)
    M = rnd(13, 3, 5)
    assert np.allclose(ottm.ttm(X, 1, M), np.einsum("i,j,k->ijk", a, M @ b, c), rtol=1e-12, atol=1e-12)


def test_planted_mistakes_are_caught():
    X = rnd(14, 4, 5, 5)
    M = rnd(15, 5, 5)
    want = ottm.ttm_loops(X, 1, M)
    transposed = np.moveaxis(np.moveaxis(X, 1, -1) @ M, -1, 1)     # M instead of M^T
    wrong_mode = ottm.ttm(X, 2, M)
    assert not np.allclose(transposed, want, atol=1e-6)
    assert not np.allclose(wrong_mode, want, atol=1e-6)
    with pytest.raises(ValueError):
        ottm.ttm(X, 0, M)                                           # I_0 = 4 does not match M's 5 columns


@pytest.mark.parametrize("dims,mode,J", [((4, 5, 6), 0, 3), ((4, 5, 6), 1, 7), ((4, 5, 6), 2, 2),
                                         ((3, 2, 4, 5), 2, 6)])
def test_equals_two_way_mttkrp_of_the_permuted_tensor(dims, mode, J):
    """With mode n moved last, Z[(p, q), i] = X[p, i, q]; the 2-way MTTKRP of Z
    for mode 0 with the single factor M^T is sum_i Z[(p, q), i] M[j, i], i.e.
    T[p, j, q] laid out as [(p, q), j].  Ties the mode-n product oracle to the
    MTTKRP oracle (plain C, its own pins)."""
    import oracle
    X = rnd(20 + mode, *dims)
    M = rnd(21 + J, J, dims[mode])
    Z = np.ascontiguousarray(np.moveaxis(X, mode, -1).reshape(-1, dims[mode]))
    A0 = np.zeros((Z.shape[0], J))                        # mode 0's own factor is not used
    M0 = oracle.mttkrp(Z, [A0, np.ascontiguousarray(M.T)], 0)
    want = np.moveaxis(M0.reshape(np.moveaxis(X, mode, -1).shape[:-1] + (J,)), -1, mode)
    assert np.allclose(ottm.ttm(X, mode, M), want, rtol=1e-12, atol=1e-12)
