"""Randomised pins of the mode-n product and rotation oracles (CPU, hypothesis):
identities that must hold for every shape, mode and matrix."""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from oracle import rotations as orot  # noqa: E402
from oracle import ttm as ottm  # noqa: E402

dims_st = st.lists(st.integers(1, 5), min_size=1, max_size=4)


@settings(max_examples=40, deadline=None)
@given(dims=dims_st, data=st.data())
def test_ttm_equals_loops_and_is_linear(dims, data):
    mode = data.draw(st.integers(0, len(dims) - 1))
    J = data.draw(st.integers(1, 4))
    rng = np.random.default_rng(data.draw(st.integers(0, 2 ** 31)))
    X, X2 = rng.standard_normal(dims), rng.standard_normal(dims)
    M = rng.standard_normal((J, dims[mode]))
    T = ottm.ttm(X, mode, M)
    assert np.allclose(T, ottm.ttm_loops(X, mode, M), rtol=1e-12, atol=1e-12)
    # linear in X
    assert np.allclose(ottm.ttm(2.0 * X - X2, mode, M), 2.0 * T - ottm.ttm(X2, mode, M), rtol=1e-12, atol=1e-12)


@settings(max_examples=40, deadline=None)
@given(dims=dims_st, data=st.data())
def test_rotations_are_the_dense_product_and_orthogonal(dims, data):
    mode = data.draw(st.integers(0, len(dims) - 1))
    N = dims[mode]
    G = data.draw(st.integers(0, N // 2))
    rng = np.random.default_rng(data.draw(st.integers(0, 2 ** 31)))
    Y = rng.standard_normal(dims)
    pairs = rng.permutation(N)[: 2 * G].reshape(G, 2)
    phi = rng.uniform(-np.pi, np.pi, G)
    c, s = np.cos(phi), np.sin(phi)
    Z = orot.apply_rotations(Y, mode, pairs, c, s)
    R = orot.rotation_matrix(N, pairs, c, s)
    assert np.allclose(Z, ottm.ttm(Y, mode, R.T), rtol=1e-12, atol=1e-12)   # Y x_n R^T
    assert np.isclose(np.linalg.norm(Z), np.linalg.norm(Y), rtol=1e-12)
