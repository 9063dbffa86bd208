"""Pins of the fp64 rotation oracle (CPU): the definition against the explicit
mode-n product with the dense rotation matrix, and properties an orthogonal
update must have."""
import numpy as np
import pytest

from oracle import rotations as rot


def case(seed, dims, mode, G):
    rng = np.random.default_rng(seed)
    Y = rng.standard_normal(dims)
    perm = rng.permutation(dims[mode])[: 2 * G].reshape(G, 2)
    phi = rng.uniform(-np.pi, np.pi, G)
    return Y, perm, np.cos(phi), np.sin(phi)


@pytest.mark.parametrize("dims,mode,G", [((6, 7, 8), 0, 3), ((6, 7, 8), 1, 2), ((5, 4, 3, 10), 3, 5),
                                         ((9, 2), 0, 4)])
def test_equals_mode_product_with_rotation_transpose(dims, mode, G):
    Y, pairs, c, s = case(1 + mode + G, dims, mode, G)
    R = rot.rotation_matrix(dims[mode], pairs, c, s)
    # (Y x_n R^T)_{..i..} = sum_j R^T[i][j] Y_{..j..}
    want = np.moveaxis(np.tensordot(R.T, np.moveaxis(Y, mode, 0), axes=(1, 0)), 0, mode)
    assert np.allclose(rot.apply_rotations(Y, mode, pairs, c, s), want, rtol=1e-13, atol=1e-13)


def test_orthogonal_update_properties():
    Y, pairs, c, s = case(7, (8, 9, 10), 1, 4)
    Z = rot.apply_rotations(Y, 1, pairs, c, s)
    assert np.isclose(np.linalg.norm(Z), np.linalg.norm(Y), rtol=1e-13)
    back = rot.apply_rotations(Z, 1, pairs, c, -s)          # the inverse rotation
    assert np.allclose(back, Y, rtol=1e-12, atol=1e-12)
    untouched = np.setdiff1d(np.arange(9), pairs.ravel())
    assert np.array_equal(Z[:, untouched, :], Y[:, untouched, :])
    # disjoint pairs act independently: one pair at a time gives the same
    W = Y.copy()
    for g in range(4):
        W = rot.apply_rotations(W, 1, pairs[g:g + 1], c[g:g + 1], s[g:g + 1])
    assert np.allclose(W, Z, rtol=1e-13, atol=1e-13)


def test_planted_sign_mistake_is_caught():
    Y, pairs, c, s = case(9, (6, 7, 8), 2, 3)
    R = rot.rotation_matrix(8, pairs, c, s)
    wrong = np.moveaxis(np.tensordot(R, np.moveaxis(Y, 2, 0), axes=(1, 0)), 0, 2)   # R instead of R^T
    assert not np.allclose(rot.apply_rotations(Y, 2, pairs, c, s), wrong, atol=1e-6)


def _mutant(Y, mode, pairs, c, s, kind):
    out = np.moveaxis(np.array(Y, dtype=np.float64), mode, 0)
    for (p, q), cg, sg in zip(pairs, c, s):
        x, y = out[p].copy(), out[q].copy()
        if kind == "sign":                 # sine sign flipped in both rows
            out[p], out[q] = cg * x - sg * y, cg * y + sg * x
        elif kind == "in_place":           # q updated from the already-updated p
            out[p] = cg * x + sg * y
            out[q] = cg * y - sg * out[p]
        elif kind == "swap":               # p and q roles exchanged
            out[q], out[p] = cg * y + sg * x, cg * x - sg * y
    return np.moveaxis(out, 0, mode)


@pytest.mark.parametrize("kind", ["sign", "in_place", "swap"])
def test_plausible_mistakes_fail_the_dense_product_pin(kind):
    Y, pairs, c, s = case(11, (6, 8, 5), 1, 3)
    R = rot.rotation_matrix(8, pairs, c, s)
    want = np.moveaxis(np.tensordot(R.T, np.moveaxis(Y, 1, 0), axes=(1, 0)), 0, 1)
    assert np.allclose(rot.apply_rotations(Y, 1, pairs, c, s), want, rtol=1e-13, atol=1e-13)
    assert not np.allclose(_mutant(Y, 1, pairs, c, s, kind), want, atol=1e-6)
