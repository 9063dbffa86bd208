"""GPU Givens rotations along a mode (mttkrp_apply_rotations through the C ABI)
against the fp64 oracle on the same seeded inputs.  fp32 arithmetic, one fused
multiply-add per output: element-wise relative error at most a few ulps, so
the check is 1e-6 relative Frobenius plus exact equality of untouched rows."""
import numpy as np
import pytest

from conftest import rel_fro
from oracle import rotations as orot

torch = pytest.importorskip("torch")
import dense_tensor_decomposition_gb300 as mk  # noqa: E402

pytestmark = pytest.mark.gpu


def case(seed, dims, mode, G):
    rng = np.random.default_rng(seed)
    Y = rng.standard_normal(dims).astype(np.float32)
    pairs = rng.permutation(dims[mode])[: 2 * G].reshape(G, 2).astype(np.int32)
    phi = rng.uniform(-np.pi, np.pi, G)
    return Y, pairs, np.cos(phi).astype(np.float32), np.sin(phi).astype(np.float32)


# Q = product of the modes after `mode`.  Row path (Q % 4 == 0, Q >= 1024),
# float4 item path (Q % 4 == 0, 32 <= Q < 1024, incl. Q = 32), shared-memory
# slab path (N * Q <= 8192: innermost mode, odd or short Q, ragged last tile),
# scalar item path (odd or short Q with long slabs); partial and full groups,
# odd mode sizes.
SHAPES = [((64, 48, 256), 0, 20), ((64, 48, 256), 1, 24), ((16, 16, 16, 16, 16), 2, 8), ((20, 40, 32), 1, 20),
          ((64, 48, 256), 2, 128), ((7, 33, 9, 5), 1, 16), ((7, 33, 9, 5), 3, 2), ((300, 257), 1, 1),
          ((50, 60, 8), 1, 30), ((300, 257), 0, 150), ((10, 3000, 8), 1, 1000)]


@pytest.mark.parametrize("dims,mode,G", SHAPES)
def test_rotations_match_oracle(dims, mode, G):
    Y, pairs, c, s = case(sum(dims) + mode + G, dims, mode, G)
    Yd = torch.from_numpy(Y.copy()).cuda()
    mk.apply_rotations(Yd, mode, torch.from_numpy(pairs).cuda(), torch.from_numpy(c).cuda(),
                       torch.from_numpy(s).cuda())
    got = Yd.cpu().numpy()
    want = orot.apply_rotations(Y, mode, pairs, c, s)
    assert rel_fro(got, want) <= 1e-6
    untouched = np.setdiff1d(np.arange(dims[mode]), pairs.ravel())
    assert np.array_equal(np.take(got, untouched, axis=mode), np.take(Y, untouched, axis=mode))


def test_inverse_rotation_restores_and_empty_group_is_a_no_op():
    Y, pairs, c, s = case(5, (40, 64, 512), 1, 32)
    Yd = torch.from_numpy(Y.copy()).cuda()
    P, C, S = (torch.from_numpy(x).cuda() for x in (pairs, c, s))
    mk.apply_rotations(Yd, 1, P, C, S)
    mk.apply_rotations(Yd, 1, P, C, -S)
    assert rel_fro(Yd.cpu().numpy(), Y) <= 1e-6
    Z = torch.from_numpy(Y.copy()).cuda()
    mk.apply_rotations(Z, 1, P[:0], C[:0], S[:0])
    assert torch.equal(Z.cpu(), torch.from_numpy(Y))


def test_rejects_bad_arguments():
    Y = torch.zeros((8, 6, 4), device="cuda")
    P = torch.tensor([[0, 1], [2, 3], [4, 5], [6, 7]], dtype=torch.int32, device="cuda")
    C = torch.ones(4, device="cuda")
    with pytest.raises(mk.MttkrpError):
        mk.apply_rotations(Y, 1, P, C, C)          # 4 pairs do not fit a mode of size 6
    with pytest.raises(mk.MttkrpError):
        mk.apply_rotations(Y, 3, P[:1], C[:1], C[:1])   # mode out of range


@pytest.mark.parametrize("dims,mode", [((512, 512, 512), 0), ((512, 512, 512), 1), ((512, 512, 512), 2),
                                       ((20,) * 6, 4), ((20,) * 6, 5)])
def test_full_size_sampled_fibres(dims, mode):
    """The bench's workloads and launch configurations (a full group of N/2
    pairs): 400 fibres along the mode, each checked against the oracle's
    rotation of the same fibre; fp32 bound per entry: 2^-22 (|c x| + |s y|)."""
    rng = np.random.default_rng(60 + mode + len(dims))
    N = dims[mode]
    G = N // 2
    pairs = rng.permutation(N)[: 2 * G].reshape(G, 2).astype(np.int32)
    phi = rng.uniform(-np.pi, np.pi, G)
    c, s = np.cos(phi).astype(np.float32), np.sin(phi).astype(np.float32)
    Yh = torch.randn(dims, generator=torch.Generator().manual_seed(61 + mode)).numpy()
    Yd = torch.from_numpy(Yh).cuda()
    mk.apply_rotations(Yd, mode, torch.from_numpy(pairs).cuda(), torch.from_numpy(c).cuda(),
                       torch.from_numpy(s).cuda())
    got = Yd.cpu().numpy()
    mag = np.zeros(N)
    for k in range(400):
        at = [int(rng.integers(0, n)) for n in dims]
        at[mode] = slice(None)
        x = Yh[tuple(at)]
        want = orot.apply_rotations(x, 0, pairs, c, s)
        mag[:] = np.abs(x)
        for (p, q), cg, sg in zip(pairs, c, s):
            mag[p] = abs(cg * x[p]) + abs(sg * x[q])
            mag[q] = abs(cg * x[q]) + abs(sg * x[p])
        assert np.all(np.abs(got[tuple(at)] - want) <= 2.0 ** -22 * mag), (k, at)
    del Yd
    torch.cuda.empty_cache()
