"""GPU dense mode-n product (mttkrp_ttm and mttkrp_ttm_ws through the C ABI)
against the fp64 oracle on the same seeded inputs.

Tolerances, from the arithmetic (u = 2^-24, fp32 unit roundoff):
  CUDA cores (mttkrp_ttm): every output is one fp32 fused multiply-add chain
    over the N = I_mode products in index order, so
    |T - T_exact| <= gamma_N * (|X| x_mode |M|), gamma_N = N u / (1 - N u).
  Tensor cores (mttkrp_ttm_ws, the fp16 two-term split): each product x m is
    formed from hi/lo parts with relative error <= 3 * 2^-22 plus the fp16
    subnormal floor of each part (2^-25 of the scaled value: 2^-38 of the
    largest |X|, or of the largest |M| in that row); tensor memory accumulates
    the three products of each of at most Kd = min(128, N rounded up to 64)
    indices toward zero (<= 2u a step, 3 Kd steps), and the drains are summed in
    fp32 (gamma over N / 128 terms).  So
    |T - T_exact| <= (6 Kd + 24 + N) u (|X| x_mode |M|) + 2^-36 N max|X| max|M|.
Both also within 1e-5 relative Frobenius."""
import numpy as np
import pytest

from conftest import rel_fro
from oracle import ttm as ottm

torch = pytest.importorskip("torch")
import dense_tensor_decomposition_gb300 as mk  # noqa: E402

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def case(seed, dims, mode, J):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal(dims).astype(np.float32)
    M = rng.standard_normal((J, dims[mode])).astype(np.float32)
    return X, M


def tc_coefficient(N):
    kd = min(128, -(-N // 64) * 64)
    return (6 * kd + 24 + N) * U


def check(got, X, mode, M, tc=False):
    want = ottm.ttm(X, mode, M)
    N = X.shape[mode]
    gamma = N * U / (1 - N * U)
    absprod = ottm.ttm(np.abs(X), mode, np.abs(M))
    if tc:
        bound = tc_coefficient(N) * absprod + 2.0 ** -36 * N * np.abs(X).max() * np.abs(M).max() + 1e-30
    else:
        bound = gamma * absprod + 1e-30
    assert rel_fro(got, want) <= 1e-5
    assert np.all(np.abs(got.astype(np.float64) - want) <= bound)


# Q = product of the modes after `mode`: float4 columns (Q % 4 == 0), scalar
# columns (Q >= 32, odd), float4 along i (innermost, N % 4 == 0), scalar along
# i (short or odd Q); J picks 32/64/128-row tiles, ragged in rows and columns;
# float4 stores along columns, along rows (innermost, J % 4 == 0) and scalars.
SHAPES = [((64, 48, 256), 0, 20), ((64, 48, 256), 1, 50), ((64, 48, 256), 2, 130), ((64, 48, 256), 2, 33),
          ((7, 33, 9, 5), 0, 7), ((7, 33, 9, 5), 1, 64), ((7, 33, 9, 5), 2, 9), ((7, 33, 9, 5), 3, 200),
          ((300, 257), 0, 300), ((300, 257), 1, 257), ((1000,), 0, 3), ((16, 16, 16, 16, 16), 2, 16),
          ((3, 1, 5), 1, 4)]


@pytest.mark.parametrize("dims,mode,J", SHAPES)
def test_ttm_matches_oracle(dims, mode, J):
    X, M = case(sum(dims) + 7 * mode + J, dims, mode, J)
    T = mk.ttm(torch.from_numpy(X).cuda(), mode, torch.from_numpy(M).cuda(), path="simt")
    assert tuple(T.shape) == tuple(dims[:mode]) + (J,) + tuple(dims[mode + 1:])
    check(T.cpu().numpy(), X, mode, M)


# shapes the tensor-core path takes: the innermost mode read K-major (row tail
# P = 130), other modes MN-major with Q = 64, 512 and 8192, a half tile past the
# last (p, q) row, contraction lengths 32, 40, 96, 128, 256 (padded to 64), J from
# 32 (64-column tiles) to 300 (128- and 256-column tiles, ragged)
TC_SHAPES = [((64, 48, 256), 2, 130), ((64, 48, 256), 2, 33), ((64, 128, 64), 1, 50), ((32, 64, 128), 0, 100),
             ((16, 40, 8, 64), 1, 300), ((130, 96), 1, 200), ((3, 200, 64), 1, 64), ((2, 128, 40, 128), 2, 256),
             # several row tiles a CTA (the kernel walks row tiles persistently), column
             # and row tails
             ((300, 64, 64), 1, 600), ((8000, 96), 1, 520)]


@pytest.mark.parametrize("dims,mode,J", TC_SHAPES)
def test_ttm_tensor_cores_match_oracle(dims, mode, J):
    assert mk.ttm_workspace_bytes(dims, mode, J) > 0
    X, M = case(5 + sum(dims) + 7 * mode + J, dims, mode, J)
    T = mk.ttm(torch.from_numpy(X).cuda(), mode, torch.from_numpy(M).cuda(), path="tc")
    check(T.cpu().numpy(), X, mode, M, tc=True)
    assert mk.device_status() == 0


def test_ttm_paths_agree_and_tc_is_deterministic():
    dims, mode, J = (32, 64, 128), 1, 96
    X, M = case(77, dims, mode, J)
    Xd, Md = torch.from_numpy(X).cuda(), torch.from_numpy(M).cuda()
    a = mk.ttm(Xd, mode, Md, path="tc")
    b = mk.ttm(Xd, mode, Md, path="tc")
    c = mk.ttm(Xd, mode, Md, path="simt")
    assert torch.equal(a, b)
    assert rel_fro(a.cpu().numpy(), c.cpu().numpy().astype(np.float64)) <= 2e-5
    with pytest.raises(mk.MttkrpError):
        mk.ttm(torch.zeros((5, 7, 3), device="cuda"), 1, torch.zeros((40, 7), device="cuda"), path="tc")


def test_tucker_reconstruction_chain_and_repeatability():
    """Core x_0 U_0 x_1 U_1 x_2 U_2 (the full-tensor reconstruction of the
    Jacobi page's Tucker setting), each product on the previous result."""
    rng = np.random.default_rng(31)
    core = rng.standard_normal((12, 10, 8)).astype(np.float32)
    Us = [rng.standard_normal((n, r)).astype(np.float32) for n, r in ((40, 12), (36, 10), (44, 8))]
    cur_d = torch.from_numpy(core).cuda()
    cur_h = core
    for k, Uk in enumerate(Us):
        cur_d = mk.ttm(cur_d, k, torch.from_numpy(Uk).cuda(), path="simt")
        got = cur_d.cpu().numpy()
        check(got, cur_h, k, Uk)
        cur_h = got                              # next step from the GPU's fp32 result
    again = torch.from_numpy(core).cuda()
    for k, Uk in enumerate(Us):
        again = mk.ttm(again, k, torch.from_numpy(Uk).cuda(), path="simt")
    assert torch.equal(again, cur_d)


@pytest.mark.parametrize("path", ["simt", "tc"])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_full_size_sampled(mode, path):
    """512^3 with a square 512 x 512 matrix (the bench's launch
    configuration), checked on 2000 sampled outputs computed one by one."""
    rng = np.random.default_rng(40 + mode)
    dims = (512, 512, 512)
    Xd = torch.randn(dims, generator=torch.Generator().manual_seed(41 + mode)).cuda()
    M = rng.standard_normal((512, 512)).astype(np.float32)
    T = mk.ttm(Xd, mode, torch.from_numpy(M).cuda(), path=path)
    idx = [rng.integers(0, 512, 2000) for _ in range(3)]
    got = T[idx[0], idx[1], idx[2]].cpu().numpy().astype(np.float64)
    X = Xd.cpu().numpy()
    want = np.empty(2000)
    bound = np.empty(2000)
    for s in range(2000):
        at = [int(idx[0][s]), int(idx[1][s]), int(idx[2][s])]
        j = at[mode]
        at[mode] = slice(None)
        x = X[tuple(at)].astype(np.float64)   # the fibre along `mode`
        want[s] = x @ M[j].astype(np.float64)
        bound[s] = np.abs(x) @ np.abs(M[j]).astype(np.float64)
    if path == "simt":
        assert np.all(np.abs(got - want) <= 512 * U / (1 - 512 * U) * bound + 1e-30)
    else:
        floor = 2.0 ** -36 * 512 * float(np.abs(X).max()) * float(np.abs(M).max())
        assert np.all(np.abs(got - want) <= tc_coefficient(512) * bound + floor)
    assert mk.device_status() == 0
    del T, Xd
    torch.cuda.empty_cache()


def test_out_buffer_and_rejects_bad_arguments():
    X = torch.randn((8, 6, 4), device="cuda")
    M = torch.randn((6, 6), device="cuda")
    out = torch.empty((8, 6, 4), device="cuda")
    assert mk.ttm(X, 1, M, out=out) is out
    with pytest.raises(mk.MttkrpError):
        mk.ttm(X, 1, M, out=X)                   # the result may not overlap X
    with pytest.raises(ValueError):
        mk.ttm(X, 1, torch.randn((6, 5), device="cuda"))   # M has 5 columns, mode 1 has 6
    with pytest.raises(ValueError):
        mk.ttm(X, 3, M)                          # mode out of range
    with pytest.raises(mk.MttkrpError):
        mk.ttm(X, 1, torch.empty((0, 6), device="cuda"))   # J = 0


def test_ttm_multi_matches_single_products_bitwise():
    """Several products of one X (mttkrp_ttm_multi): the tensor-core products
    share one image pass and must equal the single-product calls bit for bit
    (same images, same kernels); a product the tensor cores do not take (J = 8)
    runs on the CUDA cores, placed first so that the image pass follows it."""
    dims = (32, 64, 128)
    rng = np.random.default_rng(501)
    X = rng.standard_normal(dims).astype(np.float32)
    spec = [(1, 8), (0, 96), (1, 64), (2, 130), (1, 300)]
    Ms = [rng.standard_normal((J, dims[m])).astype(np.float32) for m, J in spec]
    Xd = torch.from_numpy(X).cuda()
    Md = [torch.from_numpy(M).cuda() for M in Ms]
    outs = mk.ttm_multi(Xd, [m for m, _ in spec], Md)
    for (m, J), M, T, Mt in zip(spec, Ms, outs, Md):
        single = mk.ttm(Xd, m, Mt, path="tc" if J >= 32 else "simt")
        assert torch.equal(T, single), (m, J)
        check(T.cpu().numpy(), X, m, M, tc=J >= 32)
    assert mk.device_status() == 0
    simt = mk.ttm_multi(Xd, [m for m, _ in spec], Md, path="simt")
    for (m, _), M, T, Mt in zip(spec, Ms, simt, Md):
        assert torch.equal(T, mk.ttm(Xd, m, Mt, path="simt"))


def test_ttm_multi_scaled_tensor_and_outs():
    """Values far from 1 (the shared images carry one power-of-two scale) and
    caller-given result buffers."""
    dims = (64, 128, 64)
    rng = np.random.default_rng(502)
    X = (rng.standard_normal(dims) * 3e5).astype(np.float32)
    X[5, 7, 9] = 4e7                                 # one outlier sets the scale
    Ms = [rng.standard_normal((n, n)).astype(np.float32) * 1e-3 for n in dims]   # square: T_k has X's shape
    Xd = torch.from_numpy(X).cuda()
    outs = [torch.empty(dims, device="cuda") for _ in range(3)]
    got = mk.ttm_multi(Xd, (0, 1, 2), [torch.from_numpy(M).cuda() for M in Ms], outs=outs, path="tc")
    for k in range(3):
        assert got[k] is outs[k]
        check(outs[k].cpu().numpy(), X, k, Ms[k], tc=True)
    assert mk.device_status() == 0


def test_ttm_multi_full_size_sampled():
    """512^3 with square 512 x 512 matrices for all three modes in one call (the
    bench's launch configuration), 600 sampled outputs a mode."""
    rng = np.random.default_rng(503)
    dims = (512, 512, 512)
    Xd = torch.randn(dims, generator=torch.Generator().manual_seed(504)).cuda()
    Ms = [rng.standard_normal((512, 512)).astype(np.float32) for _ in range(3)]
    outs = mk.ttm_multi(Xd, (0, 1, 2), [torch.from_numpy(M).cuda() for M in Ms])
    X = Xd.cpu().numpy()
    floor = 2.0 ** -36 * 512 * float(np.abs(X).max()) * max(float(np.abs(M).max()) for M in Ms)
    for mode in range(3):
        idx = [rng.integers(0, 512, 600) for _ in range(3)]
        got = outs[mode][idx[0], idx[1], idx[2]].cpu().numpy().astype(np.float64)
        for s in range(600):
            at = [int(idx[0][s]), int(idx[1][s]), int(idx[2][s])]
            j = at[mode]
            at[mode] = slice(None)
            x = X[tuple(at)].astype(np.float64)
            want = x @ Ms[mode][j].astype(np.float64)
            bound = np.abs(x) @ np.abs(Ms[mode][j]).astype(np.float64)
            assert abs(got[s] - want) <= tc_coefficient(512) * bound + floor
    assert mk.device_status() == 0
    del outs, Xd
    torch.cuda.empty_cache()


def test_ttm_multi_rejects_bad_arguments():
    X = torch.randn((32, 64, 128), device="cuda")
    M0, M1 = torch.randn((64, 32), device="cuda"), torch.randn((64, 64), device="cuda")
    shared = torch.empty((32, 64, 128), device="cuda")
    with pytest.raises(mk.MttkrpError):     # two results in one buffer
        mk.ttm_multi(X, (1, 1), (M1, M1), outs=(shared, shared))
    with pytest.raises(mk.MttkrpError):     # J = 8 is not taken by the tensor cores
        mk.ttm_multi(X, (0, 1), (M0, torch.randn((8, 64), device="cuda")), path="tc")
    with pytest.raises(ValueError):
        mk.ttm_multi(X, (0, 1), (M1, M1))   # M for mode 0 has 64 columns, mode 0 has 32
    with pytest.raises(ValueError):
        mk.ttm_multi(X, (), ())
    assert mk.device_status() == 0
