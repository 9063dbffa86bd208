"""A tensor of more than 2^31 elements (2048 x 1025 x 1024, 8.6 GB of fp32):
every 64-bit offset the kernels and the host planner form is exercised past
the 32-bit range.  Every mode on the planner's path (fp16-image kernels; mode 1
converts Y in place and writes the images, mode 2 reads them MN-major with a
K-step tail) and on the SIMT path, and the mode-n product of mode 1 on the
tensor cores and on the CUDA cores, against fp64 values computed from slices of the same tensor: output
rows (the first, the middle, the last -- whose terms reach the end of Y) and
sampled mode-n-product outputs.  Y is drawn on the device from a seeded
generator; the checks copy only the slices they need."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
import dense_tensor_decomposition_gb300 as mk  # noqa: E402

pytestmark = pytest.mark.gpu

DIMS, R = (2048, 1025, 1024), 32
U = 2.0 ** -24


@pytest.fixture(scope="module")
def big():
    if torch.cuda.get_device_properties(0).total_memory < 40e9:
        pytest.skip("needs about 30 GB of device memory")
    g = torch.Generator(device="cuda").manual_seed(2311)
    Y = torch.randn(DIMS, generator=g, device="cuda")
    assert Y.numel() > 2 ** 31
    rng = np.random.default_rng(2312)
    A = [rng.standard_normal((n, R)).astype(np.float32) for n in DIMS]
    yield Y, A
    del Y
    torch.cuda.empty_cache()


def expected_row(Y, A, k, i):
    """M_k(i, :) in fp64 from the slice of Y with i_k = i."""
    a = [x.astype(np.float64) for x in A]
    if k == 0:
        S = Y[i].double().cpu().numpy()              # (I1, I2)
        return np.einsum("jr,jr->r", a[1], S @ a[2])
    if k == 1:
        S = Y[:, i, :].double().cpu().numpy()        # (I0, I2)
        return np.einsum("jr,jr->r", a[0], S @ a[2])
    S = Y[:, :, i].double().cpu().numpy()            # (I0, I1)
    return np.einsum("jr,jr->r", a[0], S @ a[1])


@pytest.mark.parametrize("path", ["auto", "simt"])
def test_mttkrp_past_2_31_elements(big, path):
    Y, A = big
    plan = mk.Plan(DIMS, R, path)
    if path == "auto":
        kinds = [plan.describe(k).split()[2] for k in range(3)]
        assert kinds == ["kernel=img.nat.bn64", "kernel=img.nat.bn64", "kernel=img.mn.bn64"], kinds
        assert "tc_convert=1" in plan.describe(1)
    outs = plan.all_modes(Y, [torch.from_numpy(a).cuda() for a in A])
    torch.cuda.synchronize()
    assert mk.device_status() == 0
    for k in range(3):
        n = DIMS[k]
        for i in (0, n // 2, n - 1):
            want = expected_row(Y, A, k, i)
            got = outs[k][i].double().cpu().numpy()
            err = np.linalg.norm(got - want) / np.linalg.norm(want)
            assert err <= 1e-5, f"{path} mode {k} row {i}: {err:.3e}"
    del outs, plan
    torch.cuda.empty_cache()


@pytest.mark.parametrize("path", ["tc", "simt"])
def test_mode_n_product_past_2_31_elements(big, path):
    Y, _ = big
    J, mode, N = 64, 1, DIMS[1]
    assert mk.ttm_workspace_bytes(DIMS, mode, J) > 0
    rng = np.random.default_rng(2313)
    M = rng.standard_normal((J, N)).astype(np.float32)
    T = mk.ttm(Y, mode, torch.from_numpy(M).cuda(), path=path)
    torch.cuda.synchronize()
    assert mk.device_status() == 0
    p = torch.from_numpy(np.concatenate([[DIMS[0] - 1], rng.integers(0, DIMS[0], 199)])).cuda()
    q = torch.from_numpy(np.concatenate([[DIMS[2] - 1], rng.integers(0, DIMS[2], 199)])).cuda()
    j = rng.integers(0, J, 200)
    x = Y[p, :, q].double().cpu().numpy()            # the 200 fibres along the mode, (200, N)
    got = T[p, torch.from_numpy(j).cuda(), q].double().cpu().numpy()
    want = np.einsum("sn,sn->s", x, M[j].astype(np.float64))
    bound = np.einsum("sn,sn->s", np.abs(x), np.abs(M[j]).astype(np.float64))
    if path == "tc":
        kd = min(128, -(-N // 64) * 64)
        floor = 2.0 ** -36 * N * float(Y.abs().max()) * float(np.abs(M).max())
        assert np.all(np.abs(got - want) <= (6 * kd + 24 + N) * U * bound + floor)
    else:   # one fp32 fused multiply-add chain over the N products
        assert np.all(np.abs(got - want) <= N * U / (1 - N * U) * bound + 1e-30)
    del T
    torch.cuda.empty_cache()
