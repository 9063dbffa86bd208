"""GPU parity: the CUDA paths against the fp64 oracle on the same seeded inputs.

Every comparison is element by element in relative Frobenius norm,
||M_gpu - M_oracle||_F / ||M_oracle||_F <= 1e-5 per mode per path (the
tolerance of the MTTKRP workloads; fp32 inputs, fp32 output).  Full-size
workloads are compared on sampled output rows that the oracle computes one by
one, plus (for the two structured workloads) against the closed form
M_k = B_k (*)_{n != k} (B_n^T A_n) of an exact rank-S tensor at full size.
All calls go through the C ABI (the ctypes binding).
"""
import functools

import numpy as np
import pytest

import oracle
import synth
from conftest import rel_fro
from parity_shapes import EDGE, H2_SHAPES

torch = pytest.importorskip("torch")
import dense_tensor_decomposition_gb300 as mk  # noqa: E402

pytestmark = pytest.mark.gpu
TOL = 1e-5


def available_paths():
    paths = ["simt"]
    for path in ("tc", "tc_tf32"):
        try:
            p = mk.Plan((64, 64, 64), 64)
            p.set_path(path)
            paths.append(path)
        except mk.MttkrpError:
            pass
    return paths


PATHS = available_paths() if torch.cuda.is_available() else ["simt"]


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def make_plan(dims, R, path):
    """Plan on the given path; skip the test if that path does not take the shape
    (the tensor-core path needs 16-byte multiples for the strides its tensor
    map uses)."""
    try:
        return mk.Plan(dims, R, path)
    except mk.MttkrpError as e:
        if e.code == 2 and path != "simt":
            pytest.skip(f"{path} does not take {dims}")
        raise


def gpu_modes(Y, A, path, modes=None, plan=None):
    Yd = dev(Y)
    Ad = [dev(a) for a in A]
    if plan is None:
        plan = make_plan(Y.shape, A[0].shape[1], path)
    modes = range(Y.ndim) if modes is None else modes
    outs = {k: plan.mttkrp(Yd, Ad, k).cpu().numpy() for k in modes}
    torch.cuda.synchronize()
    return outs


def sample_rows(I, seed, n=8):
    rng = np.random.default_rng(seed)
    rows = {0, I - 1, I // 2}
    rows.update(int(x) for x in rng.integers(0, I, size=n))
    return sorted(rows)


@functools.lru_cache(maxsize=1)
def workload_inputs(index, noise=True):
    w = synth.workload(index)
    return w, synth.make_tensor(w, noise=noise), synth.make_factors(w)


# ---------------------------------------------------------------------------
# the five workloads, every mode, every path
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_workload_parity(index, path):
    w, Y, A = workload_inputs(index)
    got = gpu_modes(Y, A, path)
    for k in range(w.d):
        if w.numel <= 1 << 24:
            ref = oracle.mttkrp(Y, A, k)
            err = rel_fro(got[k], ref)
        else:
            rows = sample_rows(w.dims[k], seed=k)
            ref = oracle.mttkrp(Y, A, k, rows=rows)
            err = rel_fro(got[k][rows], ref)
        assert err <= TOL, f"{w.name} mode {k} path {path}: rel err {err:.3e}"


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("index", [2, 4])
def test_closed_form_full_size(index, path):
    """Noise-free structured workloads are exact rank-S tensors: full-size check."""
    w, Y, A = workload_inputs(index, noise=False)
    B = synth.generating_factors(w)
    got = gpu_modes(Y, A, path)
    for k in range(w.d):
        H = np.ones((B[0].shape[1], w.R))
        for n in range(w.d):
            if n != k:
                H *= B[n].T @ A[n].astype(np.float64)
        ref = B[k] @ H
        err = rel_fro(got[k], ref)
        assert err <= TOL, f"{w.name} (noise-free) mode {k} path {path}: {err:.3e}"


# ---------------------------------------------------------------------------
# shapes with tails in every dimension and the degenerate cases
# ---------------------------------------------------------------------------



@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dims,R", EDGE)
def test_edge_shapes(dims, R, path):
    Y, A = synth.random_case(300 + sum(dims) + R, dims, R)
    got = gpu_modes(Y, A, path)
    for k in range(len(dims)):
        err = rel_fro(got[k], oracle.mttkrp(Y, A, k))
        assert err <= TOL, f"{dims} R={R} mode {k} path {path}: {err:.3e}"


@pytest.mark.parametrize("path", PATHS)
def test_mode_permutation_invariance(path):
    dims, R = (7, 12, 36, 5), 37
    Y, A = synth.random_case(41, dims, R)
    base = gpu_modes(Y, A, path)
    perm = [2, 0, 3, 1]
    Yp = np.ascontiguousarray(np.transpose(Y, perm))
    Ap = [A[p] for p in perm]
    got = gpu_modes(Yp, Ap, path)
    for t in range(4):
        assert rel_fro(got[t], base[perm[t]]) <= TOL


def test_order_two_is_matrix_product():
    Y, A = synth.random_case(42, (300, 200), 48)
    for path in PATHS:
        got = gpu_modes(Y, A, path)
        Y64 = Y.astype(np.float64)
        assert rel_fro(got[0], Y64 @ A[1].astype(np.float64)) <= TOL
        assert rel_fro(got[1], Y64.T @ A[0].astype(np.float64)) <= TOL


# ---------------------------------------------------------------------------
# pointers, buffers, determinism, errors
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("path", PATHS)
def test_misaligned_inputs_take_scalar_loads(path):
    dims, R = (24, 16, 32), 20
    Y, A = synth.random_case(43, dims, R)
    ybuf = torch.zeros(Y.size + 1, device="cuda")
    ybuf[1:] = dev(Y.ravel())
    Yd = ybuf[1:].view(dims)  # 4-byte but not 16-byte aligned
    abufs = []
    Ad = []
    for a in A:
        buf = torch.zeros(a.size + 1, device="cuda")
        buf[1:] = dev(a.ravel())
        abufs.append(buf)
        Ad.append(buf[1:].view(a.shape))
    plan = make_plan(dims, R, path)
    for k in range(3):
        out = plan.mttkrp(Yd, Ad, k).cpu().numpy()
        assert rel_fro(out, oracle.mttkrp(Y, A, k)) <= TOL


@pytest.mark.parametrize("path", PATHS)
def test_output_guard_bands(path):
    dims, R = (45, 36, 20), 19
    Y, A = synth.random_case(44, dims, R)
    Yd, Ad = dev(Y), [dev(a) for a in A]
    plan = make_plan(dims, R, path)
    for k in range(3):
        n = dims[k] * R
        buf = torch.full((n + 2048,), float("nan"), device="cuda")
        out = buf[1024:1024 + n].view(dims[k], R)
        plan.mttkrp(Yd, Ad, k, out=out)
        torch.cuda.synchronize()
        assert torch.isnan(buf[:1024]).all() and torch.isnan(buf[1024 + n:]).all()
        assert rel_fro(out.cpu().numpy(), oracle.mttkrp(Y, A, k)) <= TOL


@pytest.mark.parametrize("path", PATHS)
def test_bitwise_deterministic(path):
    w, Y, A = workload_inputs(2)
    Yd, Ad = dev(Y), [dev(a) for a in A]
    plan = make_plan(w.dims, w.R, path)
    a = [o.clone() for o in plan.all_modes(Yd, Ad)]
    b = plan.all_modes(Yd, Ad)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("path", PATHS)
def test_all_modes_matches_single_calls(path):
    dims, R = (31, 22, 17, 9), 40
    Y, A = synth.random_case(45, dims, R)
    Yd, Ad = dev(Y), [dev(a) for a in A]
    plan = make_plan(dims, R, path)
    allm = [o.clone() for o in plan.all_modes(Yd, Ad)]
    for k in range(4):
        assert torch.equal(allm[k], plan.mttkrp(Yd, Ad, k))


def test_undersized_workspace_is_an_error():
    dims, R = (64, 48, 40), 32
    Y, A = synth.random_case(46, dims, R)
    Yd, Ad = dev(Y), [dev(a) for a in A]
    plan = mk.Plan(dims, R)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    plan.set_workspace_ptr(small.data_ptr(), 256)
    with pytest.raises(mk.MttkrpError) as e:
        plan.mttkrp(Yd, Ad, 0)
    assert e.value.code == 3
    assert plan.launch_count() == 0


@pytest.mark.parametrize("path", PATHS)
def test_timing_events_and_launch_count(path):
    dims, R = (96, 80, 64), 64
    Y, A = synth.random_case(47, dims, R)
    Yd, Ad = dev(Y), [dev(a) for a in A]
    plan = make_plan(dims, R, path)
    plan.set_timing(True)
    plan.all_modes(Yd, Ad)
    plan.all_modes(Yd, Ad)
    for k in range(3):
        t = plan.kernel_times(k)
        assert len(t) == 2 and all(x > 0 for x in t)
    assert plan.launch_count() >= 2 * 3 * 2
    assert mk.device_status() == 0


# ---------------------------------------------------------------------------
# value ranges for the fp16-split tensor-core kernel (power-of-two scaling)
# ---------------------------------------------------------------------------



def h2_modes(plan, d):
    """Modes the plan runs on the fp16-split tensor-core kernel."""
    return [k for k in range(d) if "tc_fp16x2=1" in plan.describe(k)]


@pytest.mark.parametrize("dims,R", H2_SHAPES)
@pytest.mark.parametrize("yscale,ascale", [(1e30, 1e-20), (1e-30, 1e10), (1e-38, 1.0), (3.0, 1e-12)])
def test_scaled_values(dims, R, yscale, ascale):
    """Magnitudes far from 1 (fp16 alone would overflow or flush them): the
    split scales Y and each inner-table column by powers of two.  (The tf32
    kernels take the raw fp32 tile as their hi operand, so their lo terms are
    lost for values within 2^-11 of the fp32 normal range; only the modes that
    run on the fp16 split are checked here.)"""
    Y, A = synth.random_case(500 + R, dims, R)
    Y = (Y.astype(np.float64) * yscale).astype(np.float32)
    A = [(a.astype(np.float64) * ascale).astype(np.float32) for a in A]
    plan = make_plan(dims, R, "auto")
    modes = h2_modes(plan, len(dims))
    assert modes
    got = gpu_modes(Y, A, "auto", modes=modes, plan=plan)
    for k in modes:
        ref = oracle.mttkrp(Y, A, k)
        assert np.isfinite(got[k]).all()
        assert rel_fro(got[k], ref) <= TOL, f"{dims} k={k} scales {yscale},{ascale}"


@pytest.mark.parametrize("yscale,ascale", [(1e20, 1e-12), (1e-25, 1e8), (3.0, 1e-11)])
def test_scaled_values_two_pre_modes(yscale, ascale):
    """The same with two pre modes on either side of the mode: the factor-product
    table G multiplies two factor rows in fp32 on every path, so the scales are
    chosen to keep those products within the fp32 normal range (with A scaled by
    1e-20, as above, they would be about 1e-40 and lose bits to gradual
    underflow before any kernel runs)."""
    dims, R = (16, 130, 8, 64), 200
    Y, A = synth.random_case(500 + R, dims, R)
    Y = (Y.astype(np.float64) * yscale).astype(np.float32)
    A = [(a.astype(np.float64) * ascale).astype(np.float32) for a in A]
    plan = make_plan(dims, R, "auto")
    modes = h2_modes(plan, len(dims))
    assert 1 in modes
    got = gpu_modes(Y, A, "auto", modes=modes, plan=plan)
    for k in modes:
        ref = oracle.mttkrp(Y, A, k)
        assert np.isfinite(got[k]).all()
        assert rel_fro(got[k], ref) <= TOL, f"{dims} k={k} scales {yscale},{ascale}"


@pytest.mark.parametrize("dims,R", H2_SHAPES + [((16, 130, 8, 64), 200)])
def test_outlier_zero_column_and_zero_tensor(dims, R):
    Y, A = synth.random_case(600 + R, dims, R)
    Y = Y.copy()
    Y.flat[12345 % Y.size] = 1.0e6          # one outlier sets the scale of Y
    A = [a.copy() for a in A]
    for a in A:
        a[:, 7] = 0.0                        # an all-zero factor column
    got = gpu_modes(Y, A, "auto")
    for k in range(len(dims)):
        ref = oracle.mttkrp(Y, A, k)
        assert rel_fro(got[k], ref) <= TOL
        assert not got[k][:, 7].any()
    zero = gpu_modes(np.zeros_like(Y), A, "auto")
    for k in range(len(dims)):
        assert not zero[k].any()


def test_image_kernel_is_planned():
    """The fp16-image kernel takes the K-major modes of these shapes from the
    natural images (tc_fp16_image=1), the innermost mode from the natural images
    read MN-major (=3) or, for stacked small-I_k tiles and rows that are not a
    multiple of 8, from the transposed images (=2), so the edge cases above
    exercise all of these."""
    cases = {((200, 96, 64), 300): [1, 1, 0], ((16, 130, 8, 64), 200): [1, 1, 0, 0],
             ((20, 20, 20, 20, 20, 20), 128): [1, 1, 1, 1, 0, 2], ((16, 64, 40), 200): [0, 0, 2],
             ((512, 512, 512), 2000): [1, 1, 3], ((128, 128, 128, 128), 256): [1, 1, 1, 3],
             ((136, 24, 120), 260): [1, 1, 0], ((4, 8, 136, 64), 160): [0, 0, 1, 0],
             ((24, 120, 200), 300): [0, 0, 3], ((64, 8, 8, 150), 200): [0, 0, 0, 2],
             ((64, 64, 132), 256): [0, 0, 2]}
    for (dims, R), want in cases.items():
        plan = make_plan(dims, R, "auto")
        got = [int(plan.describe(k).split("tc_fp16_image=")[1].split()[0]) for k in range(len(dims))]
        assert got == want, (dims, R, got)


def test_pipelined_end_to_end_matches_device_calls():
    """all_modes_pipelined: three different problems from pinned host memory, copies
    overlapped with the computation on two buffer sets, equal (bitwise) to the
    device-resident calls."""
    dims, R = (136, 24, 120), 260
    cases = [synth.random_case(900 + t, dims, R) for t in range(3)]
    plan = make_plan(dims, R, "auto")
    want = [[m.cpu().numpy() for m in plan.all_modes(dev(Y), [dev(a) for a in A])] for Y, A in cases]
    batches = [(torch.from_numpy(Y).pin_memory(), [torch.from_numpy(a).pin_memory() for a in A],
                [torch.empty(dims[k], R).pin_memory() for k in range(len(dims))]) for Y, A in cases]
    bufs = tuple((torch.empty(dims, device="cuda"), [torch.empty(d, R, device="cuda") for d in dims],
                  [torch.empty(d, R, device="cuda") for d in dims]) for _ in range(2))
    got = plan.all_modes_pipelined(batches, bufs)
    torch.cuda.synchronize()
    for t in range(3):
        for k in range(len(dims)):
            assert np.array_equal(got[t][k].numpy(), want[t][k]), (t, k)


@pytest.mark.parametrize("path", PATHS)
def test_largest_rank(path):
    """R = 4096, the largest rank the planner is sized for (16 column tiles of
    256; the stacked small-I_k kernel with 32 of 128), every mode against the
    oracle on sampled output rows."""
    dims, R = (160, 40, 64), 4096
    Y, A = synth.random_case(4096, dims, R)
    got = gpu_modes(Y, A, path)
    for k in range(3):
        rows = sample_rows(dims[k], seed=40 + k, n=4)
        ref = oracle.mttkrp(Y, A, k, rows=rows)
        err = rel_fro(got[k][rows], ref)
        assert err <= TOL, f"R=4096 mode {k} path {path}: rel err {err:.3e}"
    assert mk.device_status() == 0
