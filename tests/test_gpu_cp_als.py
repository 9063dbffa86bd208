"""GPU CP-ALS sweeps (mttkrp_cp_als_sweep through the C ABI) against the fp64
oracle sweep on the same seeded inputs.

Tolerances: the factors are stored in fp32 and the MTTKRP is fp32-accurate
(measured errors about 1e-6 relative Frobenius, bounded by 1e-5); the normal
equations A_n V = M are solved to fp64 accuracy (fp32 factor of V plus one
refinement step with a residual carried to about 2^-46), so an update's
relative error is about cond(V) times the error of M.  The tests compute
cond(V) of every update of the sweep from the oracle's own factors and check
that cond(V) x 2e-6 stays within the 1e-4 relative Frobenius tolerance they
apply per factor (1e-4 relative on lambda, 1e-5 absolute on the fit).
"""
import numpy as np
import pytest

import synth
from conftest import rel_fro
from oracle import cp_als as ocp

torch = pytest.importorskip("torch")
import dense_tensor_decomposition_gb300 as mk  # noqa: E402

pytestmark = pytest.mark.gpu


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def start(seed, dims, R):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((n, R)).astype(np.float32) for n in dims]


def sweep_conditions(A0, A1):
    """cond(V) of each update of one sweep: V_n = Hadamard of the Grams of the
    updated factors of the modes before n and the starting factors after n."""
    d = len(A0)
    conds = []
    for n in range(d):
        V = np.ones((A0[0].shape[1],) * 2)
        for m in range(d):
            if m != n:
                a = np.asarray(A1[m] if m < n else A0[m], dtype=np.float64)
                V *= a.T @ a
        conds.append(float(np.linalg.cond(V)))
    return conds


@pytest.mark.parametrize("dims,R", [((40, 36, 50), 12), ((130, 140, 150), 128), ((20, 24, 18, 22), 16),
                                    ((150, 160, 170), 100), ((300, 310, 320), 256),
                                    ((300, 290, 310), 288), ((330, 320, 310), 300)])
def test_one_sweep_matches_oracle(dims, R):
    Y, _ = synth.random_case(70 + R, dims, R)
    A0 = start(80 + R, dims, R)
    plan = mk.Plan(dims, R)
    Ad = [dev(a) for a in A0]
    lam, fits = plan.cp_als(dev(Y), Ad, sweeps=1)
    torch.cuda.synchronize()
    A1, lam1, fit1, _ = ocp.cp_als_sweep(Y, A0)
    conds = sweep_conditions(A0, A1)
    assert max(conds) * 2e-6 <= 1e-4, conds
    for n in range(len(dims)):
        assert rel_fro(Ad[n].cpu().numpy(), A1[n]) <= 1e-4, (n, conds)
    assert rel_fro(lam.cpu().numpy(), lam1) <= 1e-4
    assert abs(float(fits[0]) - fit1) <= 1e-5


def test_sweeps_track_the_oracle_on_a_low_rank_tensor():
    dims, R = (60, 70, 80), 5
    rng = np.random.default_rng(11)
    truth = [rng.standard_normal((n, R)) for n in dims]
    Y = ocp.reconstruct(truth, np.ones(R)) + 1e-3 * rng.standard_normal(dims)
    Y = Y.astype(np.float32)
    A0 = start(12, dims, R)
    plan = mk.Plan(dims, R)
    Ad = [dev(a) for a in A0]
    _, fits = plan.cp_als(dev(Y), Ad, sweeps=12)
    fits = fits.cpu().numpy()
    A = [a.astype(np.float64) for a in A0]
    ref = []
    for _ in range(12):
        A, _, fit, _ = ocp.cp_als_sweep(Y, A)
        ref.append(fit)
    assert np.allclose(fits, ref, atol=1e-4), (fits, ref)
    assert fits[-1] > 0.999


def test_bitwise_reproducible():
    dims, R = (40, 36, 50), 12
    Y, _ = synth.random_case(90, dims, R)
    A0 = start(91, dims, R)
    plan = mk.Plan(dims, R)
    runs = []
    for _ in range(2):
        Ad = [dev(a) for a in A0]
        lam, fits = plan.cp_als(dev(Y), Ad, sweeps=3)
        runs.append(([a.cpu().numpy() for a in Ad], lam.cpu().numpy(), fits.cpu().numpy()))
    for x, y in zip(runs[0][0], runs[1][0]):
        assert np.array_equal(x, y)
    assert np.array_equal(runs[0][1], runs[1][1]) and np.array_equal(runs[0][2], runs[1][2])


def test_singular_normal_equations_report_nan_fit():
    """A column that is zero in two factors makes V singular for the third mode's
    update: the Cholesky reports it and the fit is NaN (no fault, no hang)."""
    dims, R = (30, 32, 34), 6
    Y, _ = synth.random_case(95, dims, R)
    A0 = start(96, dims, R)
    A0[1][:, 2] = 0.0
    A0[2][:, 2] = 0.0
    plan = mk.Plan(dims, R)
    _, fits = plan.cp_als(dev(Y), [dev(a) for a in A0], sweeps=1)
    assert np.isnan(float(fits[0]))
    assert mk.device_status() == 0


def test_continuing_sweeps_reuse_images_without_changing_results():
    """Sweeps after the first in one cp_als call reuse max |Y| and the fp16
    images of Y (fp16-image modes); the results equal one-sweep calls that
    recompute them."""
    dims, R = (136, 130, 128), 128
    Y, _ = synth.random_case(97, dims, R)
    A0 = start(98, dims, R)
    plan = mk.Plan(dims, R)
    assert any("tc_fp16_image=1" in plan.describe(k) for k in range(3))
    Yd = dev(Y)
    Ad = [dev(a) for a in A0]
    lam_a, fits_a = plan.cp_als(Yd, Ad, sweeps=3)
    Bd = [dev(a) for a in A0]
    fits_b = []
    for _ in range(3):
        lam_b, f = plan.cp_als(Yd, Bd, sweeps=1)
        fits_b.append(float(f[0]))
    for x, y in zip(Ad, Bd):
        assert torch.equal(x, y)
    assert torch.equal(lam_a, lam_b)
    assert list(fits_a.cpu().numpy()) == fits_b
