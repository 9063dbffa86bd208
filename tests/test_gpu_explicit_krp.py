"""The matrix-based comparison variant (MTTKRP_PATH_TC_EXPLICIT_KRP) against the
fp64 oracle.

"A Performance Portable Matrix Free Dense MTTKRP in GenTen" (abstract; Fig. 3
caption) contrasts its matrix-free kernel with the matrix-multiply formulation
that forms the Khatri-Rao product explicitly.  This variant does that on the
GPU: the Khatri-Rao product of every mode but k is written into the workspace
(as the B operand images of the tensor-core kernels) and Y_(k) is multiplied
by it, with the contraction split over B chunks.  Same tolerance as every
other parity test: relative Frobenius error <= 1e-5 per mode.
"""
import numpy as np
import pytest

import oracle
import synth
from conftest import rel_fro

torch = pytest.importorskip("torch")
import dense_tensor_decomposition_gb300 as mk  # noqa: E402

pytestmark = pytest.mark.gpu
TOL = 1e-5


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def explicit_plan(dims, R):
    try:
        return mk.Plan(dims, R, "tc_explicit_krp")
    except mk.MttkrpError as e:
        if e.code == 2:
            pytest.skip(f"the explicit variant does not take {dims}")
        raise


def fields(plan, k):
    return dict(t.split("=", 1) for t in plan.describe(k).split() if "=" in t)


@pytest.mark.parametrize("index", [2, 5])
def test_workload_every_mode(index):
    w = synth.workload(index)
    Y, A = synth.make_tensor(w), synth.make_factors(w)
    plan = explicit_plan(w.dims, w.R)
    outs = plan.all_modes(dev(Y), [dev(a) for a in A])
    torch.cuda.synchronize()
    for k in range(w.d):
        f = fields(plan, k)
        assert f["krp"] == "explicit" and int(f["splits"]) > 1
        got = outs[k].cpu().numpy()
        if w.numel <= 1 << 24:
            err = rel_fro(got, oracle.mttkrp(Y, A, k))
        else:
            rows = sorted({0, w.dims[k] - 1, w.dims[k] // 2, 3, 11})
            err = rel_fro(got[rows], oracle.mttkrp(Y, A, k, rows=rows))
        assert err <= TOL, f"{w.name} mode {k} ({f['kernel']}): {err:.3e}"
    assert mk.device_status() == 0


# row, column and contraction tails; K-major modes with p- and q-side modes in
# the product; the innermost mode from the transposed images; the 3xTF32
# kernel where the fp16 images do not apply (short q-blocks)
SHAPES = [((256, 12, 16, 8), 96), ((136, 24, 120), 260), ((200, 96, 64), 300), ((24, 120, 200), 300),
          ((64, 8, 8, 150), 200), ((10, 128, 130), 256), ((128, 1, 128), 32), ((96, 20, 8, 20), 64),
          ((300, 200), 48)]


@pytest.mark.parametrize("dims,R", SHAPES)
def test_shapes_every_mode(dims, R):
    Y, A = synth.random_case(4100 + sum(dims) + R, dims, R)
    plan = explicit_plan(dims, R)
    outs = plan.all_modes(dev(Y), [dev(a) for a in A])
    torch.cuda.synchronize()
    for k in range(len(dims)):
        err = rel_fro(outs[k].cpu().numpy(), oracle.mttkrp(Y, A, k))
        assert err <= TOL, f"{dims} R={R} mode {k} ({fields(plan, k)['kernel']}): {err:.3e}"
    assert mk.device_status() == 0


def test_same_result_as_matrix_free_and_deterministic():
    dims, R = (136, 24, 120), 260
    Y, A = synth.random_case(4242, dims, R)
    Yd, Ad = dev(Y), [dev(a) for a in A]
    ex = explicit_plan(dims, R)
    a = [o.clone() for o in ex.all_modes(Yd, Ad)]
    b = ex.all_modes(Yd, Ad)
    free = mk.Plan(dims, R).all_modes(Yd, Ad)
    for k in range(3):
        assert torch.equal(a[k], b[k])
        assert rel_fro(a[k].cpu().numpy(), free[k].cpu().numpy().astype(np.float64)) <= 2 * TOL
