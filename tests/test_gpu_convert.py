"""A mode converting Y in place (tc_convert=1 in the plan's description; an
all-modes call computes it first): its main kernel loads fp32 tiles of Y,
splits them into the fp16 hi and lo tiles it multiplies, and stores them as the
images that the other modes read, so no separate image pass runs.

Checks: every mode against the fp64 oracle (relative Frobenius 1e-5, as the
other parity tests); the later modes of an all-modes call, which read the
images the kernel stored, bit for bit equal to single-mode calls, which write
the images in the separate pass (so the stored images are that pass's images,
element for element); and an entry that the sampled maxima miss, which leaves
the fp16 range, so that the exact maxima, images, the mode's G table (when it
carries the slab scales) and its result are redone after the kernel."""
import numpy as np
import pytest

import oracle
from conftest import rel_fro
from parity_shapes import CONVERT_SHAPES

torch = pytest.importorskip("torch")
import dense_tensor_decomposition_gb300 as mk  # noqa: E402

pytestmark = pytest.mark.gpu
TOL = 1e-5


def inputs(dims, R, seed):
    rng = np.random.default_rng(seed)
    Y = rng.standard_normal(dims).astype(np.float32)
    A = [rng.standard_normal((n, R)).astype(np.float32) for n in dims]
    return Y, A


@pytest.mark.parametrize("dims,R,mode", CONVERT_SHAPES)
def test_converting_mode_and_stored_images(dims, R, mode):
    plan = mk.Plan(dims, R)
    assert "tc_convert=1" in plan.describe(mode)
    Y, A = inputs(dims, R, 900 + sum(dims) + R)
    Yd = torch.from_numpy(Y).cuda()
    Ad = [torch.from_numpy(a).cuda() for a in A]
    outs = plan.all_modes(Yd, Ad)
    single = [plan.mttkrp(Yd, Ad, k) for k in range(len(dims))]
    torch.cuda.synchronize()
    assert mk.device_status() == 0
    for k in range(len(dims)):
        ref = oracle.mttkrp(Y, A, k)
        assert rel_fro(outs[k].cpu().numpy(), ref) <= TOL, f"mode {k}"
        # the converting mode converts in both calls; the other modes of the
        # all-modes call read the images it stored, the single calls those of
        # the separate pass
        assert torch.equal(outs[k], single[k]), f"mode {k}"


@pytest.mark.parametrize("factor", [1e6, 3.0])
@pytest.mark.parametrize("shape", [0, 3, 7], ids=["mode0", "mode1", "bn64"])
def test_converting_mode_unsampled_outlier(factor, shape):
    """Element 1000 of slab 1 lies in a chunk the maxima sample skips: 1e6
    leaves the fp16 range once scaled (the redo runs), 3.0 stays within it."""
    dims, R, _ = CONVERT_SHAPES[shape]
    rng = np.random.default_rng(int(factor) + 17)
    Y = rng.uniform(0.5, 1.0, size=dims).astype(np.float32)
    Y.reshape(dims[0], -1)[1, 1000] *= np.float32(factor)
    A = [rng.uniform(0.0, 1.0, size=(n, R)).astype(np.float32) for n in dims]
    plan = mk.Plan(dims, R)
    Yd = torch.from_numpy(Y).cuda()
    Ad = [torch.from_numpy(a).cuda() for a in A]
    outs = plan.all_modes(Yd, Ad)
    torch.cuda.synchronize()
    assert mk.device_status() == 0
    for k in range(len(dims)):
        got = outs[k].cpu().numpy().astype(np.float64)
        ref = oracle.mttkrp(Y, A, k)
        err = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
        assert float(err.max()) <= TOL, f"factor {factor} mode {k}: worst row {err.max():.3e}"
    again = plan.mttkrp(Yd, Ad, 1)
    assert torch.equal(again, outs[1])


def test_converting_mode_repeated_calls():
    """Calls that reuse the plan: the second all-modes call converts again and
    matches the first bit for bit."""
    dims, R, _ = CONVERT_SHAPES[2]
    Y, A = inputs(dims, R, 77)   # three row tiles, 200 of 256 columns
    plan = mk.Plan(dims, R)
    Yd = torch.from_numpy(Y).cuda()
    Ad = [torch.from_numpy(a).cuda() for a in A]
    first = plan.all_modes(Yd, Ad)
    second = plan.all_modes(Yd, Ad)
    torch.cuda.synchronize()
    for a, b in zip(first, second):
        assert torch.equal(a, b)
    assert mk.device_status() == 0


def test_converting_plan_with_misaligned_tensor():
    """Y only 4-byte aligned: the tensor maps cannot address it, so every mode
    (the converting one included) runs its SIMT plan; then an aligned call on the
    same plan converts again."""
    dims, R, mode = CONVERT_SHAPES[3]
    Y, A = inputs(dims, R, 610)
    ybuf = torch.zeros(Y.size + 1, device="cuda")
    ybuf[1:] = torch.from_numpy(Y.ravel()).cuda()
    Ym = ybuf[1:].view(dims)
    Ad = [torch.from_numpy(a).cuda() for a in A]
    plan = mk.Plan(dims, R)
    assert "tc_convert=1" in plan.describe(mode)
    outs = plan.all_modes(Ym, Ad)
    aligned = plan.all_modes(torch.from_numpy(Y).cuda(), Ad)
    torch.cuda.synchronize()
    assert mk.device_status() == 0
    for k in range(len(dims)):
        ref = oracle.mttkrp(Y, A, k)
        assert rel_fro(outs[k].cpu().numpy(), ref) <= TOL, f"misaligned, mode {k}"
        assert rel_fro(aligned[k].cpu().numpy(), ref) <= TOL, f"aligned, mode {k}"
