"""Wide value ranges on the fp16-split tensor-core kernels, every output row.

The fp16 two-term split scales Y by powers of two before rounding it to fp16
hi and lo parts.  With one scale for the whole tensor, entries far below the
tensor's largest magnitude would lose their low bits to fp16 subnormals, and
an output row built only from such entries would lose its accuracy while the
relative Frobenius error of the whole output (dominated by the large rows)
stayed small.  Y is therefore scaled per slab of mode 0.  These tests build
non-negative tensors whose halves along a mode differ by a factor of 1e9 (with
non-negative factors, so that nothing cancels) and compare EVERY output row
of every mode with the fp64 oracle, row by row, within the 1e-5 relative
tolerance of the other parity tests.

Halves along mode 0 run on the planner's own choice (the fp16-split kernels
for the modes listed).  Halves along the last mode are outside the per-slab
scaling (a slab of mode 0 then holds both halves): for such tensors the
3xTF32 kernels (path "tc_tf32") and the SIMT path keep every row accurate,
which is what the library offers for them.
"""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
import dense_tensor_decomposition_gb300 as mk  # noqa: E402

pytestmark = pytest.mark.gpu
TOL = 1e-5

# (dims, R, fp16-split kernels the planner picks for some modes)
SHAPES = [
    ((256, 96, 128), 256, {"img.nat.bn256"}),
    ((256, 64, 128), 256, {"img.nat.bn256", "img.mn.bn256"}),
    ((64, 64, 132), 256, {"img.t.bn256"}),
    ((130, 6, 7, 100), 500, {"h2.kmaj.bn224", "h2.inner.bn224"}),
    ((40, 36, 128), 450, {"img.nat.small.bn128", "h2.inner.bn224"}),
    ((48, 64, 40), 130, {"img.t.small.bn128"}),
    ((20, 3, 120), 48, {"img.nat.small.bn64"}),
]


def two_level_tensor(dims, R, axis, seed):
    """Y >= 0 (uniform in [0.5, 1)), its second half along `axis` scaled by 1e-9;
    factors uniform in [0, 1)."""
    rng = np.random.default_rng(seed)
    Y = rng.uniform(0.5, 1.0, size=dims)
    sl = [slice(None)] * len(dims)
    sl[axis] = slice(dims[axis] // 2, None)
    Y[tuple(sl)] *= 1e-9
    A = [rng.uniform(0.0, 1.0, size=(n, R)).astype(np.float32) for n in dims]
    return Y.astype(np.float32), A


def worst_row_error(got, ref):
    num = np.linalg.norm(got.astype(np.float64) - ref, axis=1)
    den = np.linalg.norm(ref, axis=1)
    assert (den > 0).all()
    return float((num / den).max())


def kernels(plan, d):
    return [plan.describe(k).split()[2][len("kernel="):] for k in range(d)]


def run(Y, A, plan):
    Yd = torch.from_numpy(Y).cuda()
    Ad = [torch.from_numpy(a).cuda() for a in A]
    outs = plan.all_modes(Yd, Ad)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in outs]


@pytest.mark.parametrize("dims,R,want", SHAPES)
def test_halves_along_mode0_every_row(dims, R, want):
    Y, A = two_level_tensor(dims, R, 0, seed=sum(dims) + R)
    plan = mk.Plan(dims, R)
    ks = kernels(plan, len(dims))
    assert want <= set(ks), ks
    got = run(Y, A, plan)
    for k in range(len(dims)):
        err = worst_row_error(got[k], oracle.mttkrp(Y, A, k))
        assert err <= TOL, f"{dims} R={R} mode {k} ({ks[k]}): worst row {err:.3e}"
    assert mk.device_status() == 0


@pytest.mark.parametrize("path", ["tc_tf32", "simt"])
@pytest.mark.parametrize("dims,R", [((256, 64, 128), 256), ((130, 6, 7, 100), 500)])
def test_halves_along_last_mode_every_row(dims, R, path):
    Y, A = two_level_tensor(dims, R, len(dims) - 1, seed=7 + R)
    plan = mk.Plan(dims, R, path)
    got = run(Y, A, plan)
    for k in range(len(dims)):
        err = worst_row_error(got[k], oracle.mttkrp(Y, A, k))
        assert err <= TOL, f"{dims} R={R} mode {k} path {path}: worst row {err:.3e}"


# Sampled maxima.  The maxima that set the fp16 scales are taken from every
# 16th chunk of 512 consecutive elements of each slab of mode 0; the image pass
# checks every scaled value and, when one leaves the fp16 range, the exact
# maxima and images are recomputed before any kernel reads them.  These tensors
# put a large entry where the sample does not look (element 1000 of a slab of
# 32768: chunk 1), so the sampled maximum is far below the true one.

@pytest.mark.parametrize("dims,R,factor,path", [
    ((4, 64, 512), 64, 1e6, "auto"),     # out of range: the exact redo runs
    ((4, 64, 512), 64, 3.0, "auto"),     # within range: kept, larger scale
    ((4, 64, 512), 256, 1e6, "auto"),
    ((64, 64, 132), 256, 1e6, "auto"),   # the transposed-image pass (img.t)
])
def test_sampled_maxima_unsampled_outlier_every_row(dims, R, factor, path):
    rng = np.random.default_rng(int(factor) + R + sum(dims))
    Y = rng.uniform(0.5, 1.0, size=dims).astype(np.float32)
    flat = Y.reshape(dims[0], -1)
    flat[1, 1000] *= np.float32(factor)
    A = [rng.uniform(0.0, 1.0, size=(n, R)).astype(np.float32) for n in dims]
    plan = mk.Plan(dims, R, path)
    assert any(k.startswith("img.") for k in kernels(plan, len(dims)))
    got = run(Y, A, plan)
    assert mk.device_status() == 0
    for k in range(len(dims)):
        err = worst_row_error(got[k], oracle.mttkrp(Y, A, k))
        assert err <= TOL, f"{dims} R={R} factor={factor} mode {k}: worst row {err:.3e}"


def test_sampled_maxima_zero_slab_and_nonfinite():
    """A slab that is all zero next to ordinary ones; then an Inf that the sample
    misses (the exact redo then takes scale 1, as the exact maxima always did)."""
    dims, R = (4, 64, 512), 64
    rng = np.random.default_rng(5)
    Y = rng.uniform(-1.0, 1.0, size=dims).astype(np.float32)
    Y[2] = 0.0
    A = [rng.uniform(-1.0, 1.0, size=(n, R)).astype(np.float32) for n in dims]
    plan = mk.Plan(dims, R)
    got = run(Y, A, plan)
    for k in range(3):
        ref = oracle.mttkrp(Y, A, k)
        assert np.linalg.norm(got[k] - ref) <= TOL * np.linalg.norm(ref)
        if k == 0:
            assert np.all(got[0][2] == 0.0)
    Y.reshape(4, -1)[1, 1000] = np.inf
    got = run(Y, A, plan)
    assert mk.device_status() == 0
    assert not np.isfinite(got[0][1]).all()     # the Inf reaches its row
    assert np.isfinite(got[0][0]).all() and np.isfinite(got[0][3]).all()
