"""Every kernel variant the planner can choose is exercised by the GPU parity tests.

The planner is host code (no GPU needed): for each (shape, path) that
tests/test_gpu_parity.py runs, it reports the kernel of every mode
(``kernel=`` in mttkrp_plan_describe).  Two checks:
  * a sweep over many random shapes and ranks finds no variant outside the
    known list (a new variant cannot appear untested);
  * each known variant is planned for at least one mode of one shape that the
    GPU parity tests run on the path that plans it.
"""
import itertools
import math
import random

import pytest

from parity_shapes import CONVERT_SHAPES, EDGE, H2_SHAPES

mk = pytest.importorskip("dense_tensor_decomposition_gb300")

# family.layout[.small].bn<columns>; families: simt, img (fp16 images of Y:
# natural, transposed, or natural read MN-major),
# h2 (fp16 split in tensor memory), tf32 (3xTF32, A in shared memory),
# tf32tm (3xTF32, A in tensor memory)
KNOWN = {
    "simt.bn64", "simt.bn128",
    "img.nat.bn64", "img.nat.bn128", "img.nat.bn256", "img.nat.small.bn64", "img.nat.small.bn128",
    "img.t.bn64", "img.t.bn128", "img.t.bn256", "img.t.small.bn64", "img.t.small.bn128",
    "img.mn.bn64", "img.mn.bn128", "img.mn.bn256",
    "h2.kmaj.bn224", "h2.inner.bn224",
    "tf32.kmaj.bn64", "tf32.kmaj.bn128", "tf32.kmaj.bn256",
    "tf32.inner.bn64", "tf32.inner.bn128", "tf32.inner.bn256",
    "tf32.kmaj.small.bn64", "tf32.kmaj.small.bn128", "tf32.kmaj.small.bn256",
    "tf32.inner.small.bn64", "tf32.inner.small.bn128", "tf32.inner.small.bn256",
    "tf32tm.inner.bn224",
}
PATHS = ("auto", "simt", "tc", "tc_tf32")

# the five workloads and the fixed shapes of the other GPU parity tests
WORKLOADS = [((32, 32, 32), 8), ((256, 256, 256), 64), ((128,) * 4, 256), ((512,) * 3, 2000),
             ((20,) * 6, 128)]
OTHER = [((7, 12, 36, 5), 37), ((300, 200), 48), ((24, 16, 32), 20), ((45, 36, 20), 19),
         ((31, 22, 17, 9), 40), ((96, 80, 64), 64), ((16, 130, 8, 64), 200)]


def kernels(dims, R, path):
    try:
        plan = mk.Plan(dims, R, path)
    except mk.MttkrpError:
        return []
    out = []
    for k in range(len(dims)):
        field = [f for f in plan.describe(k).split() if f.startswith("kernel=")]
        assert len(field) == 1
        out.append(field[0][len("kernel="):])
    return out


def test_random_shapes_plan_only_known_variants():
    rng = random.Random(2026)
    sizes = [1, 2, 3, 4, 5, 7, 8, 12, 16, 17, 20, 24, 30, 32, 33, 36, 40, 44, 48, 60, 64, 65, 96, 100,
             120, 128, 129, 130, 136, 150, 160, 200, 256, 300, 512]
    ranks = [1, 3, 8, 17, 31, 32, 33, 48, 64, 65, 96, 100, 128, 130, 159, 160, 192, 200, 224, 256, 260,
             300, 447, 448, 460, 500, 1000, 2000]
    found = set()
    for _ in range(1500):
        d = rng.randint(2, 6)
        dims = tuple(rng.choice(sizes) for _ in range(d))
        if math.prod(dims) > 1 << 28:
            continue
        R = rng.choice(ranks)
        for path in PATHS:
            found.update(kernels(dims, R, path))
    assert found <= KNOWN, sorted(found - KNOWN)


def test_every_variant_is_gpu_tested():
    """(shape, path) pairs as the GPU parity tests run them: the edge shapes and
    workloads on every forced path, the value-range shapes on the planner's own
    choice."""
    planned = {}
    for (dims, R), path in itertools.product(EDGE + WORKLOADS + OTHER, ("simt", "tc", "tc_tf32")):
        for k, v in enumerate(kernels(dims, R, path)):
            planned.setdefault(v, (dims, R, path, k))
    for dims, R in H2_SHAPES:
        for k, v in enumerate(kernels(dims, R, "auto")):
            planned.setdefault(v, (dims, R, "auto", k))
    missing = sorted(KNOWN - set(planned))
    assert not missing, f"variants no GPU parity shape plans: {missing}"


def test_headline_workload_kernels():
    """The planner's choice on the largest workload, and the 3xTF32 kernels the
    forced path takes there (the innermost mode with A in tensor memory)."""
    assert kernels((512,) * 3, 2000, "auto") == ["img.nat.bn256", "img.nat.bn256", "img.mn.bn256"]
    assert kernels((512,) * 3, 2000, "tc_tf32") == ["tf32.kmaj.bn256", "tf32.kmaj.bn256",
                                                     "tf32tm.inner.bn224"]


def test_converting_mode_is_gpu_tested():
    """The shapes tests/test_gpu_convert.py runs convert Y in the mode listed
    with them (tc_convert=1) and in no other; the 128^4 workload converts in
    mode 2 (its 128 x 128 tiles of one pre index are contiguous); no mode of the
    512^3, R = 2000 workload does (eight column tiles would each convert)."""
    for dims, R, mode in CONVERT_SHAPES + [((128,) * 4, 256, 2), ((256,) * 3, 64, 1)]:
        plan = mk.Plan(dims, R)
        flags = ["tc_convert=1" in plan.describe(k) for k in range(len(dims))]
        assert flags == [k == mode for k in range(len(dims))], (dims, R, flags)
    plan = mk.Plan((512,) * 3, 2000)
    assert not any("tc_convert=1" in plan.describe(k) for k in range(3))


def test_converting_mode_rules_on_random_shapes():
    """Over random shapes and ranks: at most one mode converts Y in place; it is a
    natural K-major image mode (kernel img.nat.bn*) with one column tile and an
    inner group of whole modes after it (J = Jq, a multiple of 64); and no plan
    with a transposed-image mode converts."""
    rng = random.Random(7)
    sizes = [2, 3, 8, 16, 20, 32, 40, 64, 96, 100, 128, 130, 200, 256, 512]
    ranks = [8, 32, 48, 64, 100, 128, 200, 256, 300, 1000]
    seen = 0
    for _ in range(800):
        d = rng.randint(2, 5)
        dims = tuple(rng.choice(sizes) for _ in range(d))
        if math.prod(dims) > 1 << 27:
            continue
        R = rng.choice(ranks)
        plan = mk.Plan(dims, R)
        descs = [dict(f.split("=", 1) for f in plan.describe(k).split() if "=" in f) for k in range(d)]
        conv = [k for k in range(d) if descs[k]["tc_convert"] == "1"]
        assert len(conv) <= 1, (dims, R, conv)
        if not conv:
            continue
        seen += 1
        k = conv[0]
        f = descs[k]
        assert f["kernel"].startswith("img.nat.bn") and ".small" not in f["kernel"], (dims, R, f["kernel"])
        bn = int(f["kernel"].split("bn")[1])
        assert -(-R // bn) == 1, (dims, R, bn)
        assert f["J"] == f["Jq"] and int(f["J"]) % 64 == 0, (dims, R, f["J"], f["Jq"])
        assert all(x["tc_fp16_image"] != "2" for x in descs), (dims, R)
    assert seen >= 20, seen
