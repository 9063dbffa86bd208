"""Workspace of the two MTTKRP formulations, from the planner (no GPU).

The GenTen page (abstract and TL;DR; Fig. 3 caption) compares the memory of
its matrix-free MTTKRP with the matrix-multiply one that forms the Khatri-Rao
product of the other modes explicitly: the latter needs R * prod_{n != k} I_n
numbers, the former tiles of O(R * sum_n I_n).  The planner reports that
product's fp32 bytes (krp_bytes) for every plan and splits the workspace by
purpose: split partial sums, tables (factor products and B operand images; for
the explicit variant, the whole product), and the plan-wide fp16 images of Y.
"""
import math

import pytest

mk = pytest.importorskip("dense_tensor_decomposition_gb300")

WORKLOADS = [((256, 256, 256), 64), ((128,) * 4, 256), ((512,) * 3, 2000), ((20,) * 6, 128)]


def fields(plan, k):
    return {k2: v for k2, v in (t.split("=", 1) for t in plan.describe(k).split() if "=" in t)}


@pytest.mark.parametrize("dims,R", WORKLOADS)
def test_explicit_tables_hold_the_product_matrix_free_tables_are_50x_smaller(dims, R):
    ex = mk.Plan(dims, R, "tc_explicit_krp")
    free = mk.Plan(dims, R)
    for k in range(len(dims)):
        krp = 4 * R * math.prod(dims) // dims[k]
        fe, ff = fields(ex, k), fields(free, k)
        assert int(fe["krp_bytes"]) == krp == int(ff["krp_bytes"])
        assert fe["krp"] == "explicit" and ff["krp"] == "free"
        assert int(fe["ws_tables"]) >= krp
        assert int(ff["ws_tables"]) * 50 < krp          # the page's "2 %"
        for f, plan in ((fe, ex), (ff, free)):
            parts = int(f["ws_partials"]) + int(f["ws_tables"]) + int(f["ws_images"])
            assert parts <= plan.workspace_bytes(k)


def test_images_are_the_only_tensor_sized_part_of_the_matrix_free_workspace():
    """Tables of the rank-2000 512^3 problem: a few MB; the fp16 images of Y (the
    fp16-split kernels' input) are 4 bytes an element, the size of Y."""
    dims, R = (512,) * 3, 2000
    free = mk.Plan(dims, R)
    f = fields(free, 0)
    assert int(f["ws_tables"]) < 16 << 20
    assert 4 * math.prod(dims) <= int(f["ws_images"]) <= 2 * 4 * math.prod(dims) + (1 << 20)
