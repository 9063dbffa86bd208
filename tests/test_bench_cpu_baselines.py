"""bench.py's oracle CPU-baseline legs for the rotation, mode-n product and
CP-ALS lines, on small host arrays (no GPU): units, positive rates, and a
sample that grows with the time allowed but never exceeds the tensor."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def small_case(dims=(48, 40, 36)):
    rng = np.random.default_rng(3)
    Y = rng.standard_normal(dims).astype(np.float32)
    groups = []
    for n in dims:
        G = n // 2
        pairs = rng.permutation(n)[: 2 * G].reshape(G, 2).astype(np.int32)
        phi = rng.uniform(-np.pi, np.pi, G)
        groups.append((pairs, np.cos(phi).astype(np.float32), np.sin(phi).astype(np.float32)))
    return rng, Y, groups


def test_mode_sample_cuts_along_another_mode():
    Y = np.zeros((10, 20, 30), dtype=np.float32)
    assert bench._mode_sample(Y, 1, 2 * 600).shape == (2, 20, 30)     # cut along mode 0
    assert bench._mode_sample(Y, 0, 3 * 300).shape == (10, 3, 30)     # mode 0 itself: cut along mode 1
    assert bench._mode_sample(Y, 2, 10 ** 9).shape == Y.shape          # never more than the tensor
    assert bench._mode_sample(Y, 2, 1).shape == (1, 20, 30)            # at least one index


def test_rotation_and_ttm_baselines():
    rng, Y, groups = small_case()
    rot = bench.rotations_cpu_baseline(Y, groups, 0.2)
    assert rot["unit"] == "GB/s" and rot["value"] > 0 and rot["kind"] == "oracle" and rot["cores"] == 1
    Ms = [rng.standard_normal((8, n)).astype(np.float32) for n in Y.shape]
    ttm = bench.ttm_cpu_baseline(Y, Ms, 0.2)
    assert ttm["unit"] == "TFLOP/s" and ttm["value"] > 0 and ttm["cores"] >= 1


def test_cp_als_baseline():
    rng, Y, _ = small_case()
    A0 = [rng.standard_normal((n, 4)).astype(np.float32) for n in Y.shape]
    cpu = bench.cp_als_cpu_baseline(Y, A0)
    assert cpu["unit"] == "ms" and cpu["value"] > 0 and cpu["kind"] == "oracle"
