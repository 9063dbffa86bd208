"""The seeded input generator: reference vectors, determinism, distributions."""
import os
import subprocess
import sys

import numpy as np

import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def test_splitmix64_reference_sequence():
    want = [int(l, 16) for l in open(os.path.join(HERE, "golden", "splitmix64_seed0.txt"))
            if l.strip() and not l.startswith("#")]
    assert synth.splitmix_sequence(0, 3) == want


def test_draws_are_pure_functions_of_seed_stream_index():
    a = synth.uniform(5, 3, (1000,), 0.0, 1.0)
    b = synth.uniform(5, 3, (1000,), 0.0, 1.0)
    c = synth.uniform(5, 4, (1000,), 0.0, 1.0)
    np.testing.assert_array_equal(a, b)
    assert not np.array_equal(a, c)
    # a prefix of a longer draw is the shorter draw
    np.testing.assert_array_equal(synth.uniform(5, 3, (10,), 0.0, 1.0), a[:10])


def test_distributions():
    u = synth.uniform(1, 0, (200000,), -1.0, 1.0, dtype=np.float64)
    assert u.min() >= -1.0 and u.max() < 1.0
    assert abs(u.mean()) < 0.01 and abs(u.var() - 1 / 3) < 0.01
    z = synth.normal(1, 1, (200000,), 2.0, 0.5, dtype=np.float64)
    assert abs(z.mean() - 2.0) < 0.01 and abs(z.std() - 0.5) < 0.01


def test_thread_count_independence():
    code = ("import synth, sys; import numpy as np;"
            "y = synth.make_tensor(synth.Workload(2, 'x', (9, 8, 7), 3, ''));"
            "sys.stdout.write(y.tobytes().hex())")
    root = os.path.dirname(HERE)
    outs = [subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True,
                           text=True, check=True,
                           env=dict(os.environ, OMP_NUM_THREADS=nt, PYTHONPATH=root)).stdout
            for nt in ("1", "5")]
    assert outs[0] == outs[1]


def test_rank_sum_matches_definition():
    B = [synth.normal(3, 16 + n, (d, 4), 0.0, 1.0, dtype=np.float64)
         for n, d in enumerate((3, 4, 5))]
    Y = synth.rank_sum(B, dtype=np.float64)
    ref = np.einsum("is,js,ks->ijk", *B)
    np.testing.assert_allclose(Y, ref, rtol=1e-13, atol=1e-13)


def test_workload_table():
    assert [synth.workload(i).dims for i in range(1, 6)] == [
        (32, 32, 32), (256, 256, 256), (128,) * 4, (512,) * 3, (20,) * 6]
    assert [synth.workload(i).R for i in range(1, 6)] == [8, 64, 256, 2000, 128]
    w = synth.workload(1)
    Y = synth.make_tensor(w)
    A = synth.make_factors(w)
    assert Y.dtype == np.float32 and Y.shape == w.dims
    assert Y.min() >= -1 and Y.max() <= 1
    assert all(a.shape == (32, 8) and a.min() >= 0 and a.max() <= 1 for a in A)
    assert w.flops_per_mode() == 2 * 8 * 32 ** 3
