"""Plant plausible mistakes in a copy of the oracle and check that a pin catches each.

Each mutant is the oracle's C source with one textual change (a dropped factor,
a wrong stride, a transposed operand, a lost term, a wrong sign), compiled to a
temporary library on the host.  The pins used are the ones of
test_oracle_pins.py that do not depend on the oracle: the explicit Khatri-Rao
brute force and the rank-S closed form.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

import synth
from test_oracle_pins import brute_force_krp

ORACLE_C = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "oracle", "oracle.c")

MUTANTS = {
    "drop_first_factor": ("for (int t = 0; t < m; ++t) {\n                    const double* arow",
                          "for (int t = 1; t < m; ++t) {\n                    const double* arow"),
    "sum_instead_of_product": ("w[r] *= arow[r];", "w[r] += arow[r];"),
    "wrong_stride_index": ("base += jdx[t] * stride[other[t]];", "base += jdx[t] * stride[t];"),
    "transposed_row_stride": ("int64_t off = base + i * stride[k];",
                              "int64_t off = base + i * stride[d - 1 - k];"),
    "wrong_sign": ("a[r] += y * w[r];", "a[r] -= y * w[r];"),
    "odometer_wrong_order": ("for (int t = m - 1; t >= 0; --t) {\n                    if (++jdx[t]",
                             "for (int t = 0; t < m; ++t) {\n                    if (++jdx[t]"),
    "lost_last_chunk_sum": ("for (int64_t c = 0; c < nchunk; ++c) {\n        const double* src",
                            "for (int64_t c = 0; c + 1 < nchunk; ++c) {\n        const double* src"),
}


def build_mutant(tmp_path, name):
    src = open(ORACLE_C).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path_c = tmp_path / f"{name}.c"
    path_so = tmp_path / f"{name}.so"
    path_c.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-fopenmp", "-o", str(path_so),
                    str(path_c)], check=True)
    lib = ctypes.CDLL(str(path_so))
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.oracle_mttkrp.argtypes = [ci, vp, i64, vp, ci, vp, ci, vp, i64, vp]
    lib.oracle_mttkrp.restype = ci
    return lib


def run(lib, Y, A, k):
    Y = np.ascontiguousarray(Y, dtype=np.float64)
    A = [np.ascontiguousarray(a, dtype=np.float64) for a in A]
    dims = np.array(Y.shape, dtype=np.int64)
    R = A[0].shape[1]
    out = np.zeros((Y.shape[k], R))
    ptrs = (ctypes.c_void_p * len(A))(*[a.ctypes.data for a in A])
    lib.oracle_mttkrp(Y.ndim, dims.ctypes.data, R, Y.ctypes.data, 1, ptrs, k, None,
                      Y.shape[k], out.ctypes.data)
    return out


def check_mutant(so_dir, name):
    """Runs in a child process: a mutant may read outside Y, which must not take
    the test session down with it.  Exit code 0 = caught, 3 = survived."""
    import pathlib
    lib = build_mutant(pathlib.Path(so_dir), name)
    caught = False
    # 4-way, non-cubical so that strides and index orders are all distinct;
    # a long first mode so the column range is cut into several chunks
    for dims, R in (((3, 4, 5, 2), 3), ((200, 3, 2), 5)):
        Y, A = synth.random_case(77, dims, R, dtype=np.float64)
        for k in range(len(dims)):
            ref = brute_force_krp(Y, A, k)
            got = run(lib, Y, A, k)
            if np.linalg.norm(got - ref) > 1e-10 * np.linalg.norm(ref):
                caught = True
    sys.exit(0 if caught else 3)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = (f"import sys; sys.path[:0] = [{root!r}, {os.path.join(root, 'tests')!r}];"
            f"import test_oracle_mutations as t; t.check_mutant({str(tmp_path)!r}, {name!r})")
    res = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True)
    # 3 = the mutant survived; any other non-zero status (a crash on a wild
    # read) also means the mutant is visibly wrong
    assert res.returncode != 3, f"mutant {name} survived the brute-force pin"
    if res.returncode != 0:
        assert "Traceback" not in res.stderr or "mutation anchor" not in res.stderr, res.stderr
