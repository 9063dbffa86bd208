"""fp64 reference oracle for dense MTTKRP (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library never imports it, and
it imports nothing from the GPU library.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP); this module only
compiles it with gcc and marshals numpy arrays to it.  What it computes is the
definition of the matricized tensor times Khatri-Rao product of "A Performance
Portable Matrix Free Dense MTTKRP in GenTen" (abstract):

    M_k(i, r) = sum_{(i_n), n != k} Y(i_0..i_{d-1}) prod_{n != k} A_n(i_n, r).

Pins (``tests/test_oracle_pins.py``): brute force against an explicitly formed
Khatri-Rao matrix, the closed form for exact rank-S tensors, mode-permutation
invariance, and special cases that reduce to a matrix product, marginal sums,
fibres of Y and exact scaling.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c (gcc -O3 -fopenmp -ffp-contract=off) into an in-tree library."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O3", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            lib.oracle_mttkrp_naive.argtypes = [ci, vp, i64, vp, vp, ci, vp]
            lib.oracle_mttkrp_naive.restype = ci
            lib.oracle_mttkrp.argtypes = [ci, vp, i64, vp, ci, vp, ci, vp, i64, vp]
            lib.oracle_mttkrp.restype = ci
            lib.oracle_threads.argtypes = []
            lib.oracle_threads.restype = ci
            _lib = lib
    return _lib


def _prep(Y, factors):
    Y = np.asarray(Y)
    if Y.dtype not in (np.float32, np.float64):
        raise TypeError("Y must be float32 or float64")
    Y = np.ascontiguousarray(Y)
    d = Y.ndim
    if len(factors) != d:
        raise ValueError("need one factor per mode")
    A = [np.ascontiguousarray(np.asarray(a, dtype=np.float64)) for a in factors]
    R = A[0].shape[1]
    for n, a in enumerate(A):
        if a.shape != (Y.shape[n], R):
            raise ValueError(f"factor {n} has shape {a.shape}, expected {(Y.shape[n], R)}")
    dims = np.array(Y.shape, dtype=np.int64)
    return Y, A, dims, R


def _check_mode(Y, k):
    if not 0 <= k < Y.ndim:
        raise ValueError(f"mode {k} out of range for a {Y.ndim}-way tensor")


def mttkrp(Y, factors, k: int, rows=None) -> np.ndarray:
    """fp64 MTTKRP of mode k (all rows, or only the listed rows i_k)."""
    Y, A, dims, R = _prep(Y, factors)
    _check_mode(Y, k)
    ptrs = (ctypes.c_void_p * len(A))(*[a.ctypes.data for a in A])
    if rows is None:
        out = np.empty((Y.shape[k], R), dtype=np.float64)
        rp, nrows = None, Y.shape[k]
    else:
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        out = np.empty((rows.size, R), dtype=np.float64)
        rp, nrows = rows.ctypes.data, rows.size
    rc = _load().oracle_mttkrp(Y.ndim, dims.ctypes.data, R, Y.ctypes.data,
                               int(Y.dtype == np.float64), ptrs, k, rp, nrows,
                               out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_mttkrp failed ({rc})")
    return out


def mttkrp_naive(Y, factors, k: int) -> np.ndarray:
    """fp64 MTTKRP by the element-at-a-time definition (tiny inputs only)."""
    Y, A, dims, R = _prep(Y, factors)
    _check_mode(Y, k)
    Y = np.ascontiguousarray(Y, dtype=np.float64)
    ptrs = (ctypes.c_void_p * len(A))(*[a.ctypes.data for a in A])
    out = np.empty((Y.shape[k], R), dtype=np.float64)
    rc = _load().oracle_mttkrp_naive(Y.ndim, dims.ctypes.data, R, Y.ctypes.data, ptrs, k,
                                     out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_mttkrp_naive failed ({rc})")
    return out


def threads() -> int:
    return int(_load().oracle_threads())
