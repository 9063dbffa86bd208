"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench.

This package holds no MTTKRP arithmetic.  It draws counter-based random numbers
(SplitMix64 of (seed, stream, index); see ``synth.c``) and, for the structured
workloads, evaluates a tensor defined as a sum of rank-one terms.  Values
depend only on (seed, stream, index), never on the thread count.

The five workloads follow the problem sizes of the dense matrix-free MTTKRP
study ("A Performance Portable Matrix Free Dense MTTKRP in GenTen", abstract:
rank up to 2000, 3-way and higher-order dense tensors).  Its real datasets
(tearing-mode and island-coalescence tensors, TL;DR and Figs. 3-5) are not
available, so seeded synthetic tensors of the stated shapes stand in for them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "_libsynth.so")
_lock = threading.Lock()
_lib = None

SEED_BASE = 20261202
# stream ids: Y = 0, factor A_n = 1 + n, generating factor B_n = 16 + n,
# additive noise = 32, bump centres = 33
STREAM_Y = 0
STREAM_NOISE = 32
STREAM_CENTRES = 33


def stream_factor(n: int) -> int:
    return 1 + n


def stream_generating_factor(n: int) -> int:
    return 16 + n


def build(force: bool = False) -> str:
    """Compile synth.c into an in-tree shared library (plain gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            u64, i64, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
            vp = ctypes.c_void_p
            lib.synth_mix64.argtypes = [u64]
            lib.synth_mix64.restype = u64
            lib.synth_splitmix_next.argtypes = [ctypes.POINTER(u64)]
            lib.synth_splitmix_next.restype = u64
            lib.synth_draw.argtypes = [u64, u64, u64]
            lib.synth_draw.restype = u64
            for name in ("synth_uniform_f32", "synth_uniform_f64",
                         "synth_normal_f32", "synth_normal_f64"):
                fn = getattr(lib, name)
                fn.argtypes = [u64, u64, i64, dbl, dbl, vp]
                fn.restype = None
            lib.synth_rank_sum.argtypes = [ctypes.c_int, vp, i64, vp, dbl, u64, u64, vp, vp]
            lib.synth_rank_sum.restype = ctypes.c_int
            _lib = lib
    return _lib


def mix64(z: int) -> int:
    return _load().synth_mix64(z)


def splitmix_sequence(state: int, n: int) -> list[int]:
    s = ctypes.c_uint64(state)
    return [_load().synth_splitmix_next(ctypes.byref(s)) for _ in range(n)]


def uniform(seed: int, stream: int, shape, lo: float, hi: float, dtype=np.float32) -> np.ndarray:
    out = np.empty(shape, dtype=dtype)
    fn = _load().synth_uniform_f32 if out.dtype == np.float32 else _load().synth_uniform_f64
    fn(seed, stream, out.size, lo, hi, out.ctypes.data)
    return out


def normal(seed: int, stream: int, shape, mean: float, std: float, dtype=np.float32) -> np.ndarray:
    out = np.empty(shape, dtype=dtype)
    fn = _load().synth_normal_f32 if out.dtype == np.float32 else _load().synth_normal_f64
    fn(seed, stream, out.size, mean, std, out.ctypes.data)
    return out


def rank_sum(B: list[np.ndarray], noise_std: float = 0.0, seed: int = 0,
             noise_stream: int = STREAM_NOISE, dtype=np.float32) -> np.ndarray:
    """Y = sum_s prod_n B_n(i_n, s) (+ N(0, noise_std)), B_n fp64 of shape I_n x S."""
    B = [np.ascontiguousarray(b, dtype=np.float64) for b in B]
    d = len(B)
    S = B[0].shape[1]
    assert all(b.ndim == 2 and b.shape[1] == S for b in B)
    dims = np.array([b.shape[0] for b in B], dtype=np.int64)
    out = np.empty(tuple(int(x) for x in dims), dtype=dtype)
    ptrs = (ctypes.c_void_p * d)(*[b.ctypes.data for b in B])
    o32 = out.ctypes.data if out.dtype == np.float32 else None
    o64 = out.ctypes.data if out.dtype == np.float64 else None
    rc = _load().synth_rank_sum(d, dims.ctypes.data, S, ptrs, noise_std, seed,
                                noise_stream, o32, o64)
    if rc != 0:
        raise ValueError("synth_rank_sum: bad arguments")
    return out


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------

class Workload:
    """One seeded MTTKRP workload: dims, rank and the recipe of Y and factors."""

    def __init__(self, index: int, name: str, dims, R: int, desc: str):
        self.index = index
        self.name = name
        self.dims = tuple(int(x) for x in dims)
        self.R = int(R)
        self.desc = desc
        self.seed = SEED_BASE + index

    @property
    def d(self) -> int:
        return len(self.dims)

    @property
    def numel(self) -> int:
        return int(np.prod(self.dims, dtype=np.int64))

    def flops_per_mode(self) -> int:
        return 2 * self.R * self.numel

    def bytes_per_mode(self, k: int) -> int:
        """Algorithmic bytes: Y once, the d-1 factors, the output (fp32)."""
        others = sum(self.dims[n] for n in range(self.d) if n != k)
        return 4 * (self.numel + self.R * others + self.dims[k] * self.R)

    def __repr__(self):
        return f"Workload({self.name}, dims={self.dims}, R={self.R})"


WORKLOADS = {
    1: Workload(1, "dense3_32cubed_r8", (32, 32, 32), 8,
                "3-way 32^3, Y ~ U[-1,1], A_n ~ U[0,1], R=8"),
    2: Workload(2, "rank10_3way_256cubed_r64", (256, 256, 256), 64,
                "3-way 256^3 = sum of 10 rank-one terms (N(0,1) columns) + N(0,0.01) noise; "
                "A_n ~ N(0, 0.125), R=64"),
    3: Workload(3, "dense4_128pow4_r256", (128, 128, 128, 128), 256,
                "4-way 128^4 (1 GiB), Y ~ N(0,1), A_n ~ U[0,1], R=256"),
    4: Workload(4, "bumps3_512cubed_r2000", (512, 512, 512), 2000,
                "3-way 512^3 (512 MiB), 32 Gaussian bumps (sigma 0.05) + N(0,1e-3) noise; "
                "A_n ~ N(0,1), R=2000"),
    5: Workload(5, "dense6_20pow6_r128", (20, 20, 20, 20, 20, 20), 128,
                "6-way 20^6 (64M), Y ~ U[-1,1], A_n ~ U[-1,1], R=128"),
}

BUMP_COUNT = 32
BUMP_SIGMA = 0.05
RANK10_TERMS = 10


def workload(key) -> Workload:
    if isinstance(key, Workload):
        return key
    if isinstance(key, int):
        return WORKLOADS[key]
    for w in WORKLOADS.values():
        if w.name == key or f"c{w.index}" == key:
            return w
    raise KeyError(key)


def generating_factors(w: Workload) -> list[np.ndarray] | None:
    """The fp64 rank-one factors B_n that define Y for the structured workloads.

    Workload 2: S = 10 columns ~ N(0,1).  Workload 4: one column per Gaussian
    bump; exp(-|x-c|^2/(2 sigma^2)) is separable over the axes, so the field
    is exactly the rank-32 tensor with B_a(i, j) = exp(-(x_i - c_{j,a})^2 /
    (2 sigma^2)), x_i = (i + 0.5)/I the cell centres of the unit cube.
    Returns None for the unstructured workloads.
    """
    if w.index == 2:
        return [normal(w.seed, stream_generating_factor(n), (w.dims[n], RANK10_TERMS),
                       0.0, 1.0, dtype=np.float64) for n in range(w.d)]
    if w.index == 4:
        centres = uniform(w.seed, STREAM_CENTRES, (BUMP_COUNT, w.d), 0.0, 1.0, dtype=np.float64)
        B = []
        for a in range(w.d):
            x = (np.arange(w.dims[a], dtype=np.float64) + 0.5) / w.dims[a]
            diff = x[:, None] - centres[None, :, a]
            B.append(np.exp(-(diff * diff) / (2.0 * BUMP_SIGMA * BUMP_SIGMA)))
        return B
    return None


def make_tensor(w: Workload, noise: bool = True, dtype=np.float32) -> np.ndarray:
    if w.index in (1, 5):
        return uniform(w.seed, STREAM_Y, w.dims, -1.0, 1.0, dtype=dtype)
    if w.index == 3:
        return normal(w.seed, STREAM_Y, w.dims, 0.0, 1.0, dtype=dtype)
    B = generating_factors(w)
    noise_std = (0.01 if w.index == 2 else 1e-3) if noise else 0.0
    return rank_sum(B, noise_std=noise_std, seed=w.seed, dtype=dtype)


def make_factors(w: Workload, dtype=np.float32) -> list[np.ndarray]:
    out = []
    for n in range(w.d):
        shape = (w.dims[n], w.R)
        s = stream_factor(n)
        if w.index == 1 or w.index == 3:
            out.append(uniform(w.seed, s, shape, 0.0, 1.0, dtype=dtype))
        elif w.index == 2:
            out.append(normal(w.seed, s, shape, 0.0, 0.125, dtype=dtype))
        elif w.index == 4:
            out.append(normal(w.seed, s, shape, 0.0, 1.0, dtype=dtype))
        else:
            out.append(uniform(w.seed, s, shape, -1.0, 1.0, dtype=dtype))
    return out


def random_case(seed: int, dims, R: int, dtype=np.float32, y_dist: str = "uniform"):
    """A small seeded case of arbitrary shape: Y ~ U[-1,1] (or N(0,1)), A_n ~ U[-1,1]."""
    dims = tuple(int(x) for x in dims)
    if y_dist == "normal":
        Y = normal(seed, STREAM_Y, dims, 0.0, 1.0, dtype=dtype)
    else:
        Y = uniform(seed, STREAM_Y, dims, -1.0, 1.0, dtype=dtype)
    A = [uniform(seed, stream_factor(n), (dims[n], R), -1.0, 1.0, dtype=dtype)
         for n in range(len(dims))]
    return Y, A
