"""The allocation-free entry point, mttkrp_noalloc, through the C ABI.

mttkrp_noalloc serves callers that must not allocate device memory (a library
inside a program whose own allocator owns the GPU's memory, or a
latency-critical path where cudaMalloc/cudaFree may block until the device is
idle): its scratch is a fixed static device array inside the library.  Here its
output is checked against the fp64 oracle and against the regular
workspace-based entry point, within the 1e-5 relative Frobenius tolerance of
the other GPU tests, on two calls in a row (the second call reuses scratch the
first one left behind).  This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from conftest import rel_fro

torch = pytest.importorskip("torch")
import dense_tensor_decomposition_gb300 as mk  # noqa: E402

pytestmark = pytest.mark.gpu
TOL = 1e-5


def noalloc_fn():
    lib = mk.load_library()
    fn = lib.mttkrp_noalloc
    vp = ctypes.c_void_p
    fn.argtypes = [ctypes.c_int, vp, ctypes.c_int64, vp, vp, ctypes.c_int, vp, vp]
    fn.restype = ctypes.c_int
    return lib, fn


def call_noalloc(fn, dims, R, Yd, Ad, mode, out):
    arr = (ctypes.c_int64 * len(dims))(*dims)
    ptrs = (ctypes.c_void_p * len(dims))(*[a.data_ptr() for a in Ad])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(len(dims), arr, R, ctypes.c_void_p(Yd.data_ptr()), ptrs, mode,
              ctypes.c_void_p(out.data_ptr()), stream)


@pytest.mark.parametrize("dims,R", [((64, 48, 40), 32), ((37, 41, 9, 5), 19),
                                    ((256, 256, 256), 64)])
def test_noalloc_matches_workspace_entry_point(dims, R):
    lib, fn = noalloc_fn()
    Y, A = synth.random_case(777 + R, dims, R)
    Yd = torch.from_numpy(Y).cuda()
    Ad = [torch.from_numpy(a).cuda() for a in A]
    plan = mk.Plan(dims, R, "simt")
    for k in range(len(dims)):
        ref = oracle.mttkrp(Y, A, k)
        ws = plan.mttkrp(Yd, Ad, k).cpu().numpy()
        for call in range(2):
            out = torch.full((dims[k], R), float("nan"), device="cuda")
            rc = call_noalloc(fn, dims, R, Yd, Ad, k, out)
            assert rc == 0, lib.mttkrp_last_error().decode()
            torch.cuda.synchronize()
            got = out.cpu().numpy()
            assert np.isfinite(got).all()
            err = rel_fro(got, ref)
            assert err <= TOL, f"{dims} R={R} mode {k} call {call}: {err:.3e} against the oracle"
            err = rel_fro(got, ws)
            assert err <= TOL, f"{dims} R={R} mode {k} call {call}: {err:.3e} against mttkrp()"


def test_noalloc_rejects_problems_beyond_the_static_scratch():
    lib, fn = noalloc_fn()
    dims, R = (128, 128, 128, 128), 256  # needs ~57 MB of scratch
    Yd = torch.zeros(1, device="cuda")
    Ad = [torch.zeros(1, device="cuda") for _ in dims]
    out = torch.zeros(1, device="cuda")
    rc = call_noalloc(fn, dims, R, Yd, Ad, 0, out)
    assert rc == 3
    assert b"static scratch" in lib.mttkrp_last_error()
