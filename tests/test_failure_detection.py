"""Failure detection without a GPU fault.

Host side: argument errors, missing or undersized workspace and NULL pointers
are reported as status codes before anything is enqueued (test_abi.py covers
these on the CPU).  Device side: every wait inside the tensor-core kernel is
bounded in time.  The test hook mttkrp_test_withhold_signal makes the next
launch withhold one accumulator-ready signal (a flag that nothing sets), so the
epilogue's wait expires after about one second; the kernel records a status
bit, drains its own copies and MMAs, frees its tensor memory and returns.  The
host reads the bit with mttkrp_device_status(), and the next call on the same
context computes correct results.
"""
import ctypes
import time

import numpy as np
import pytest

import oracle
import synth
from conftest import rel_fro

torch = pytest.importorskip("torch")
import dense_tensor_decomposition_gb300 as mk  # noqa: E402

pytestmark = pytest.mark.gpu


# one CTA (one row tile, one column tile, few pre indices); and the kernel that
# converts Y in place (64 CTAs, with its converter warps and image stores)
@pytest.mark.parametrize("dims,R,path,convert", [((128, 16, 32), 64, "tc", False),
                                                 ((256, 64, 128), 256, "auto", True)])
def test_expired_wait_sets_status_and_context_survives(dims, R, path, convert):
    lib = mk.load_library()
    lib.mttkrp_test_withhold_signal.argtypes = [ctypes.c_int]
    lib.mttkrp_test_withhold_signal.restype = ctypes.c_int
    try:
        plan = mk.Plan(dims, R, path)
    except mk.MttkrpError:
        pytest.skip("tensor-core path unavailable")
    assert ("tc_convert=1" in plan.describe(0)) == convert
    Y, A = synth.random_case(808, dims, R)
    Yd = torch.from_numpy(Y).cuda()
    Ad = [torch.from_numpy(a).cuda() for a in A]
    assert mk.device_status() == 0
    ref = oracle.mttkrp(Y, A, 0)

    lib.mttkrp_test_withhold_signal(1)
    t0 = time.time()
    plan.mttkrp(Yd, Ad, 0)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    status = mk.device_status()
    assert status != 0, "the expired wait was not reported"
    assert 0.5 < elapsed < 30.0, elapsed
    assert lib.mttkrp_test_withhold_signal(0) == 0  # the hook disarmed itself

    # the context is still usable and the next call is correct
    out = plan.mttkrp(Yd, Ad, 0)
    torch.cuda.synchronize()
    assert mk.device_status() == 0
    assert rel_fro(out.cpu().numpy(), ref) <= 1e-5
