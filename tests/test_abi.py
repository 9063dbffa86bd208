"""The C ABI on the host: the library loads, exports every declared symbol, and
validates arguments before touching the GPU.  No compute call reaches a kernel
here (every call below fails validation on the host or is host-only)."""
import ctypes

import numpy as np
import pytest

import dense_tensor_decomposition_gb300 as mk
import synth


@pytest.fixture(scope="module")
def lib():
    mk.build()
    return mk.load_library()


def test_exports_every_declared_symbol(lib):
    names = mk.exported_symbols()
    assert len(names) >= 15
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, f"declared in include/mttkrp.h but not exported: {missing}"


def test_version_and_strerror(lib):
    assert lib.mttkrp_version() >= 100
    assert lib.mttkrp_strerror(0) == b"ok"
    for code in range(1, 7):
        assert lib.mttkrp_strerror(code) not in (b"ok", b"unknown error code")
    assert lib.mttkrp_strerror(99) == b"unknown error code"


def _plan_rc(lib, dims, R):
    arr = (ctypes.c_int64 * max(1, len(dims)))(*dims)
    h = ctypes.c_void_p()
    rc = lib.mttkrp_plan(len(dims), arr, R, ctypes.byref(h))
    if rc == 0:
        lib.mttkrp_plan_destroy(h)
    return rc


@pytest.mark.parametrize("dims,R", [((5,), 3), ((2,) * 9, 3), ((4, 0, 3), 2), ((4, -1), 2),
                                    ((3, 4), 0), ((3, 4), 70000), ((1 << 21, 1 << 21), 4)])
def test_plan_rejects_invalid(lib, dims, R):
    assert _plan_rc(lib, dims, R) == 1
    assert lib.mttkrp_last_error() != b""


def test_plan_rejects_null(lib):
    h = ctypes.c_void_p()
    assert lib.mttkrp_plan(3, None, 4, ctypes.byref(h)) == 1
    arr = (ctypes.c_int64 * 3)(2, 3, 4)
    assert lib.mttkrp_plan(3, arr, 4, None) == 1


@pytest.mark.parametrize("dims,R", [((2, 3), 1), ((7, 5, 3), 9), ((1, 1, 1), 1),
                                    ((3,) * 8, 5), ((1000, 3), 4096)])
def test_plan_accepts_valid(lib, dims, R):
    assert _plan_rc(lib, dims, R) == 0


def _parse(desc):
    out = {}
    for tok in desc.split():
        k, v = tok.split("=", 1)
        out[k] = v
    return out


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_planner_invariants_on_workloads(index):
    w = synth.workload(index)
    p = mk.Plan(w.dims, w.R)
    for k in range(w.d):
        info = _parse(p.describe(k))
        group = [int(x) for x in info["inner_group"].strip("[]").split(",") if x]
        pre = [int(x) for x in info["pre_modes"].strip("[]").split(",") if x]
        # the modes other than k are split into the inner group and the pre modes
        assert sorted(group + pre) == [n for n in range(w.d) if n != k]
        J, npre = int(info["J"]), int(info["npre"])
        assert J == int(np.prod([w.dims[n] for n in group]))
        assert npre == int(np.prod([w.dims[n] for n in pre])) if pre else npre == 1
        assert J * npre * w.dims[k] == w.numel
        splits, pps = int(info["splits"]), int(info["pre_per_split"])
        assert splits * pps >= npre and (splits - 1) * pps < npre
        assert int(info["workspace"]) == p.workspace_bytes(k) > 0
        assert p.mode_path(k) in ("simt", "tc")
    assert p.workspace_bytes(-1) == max(p.workspace_bytes(k) for k in range(w.d))


def test_compute_calls_validate_before_launch(lib):
    """Errors that must be reported on the host, before any kernel is enqueued."""
    p = mk.Plan((6, 5, 4), 3)
    h = p._h
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: every call fails validation
    facs = (ctypes.c_void_p * 3)(1 << 20, 1 << 20, 1 << 20)
    outs = (ctypes.c_void_p * 3)(1 << 20, 1 << 20, 1 << 20)
    # no workspace attached
    assert lib.mttkrp(h, fake, facs, 0, fake, None) == 3
    assert lib.mttkrp_all_modes(h, fake, facs, outs, None) == 3
    # workspace too small
    assert lib.mttkrp_set_workspace(h, ctypes.c_void_p(1 << 20), 256) == 0
    assert lib.mttkrp(h, fake, facs, 1, fake, None) == 3
    # misaligned workspace
    assert lib.mttkrp_set_workspace(h, ctypes.c_void_p((1 << 20) + 8), 1 << 30) == 1
    # mode out of range, NULL pointers
    assert lib.mttkrp(h, fake, facs, 3, fake, None) == 1
    assert lib.mttkrp(h, fake, facs, -1, fake, None) == 1
    assert lib.mttkrp(h, None, facs, 0, fake, None) == 1
    assert lib.mttkrp(h, fake, None, 0, fake, None) == 1
    assert lib.mttkrp(h, fake, facs, 0, None, None) == 1
    assert lib.mttkrp(None, fake, facs, 0, fake, None) == 1
    nullfacs = (ctypes.c_void_p * 3)(1 << 20, None, 1 << 20)
    assert lib.mttkrp_set_workspace(h, ctypes.c_void_p(1 << 20), 1 << 40) == 0
    assert lib.mttkrp(h, fake, nullfacs, 0, fake, None) == 1
    assert lib.mttkrp_all_modes(h, fake, nullfacs, outs, None) == 1
    # misaligned Y
    assert lib.mttkrp(h, ctypes.c_void_p((1 << 20) + 2), facs, 0, fake, None) == 1
    assert p.launch_count() == 0


def test_set_path_and_describe(lib):
    p = mk.Plan((40, 30, 20), 16)
    p.set_path("simt")
    assert all(p.mode_path(k) == "simt" for k in range(3))
    with pytest.raises(ValueError):
        p.describe(3)
    assert lib.mttkrp_plan_set_path(p._h, 7) == 1
    assert lib.mttkrp_plan_mode_path(p._h, 5) == -1
    assert lib.mttkrp_workspace_bytes(p._h, 9) == 0


def test_timing_queries_without_gpu_work(lib):
    p = mk.Plan((4, 5, 6), 2)
    p.set_timing(True)
    assert p.kernel_times(0) == []
    assert lib.mttkrp_plan_kernel_times(p._h, 7, None, 0) < 0


def test_python_binding_rejects_cpu_tensors():
    torch = pytest.importorskip("torch")
    p = mk.Plan((4, 5, 6), 2)
    Y = torch.zeros(4, 5, 6)
    A = [torch.zeros(n, 2) for n in (4, 5, 6)]
    with pytest.raises(TypeError):
        p.mttkrp(Y, A, 0)


def test_image_kernel_planning_and_workspace():
    """Host-only planner decisions for the fp16-image kernel: the K-major and
    innermost modes of the headline shape take it (the innermost mode reading
    the natural images MN-major, flag 3), the workspace grows by one image
    layout (hi + lo, 2 bytes an element each), a stacked small innermost mode
    needs the transposed layout too (flag 2), and tensors above 12 Gi elements
    fall back to the kernels that need no images."""
    def image_flags(p, d):
        return [int(p.describe(k).split("tc_fp16_image=")[1].split()[0]) for k in range(d)]

    p = mk.Plan((512, 512, 512), 2000)
    assert image_flags(p, 3) == [1, 1, 3]
    numel = 512 ** 3
    assert 2 * numel * 2 <= p.workspace_bytes(-1) < 2 * 2 * numel * 2   # natural only, hi + lo
    assert p.workspace_bytes(0) == p.workspace_bytes(-1)        # every image mode sees the region
    q = mk.Plan((20,) * 6, 128)
    assert image_flags(q, 6) == [1, 1, 1, 1, 0, 2]
    assert q.workspace_bytes(-1) >= 2 * 2 * 20 ** 6 * 2         # natural + transposed
    big = mk.Plan((4096, 4096, 1024), 256)
    assert image_flags(big, 3) == [0, 0, 0]
    assert big.workspace_bytes(-1) < 4096 * 4096 * 1024        # no image region


def _fake(addr):
    return ctypes.c_void_p(addr)


@pytest.mark.parametrize("d,dims,mode,J,x,m,t,why", [
    (0, (4,), 0, 2, 0x1000, 0x2000, 0x3000, "order"),
    (9, (2,) * 9, 0, 2, 0x1000, 0x2000, 0x3000, "order"),
    (3, (4, 5, 6), 3, 2, 0x1000, 0x2000, 0x3000, "mode"),
    (3, (4, 5, 6), 1, 0, 0x1000, 0x2000, 0x3000, "J"),
    (3, (4, 0, 6), 1, 2, 0x1000, 0x2000, 0x3000, "dims"),
    (3, (4, 5, 6), 1, 2, 0, 0x2000, 0x3000, "NULL"),
    (3, (4, 5, 6), 1, 2, 0x1000, 0x2000, 0x1002, "aligned"),
    (3, (4, 5, 6), 1, 5, 0x1000, 0x100000, 0x1000 + 4 * 119, "overlap"),     # T's start inside X
    (3, (4, 5, 6), 1, 2, 0x100000, 0x1000, 0x1000 + 4 * 9, "overlap"),       # T's start inside M
])
def test_ttm_rejects_invalid_before_any_launch(lib, d, dims, mode, J, x, m, t, why):
    arr = (ctypes.c_int64 * len(dims))(*dims)
    assert lib.mttkrp_ttm(d, arr, _fake(x), mode, _fake(m), J, _fake(t), None) == 1
    assert why.lower() in lib.mttkrp_last_error().decode().lower()


@pytest.mark.parametrize("d,dims,mode,G,why", [
    (1, (4,), 0, 1, "order"), (3, (4, 5, 6), 3, 1, "mode"), (3, (4, 5, 6), 1, 3, "fit"),
    (3, (4, -5, 6), 1, 1, "dims")])
def test_rotations_reject_invalid_before_any_launch(lib, d, dims, mode, G, why):
    arr = (ctypes.c_int64 * len(dims))(*dims)
    f = _fake(0x1000)
    assert lib.mttkrp_apply_rotations(d, arr, f, mode, f, f, f, G, None) == 1
    assert why.lower() in lib.mttkrp_last_error().decode().lower()


def _ttm_multi_rc(lib, dims, modes, Ms, Js, Ts, x=0x1000, ws=None, ws_bytes=0):
    n = len(modes)
    arr = (ctypes.c_int64 * len(dims))(*dims)
    cm = (ctypes.c_int * n)(*modes)
    cj = (ctypes.c_int64 * n)(*Js)
    cM = (ctypes.c_void_p * n)(*Ms)
    cT = (ctypes.c_void_p * n)(*Ts)
    return lib.mttkrp_ttm_multi(len(dims), arr, _fake(x), n, cm, cM, cj, cT, _fake(ws) if ws else None,
                                ws_bytes, None)


@pytest.mark.parametrize("modes,Ms,Js,Ts,why", [
    ((0, 3), (0x100000, 0x200000), (4, 4), (0x300000, 0x400000), "mode"),
    ((0, 1), (0x100000, 0x200000), (4, 0), (0x300000, 0x400000), "J"),
    ((0, 1), (0x100000, 0), (4, 4), (0x300000, 0x400000), "NULL"),
    ((0, 1), (0x100000, 0x200000), (4, 4), (0x300000, 0x300000 + 16), "overlaps result"),
    ((0, 1), (0x100000, 0x300000 + 64), (4, 4), (0x300000, 0x400000), "overlaps result or matrix"),
])
def test_ttm_multi_rejects_invalid_before_any_launch(lib, modes, Ms, Js, Ts, why):
    assert _ttm_multi_rc(lib, (4, 5, 6), modes, Ms, Js, Ts) == 1
    assert why.lower() in lib.mttkrp_last_error().decode().lower()


def test_ttm_multi_rejects_bad_counts_and_small_workspace(lib):
    arr = (ctypes.c_int64 * 3)(4, 5, 6)
    assert lib.mttkrp_ttm_multi(3, arr, _fake(0x1000), 0, None, None, None, None, None, 0, None) == 1
    assert lib.mttkrp_ttm_multi(3, arr, _fake(0x1000), 65, None, None, None, None, None, 0, None) == 1
    dims = (256, 128, 64)
    need = mk.ttm_multi_workspace_bytes(dims, (0, 1, 2), (64, 64, 64))
    assert need > 0
    rc = _ttm_multi_rc(lib, dims, (0, 1, 2), (0x100000, 0x200000, 0x300000), (64, 64, 64),
                       (0x10000000, 0x20000000, 0x30000000), x=0x40000000, ws=0x50000000, ws_bytes=need - 256)
    assert rc == 3 and b"workspace" in lib.mttkrp_last_error()


def test_ttm_multi_workspace_is_largest_single_product(lib):
    dims = (256, 128, 64)
    single = [mk.ttm_workspace_bytes(dims, m, J) for m, J in ((0, 64), (1, 256), (2, 96), (1, 8))]
    assert single[3] == 0 and min(single[:3]) > 0
    assert mk.ttm_multi_workspace_bytes(dims, (0, 1, 2, 1), (64, 256, 96, 8)) == max(single)
    assert mk.ttm_multi_workspace_bytes(dims, (1,), (8,)) == 0
    # the images of X come first and are the same for every product: more
    # than 4 bytes an element, less than 4 bytes plus the largest M^T region
    numel = 256 * 128 * 64
    assert 4 * numel < max(single) < 4 * numel + 8 * 1024 * 1024
