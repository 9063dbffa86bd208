"""Dense, matrix-free MTTKRP on one GB300 (sm_103a).

A thin ctypes binding of ``libmttkrp.so`` (C ABI in ``include/mttkrp.h``):
it only checks and marshals arguments.  Every step of the computation runs in
the library's CUDA kernels; PyTorch supplies device memory and streams.  There
is no CPU fallback: if the library is missing this module raises.

    M_k(i, r) = sum_{(i_n), n != k} Y(i_0..i_{d-1}) prod_{n != k} A_n(i_n, r)

("A Performance Portable Matrix Free Dense MTTKRP in GenTen", abstract: the
matricized tensor times Khatri-Rao product, computed without forming the
Khatri-Rao matrix.)
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from ._build import LIB as LIB_PATH, build  # noqa: F401

__all__ = ["Plan", "mttkrp", "all_modes", "apply_rotations", "ttm", "ttm_workspace_bytes", "ttm_multi",
           "ttm_multi_workspace_bytes", "probe_fma", "probe_mma",
           "MttkrpError",
           "build", "load_library",
           "exported_symbols", "PATH_AUTO", "PATH_SIMT", "PATH_TC", "PATH_TC_TF32", "PATH_TC_EXPLICIT_KRP"]

PATH_AUTO, PATH_SIMT, PATH_TC, PATH_TC_TF32, PATH_TC_EXPLICIT_KRP = 0, 1, 2, 3, 4
_PATH_NAMES = {"auto": PATH_AUTO, "simt": PATH_SIMT, "tc": PATH_TC, "tc_tf32": PATH_TC_TF32,
               "tc_explicit_krp": PATH_TC_EXPLICIT_KRP}

_lock = threading.Lock()
_lib = None


class MttkrpError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str):
        self.code = code
        super().__init__(f"{where}: {detail} (code {code})")


def load_library():
    """Load libmttkrp.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "dense_tensor_decomposition_gb300.build() (needs nvcc)")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i64, ci, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        lib.mttkrp_plan.argtypes = [ci, vp, i64, ctypes.POINTER(vp)]
        lib.mttkrp_plan.restype = ci
        lib.mttkrp_plan_set_path.argtypes = [vp, ci]
        lib.mttkrp_plan_set_path.restype = ci
        lib.mttkrp_workspace_bytes.argtypes = [vp, ci]
        lib.mttkrp_workspace_bytes.restype = sz
        lib.mttkrp_set_workspace.argtypes = [vp, vp, sz]
        lib.mttkrp_set_workspace.restype = ci
        lib.mttkrp.argtypes = [vp, vp, vp, ci, vp, vp]
        lib.mttkrp.restype = ci
        lib.mttkrp_all_modes.argtypes = [vp, vp, vp, vp, vp]
        lib.mttkrp_all_modes.restype = ci
        lib.mttkrp_plan_mode_path.argtypes = [vp, ci]
        lib.mttkrp_plan_mode_path.restype = ci
        lib.mttkrp_plan_describe.argtypes = [vp, ci, ctypes.c_char_p, sz]
        lib.mttkrp_plan_describe.restype = ci
        lib.mttkrp_plan_set_timing.argtypes = [vp, ci]
        lib.mttkrp_plan_set_timing.restype = ci
        lib.mttkrp_plan_kernel_times.argtypes = [vp, ci, ctypes.POINTER(ctypes.c_float), ci]
        lib.mttkrp_plan_kernel_times.restype = ci
        lib.mttkrp_plan_launch_count.argtypes = [vp]
        lib.mttkrp_plan_launch_count.restype = i64
        lib.mttkrp_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
        lib.mttkrp_device_status.restype = ci
        lib.mttkrp_plan_destroy.argtypes = [vp]
        lib.mttkrp_plan_destroy.restype = None
        lib.mttkrp_strerror.argtypes = [ci]
        lib.mttkrp_strerror.restype = ctypes.c_char_p
        lib.mttkrp_last_error.argtypes = []
        lib.mttkrp_last_error.restype = ctypes.c_char_p
        lib.mttkrp_version.argtypes = []
        lib.mttkrp_version.restype = ci
        lib.mttkrp_apply_rotations.argtypes = [ci, vp, vp, ci, vp, vp, vp, ci, vp]
        lib.mttkrp_apply_rotations.restype = ci
        lib.mttkrp_ttm.argtypes = [ci, vp, vp, ci, vp, i64, vp, vp]
        lib.mttkrp_ttm.restype = ci
        lib.mttkrp_ttm_workspace_bytes.argtypes = [ci, vp, ci, i64]
        lib.mttkrp_ttm_workspace_bytes.restype = sz
        lib.mttkrp_ttm_ws.argtypes = [ci, vp, vp, ci, vp, i64, vp, vp, sz, vp]
        lib.mttkrp_ttm_ws.restype = ci
        lib.mttkrp_ttm_multi_workspace_bytes.argtypes = [ci, vp, ci, vp, vp]
        lib.mttkrp_ttm_multi_workspace_bytes.restype = sz
        lib.mttkrp_ttm_multi.argtypes = [ci, vp, vp, ci, vp, vp, vp, vp, vp, sz, vp]
        lib.mttkrp_ttm_multi.restype = ci
        lib.mttkrp_cp_als_scratch_bytes.argtypes = [vp]
        lib.mttkrp_cp_als_scratch_bytes.restype = sz
        lib.mttkrp_cp_als_sweep.argtypes = [vp, vp, vp, vp, vp, ci, vp, vp, sz, vp]
        lib.mttkrp_cp_als_sweep.restype = ci
        lib.mttkrp_probe_fma.argtypes = [ci, ci, vp, vp]
        lib.mttkrp_probe_fma.restype = ci
        lib.mttkrp_probe_mma.argtypes = [ci, ci, ci, vp]
        lib.mttkrp_probe_mma.restype = ci
        _lib = lib
        return lib


def exported_symbols(header: str | None = None) -> list[str]:
    """Names of the functions declared in include/mttkrp.h."""
    if header is None:
        header = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                              "include", "mttkrp.h")
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mttkrp\w*)\s*\(", text)))


def _check(rc: int, where: str):
    if rc != 0:
        lib = load_library()
        detail = lib.mttkrp_last_error().decode() or lib.mttkrp_strerror(rc).decode()
        raise MttkrpError(rc, where, detail)


def _stream_handle(device, stream=None):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


class Plan:
    """Planner decisions for one tensor shape and rank, plus its workspace.

    The workspace is a PyTorch uint8 tensor on the tensors' device, sized by the
    library (``mttkrp_workspace_bytes``) and attached on first use.
    """

    def __init__(self, dims, R: int, path: str | int = "auto"):
        self._lib = load_library()
        self.dims = tuple(int(x) for x in dims)
        self.R = int(R)
        self.d = len(self.dims)
        arr = (ctypes.c_int64 * self.d)(*self.dims)
        h = ctypes.c_void_p()
        _check(self._lib.mttkrp_plan(self.d, arr, self.R, ctypes.byref(h)), "mttkrp_plan")
        self._h = h
        self._ws = None
        self._ws_device = None
        self._ws_user = False
        if path not in ("auto", PATH_AUTO):
            self.set_path(path)

    # -- planner queries -------------------------------------------------
    def set_path(self, path):
        p = _PATH_NAMES[path] if isinstance(path, str) else int(path)
        _check(self._lib.mttkrp_plan_set_path(self._h, p), "mttkrp_plan_set_path")
        if not self._ws_user:
            self._ws = None  # requirement may have changed

    def workspace_bytes(self, mode: int = -1) -> int:
        return int(self._lib.mttkrp_workspace_bytes(self._h, mode))

    def mode_path(self, mode: int) -> str:
        p = self._lib.mttkrp_plan_mode_path(self._h, mode)
        return {PATH_SIMT: "simt", PATH_TC: "tc"}.get(p, "invalid")

    def describe(self, mode: int) -> str:
        buf = ctypes.create_string_buffer(1024)
        n = self._lib.mttkrp_plan_describe(self._h, mode, buf, 1024)
        if n < 0:
            raise ValueError(f"invalid mode {mode}")
        return buf.value.decode()

    def set_timing(self, enable: bool = True):
        """Record CUDA events around every main kernel (resets earlier records)."""
        rc = self._lib.mttkrp_plan_set_timing(self._h, int(bool(enable)))
        if rc < 0:
            _check(-rc, "mttkrp_plan_set_timing")

    def kernel_times(self, mode: int) -> list[float]:
        """Durations (ms) of the main kernel of `mode` recorded since set_timing()."""
        n = self._lib.mttkrp_plan_kernel_times(self._h, mode, None, 0)
        if n < 0:
            _check(-n, "mttkrp_plan_kernel_times")
        buf = (ctypes.c_float * max(n, 1))()
        n2 = self._lib.mttkrp_plan_kernel_times(self._h, mode, buf, n)
        if n2 < 0:
            _check(-n2, "mttkrp_plan_kernel_times")
        return [float(buf[i]) for i in range(n)]

    def launch_count(self) -> int:
        return int(self._lib.mttkrp_plan_launch_count(self._h))

    # -- workspace ---------------------------------------------------------
    def attach_workspace(self, device):
        """Allocate (through PyTorch) and attach a workspace, unless the caller
        attached its own memory with set_workspace_ptr()."""
        import torch
        if self._ws_user:
            return
        need = self.workspace_bytes(-1)
        if self._ws is not None and self._ws_device == device and self._ws.numel() >= need:
            return
        self._ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        self._ws_device = device
        _check(self._lib.mttkrp_set_workspace(self._h, ctypes.c_void_p(self._ws.data_ptr()),
                                              self._ws.numel()), "mttkrp_set_workspace")

    def set_workspace_ptr(self, ptr: int, nbytes: int):
        """Attach caller-owned device memory (raw pointer) as the workspace.
        The plan then never allocates one itself; the library checks the size."""
        self._ws = None
        self._ws_user = True
        _check(self._lib.mttkrp_set_workspace(self._h, ctypes.c_void_p(ptr), nbytes),
               "mttkrp_set_workspace")

    # -- argument checks -------------------------------------------------
    def _check_inputs(self, Y, factors, skip_mode=None):
        import torch
        if not isinstance(Y, torch.Tensor) or not Y.is_cuda:
            raise TypeError("Y must be a CUDA tensor")
        if Y.dtype != torch.float32 or tuple(Y.shape) != self.dims or not Y.is_contiguous():
            raise ValueError(f"Y must be a contiguous float32 tensor of shape {self.dims}")
        if len(factors) != self.d:
            raise ValueError(f"need {self.d} factors")
        ptrs = []
        for n, a in enumerate(factors):
            if a is None:
                if n != skip_mode:
                    raise ValueError(f"factor {n} is None")
                ptrs.append(None)
                continue
            if a.device != Y.device or a.dtype != torch.float32 or not a.is_contiguous() \
                    or tuple(a.shape) != (self.dims[n], self.R):
                raise ValueError(f"factor {n} must be a contiguous float32 "
                                 f"{(self.dims[n], self.R)} tensor on {Y.device}")
            ptrs.append(a.data_ptr())
        return (ctypes.c_void_p * self.d)(*ptrs)

    def _check_out(self, out, mode, device):
        import torch
        shape = (self.dims[mode], self.R)
        if out is None:
            return torch.empty(shape, dtype=torch.float32, device=device)
        if out.device != device or out.dtype != torch.float32 or not out.is_contiguous() \
                or tuple(out.shape) != shape:
            raise ValueError(f"out must be a contiguous float32 {shape} tensor on {device}")
        return out

    # -- compute -----------------------------------------------------------
    def mttkrp(self, Y, factors, mode: int, out=None, stream=None):
        """M_mode (I_mode x R) for device tensors; enqueued on the current stream."""
        if not 0 <= mode < self.d:
            raise ValueError(f"mode {mode} out of range")
        ptrs = self._check_inputs(Y, factors, skip_mode=mode)
        out = self._check_out(out, mode, Y.device)
        self.attach_workspace(Y.device)
        _check(self._lib.mttkrp(self._h, ctypes.c_void_p(Y.data_ptr()), ptrs, mode,
                                ctypes.c_void_p(out.data_ptr()), _stream_handle(Y.device, stream)),
               "mttkrp")
        return out

    def all_modes(self, Y, factors, outs=None, stream=None):
        """[M_0, ..., M_{d-1}] for device tensors, one call into the library."""
        ptrs = self._check_inputs(Y, factors)
        if outs is None:
            outs = [None] * self.d
        outs = [self._check_out(o, k, Y.device) for k, o in enumerate(outs)]
        optrs = (ctypes.c_void_p * self.d)(*[o.data_ptr() for o in outs])
        self.attach_workspace(Y.device)
        _check(self._lib.mttkrp_all_modes(self._h, ctypes.c_void_p(Y.data_ptr()), ptrs, optrs,
                                          _stream_handle(Y.device, stream)), "mttkrp_all_modes")
        return outs

    def all_modes_from_host(self, Y_host, factors_host, dev_bufs, outs_host, stream=None):
        """End-to-end call from pinned host memory: copy in, compute every mode, copy out.

        dev_bufs = (Y_dev, [A_dev...], [M_dev...]) preallocated device tensors.
        Copies are enqueued on the same stream as the kernels.
        """
        Y_dev, A_dev, M_dev = dev_bufs
        Y_dev.copy_(Y_host, non_blocking=True)
        for a_d, a_h in zip(A_dev, factors_host):
            a_d.copy_(a_h, non_blocking=True)
        self.all_modes(Y_dev, A_dev, outs=M_dev, stream=stream)
        for m_h, m_d in zip(outs_host, M_dev):
            m_h.copy_(m_d, non_blocking=True)
        return outs_host

    def cp_als(self, Y, factors, sweeps: int = 1, stream=None):
        """`sweeps` CP-ALS sweeps on device tensors (mttkrp_cp_als_sweep): the
        factors are updated in place (normalised columns).  Returns (lambda, fits):
        the last column norms (R fp32) and the fit after every sweep (fp64), both
        on the device and not synchronised."""
        import torch
        if sweeps < 1:
            raise ValueError("sweeps must be >= 1")
        ptrs = self._check_inputs(Y, factors)
        self.attach_workspace(Y.device)
        need = int(self._lib.mttkrp_cp_als_scratch_bytes(self._h))
        if getattr(self, "_cp_scratch", None) is None or self._cp_scratch.numel() < need \
                or self._cp_scratch.device != Y.device:
            self._cp_scratch = torch.empty(max(need, 256), dtype=torch.uint8, device=Y.device)
        lam = torch.empty(self.R, dtype=torch.float32, device=Y.device)
        fits = torch.empty(sweeps, dtype=torch.float64, device=Y.device)
        norm = torch.empty(1, dtype=torch.float64, device=Y.device)
        fptrs = (ctypes.c_void_p * self.d)(*[f.data_ptr() for f in factors])
        for t in range(sweeps):
            _check(self._lib.mttkrp_cp_als_sweep(
                self._h, ctypes.c_void_p(Y.data_ptr()), fptrs, ctypes.c_void_p(lam.data_ptr()),
                ctypes.c_void_p(norm.data_ptr()), int(t > 0), ctypes.c_void_p(fits.data_ptr() + 8 * t),
                ctypes.c_void_p(self._cp_scratch.data_ptr()), self._cp_scratch.numel(),
                _stream_handle(Y.device, stream)), "mttkrp_cp_als_sweep")
        return lam, fits

    def all_modes_pipelined(self, batches, dev_bufs, stream=None, copy_stream=None):
        """End to end over a sequence of problems in pinned host memory, with the
        copies overlapped with the computation.

        batches = [(Y_host, [A_host...], [M_host...]), ...]; dev_bufs = two device
        buffer sets (Y_dev, [A_dev...], [M_dev...]) used alternately.  The copy in of
        problem t + 1 runs on a copy stream while problem t is computed on `stream`;
        the outputs of problem t are copied out on the copy stream after its
        computation.  Everything is enqueued; `stream` has waited for the last copy
        out when this returns.
        """
        import torch
        if len(dev_bufs) != 2:
            raise ValueError("dev_bufs must hold two device buffer sets")
        device = dev_bufs[0][0].device
        comp = stream if stream is not None else torch.cuda.current_stream(device)
        cs = copy_stream if copy_stream is not None else torch.cuda.Stream(device=device)
        cs.wait_stream(comp)
        n = len(batches)
        ready, done = [None] * n, [None] * n

        def copy_in(t):
            Y_h, A_h, _ = batches[t]
            Y_d, A_d, _ = dev_bufs[t % 2]
            if t >= 2:
                cs.wait_event(done[t - 2])   # the buffers' previous problem has been computed
            with torch.cuda.stream(cs):
                Y_d.copy_(Y_h, non_blocking=True)
                for a_d, a_h in zip(A_d, A_h):
                    a_d.copy_(a_h, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(cs)
            return ev

        if n:
            ready[0] = copy_in(0)
        for t in range(n):
            if t + 1 < n:
                ready[t + 1] = copy_in(t + 1)
            Y_d, A_d, M_d = dev_bufs[t % 2]
            comp.wait_event(ready[t])
            self.all_modes(Y_d, A_d, outs=M_d, stream=comp)
            done[t] = torch.cuda.Event()
            done[t].record(comp)
            cs.wait_event(done[t])
            with torch.cuda.stream(cs):
                for m_h, m_d in zip(batches[t][2], M_d):
                    m_h.copy_(m_d, non_blocking=True)
        comp.wait_stream(cs)
        return [b[2] for b in batches]

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.mttkrp_plan_destroy(self._h)
            self._h = ctypes.c_void_p()
        self._ws = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def mttkrp(Y, factors, mode: int, path="auto"):
    """One-shot MTTKRP of one mode (plans on every call)."""
    plan = Plan(tuple(Y.shape), factors[(mode + 1) % len(factors)].shape[1], path)
    return plan.mttkrp(Y, factors, mode)


def all_modes(Y, factors, path="auto"):
    plan = Plan(tuple(Y.shape), factors[0].shape[1], path)
    return plan.all_modes(Y, factors)


def apply_rotations(Y, mode: int, pairs, c, s, stream=None):
    """In place: Y x_mode R^T for disjoint Givens pairs (mttkrp_apply_rotations).
    pairs: int32 CUDA tensor (G, 2); c, s: float32 CUDA tensors (G,)."""
    import torch
    lib = load_library()
    if not isinstance(Y, torch.Tensor) or not Y.is_cuda or Y.dtype != torch.float32 or not Y.is_contiguous():
        raise TypeError("Y must be a contiguous float32 CUDA tensor")
    G = int(pairs.shape[0]) if pairs is not None else 0
    for t, dt in ((pairs, torch.int32), (c, torch.float32), (s, torch.float32)):
        if t is not None and (not t.is_cuda or t.dtype != dt or not t.is_contiguous() or t.device != Y.device):
            raise TypeError("pairs (int32), c and s (float32) must be contiguous CUDA tensors on Y's device")
    if pairs is not None and tuple(pairs.shape) != (G, 2) or (G and (c.numel() != G or s.numel() != G)):
        raise ValueError("pairs must be (G, 2), c and s (G,)")
    dims = (ctypes.c_int64 * Y.dim())(*Y.shape)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() else None
    _check(lib.mttkrp_apply_rotations(Y.dim(), dims, ctypes.c_void_p(Y.data_ptr()), mode, ptr(pairs), ptr(c),
                                      ptr(s), G, _stream_handle(Y.device, stream)), "mttkrp_apply_rotations")
    return Y


def ttm_workspace_bytes(shape, mode: int, J: int) -> int:
    """Workspace bytes of the tensor-core mode-n product (0: it does not take the shape)."""
    dims = (ctypes.c_int64 * len(shape))(*shape)
    return int(load_library().mttkrp_ttm_workspace_bytes(len(shape), dims, mode, int(J)))


def ttm(X, mode: int, M, out=None, stream=None, path: str = "auto"):
    """T = X x_mode M: M is a float32 CUDA matrix J x X.shape[mode]; returns T
    (X's shape with that mode's size replaced by J), written into `out` when
    given (contiguous float32, not overlapping X or M).  path "simt": the CUDA-core
    kernel (mttkrp_ttm); "auto": the tensor cores when they take the shape and
    J >= 64 (mttkrp_ttm_ws with a PyTorch-allocated workspace; below that the two
    passes over X that the tensor-core path needs cost more than the CUDA cores'
    arithmetic), else the CUDA cores; "tc": the tensor cores or an error."""
    import torch
    lib = load_library()
    for name, t in (("X", X), ("M", M)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous float32 CUDA tensor")
    if M.device != X.device or M.dim() != 2 or not 0 <= mode < X.dim() or M.shape[1] != X.shape[mode]:
        raise ValueError("M must be J x X.shape[mode] on X's device")
    shape = list(X.shape)
    shape[mode] = int(M.shape[0])
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=X.device)
    elif (not isinstance(out, torch.Tensor) or out.device != X.device or out.dtype != torch.float32
          or not out.is_contiguous() or list(out.shape) != shape):
        raise ValueError(f"out must be a contiguous float32 CUDA tensor of shape {shape}")
    dims = (ctypes.c_int64 * X.dim())(*X.shape)
    if path not in ("auto", "simt", "tc"):
        raise ValueError(f"unknown path {path!r}")
    use_tc = path == "tc" or (path == "auto" and int(M.shape[0]) >= 64)
    need = int(lib.mttkrp_ttm_workspace_bytes(X.dim(), dims, mode, int(M.shape[0]))) if use_tc else 0
    if path == "tc" and need == 0:
        raise MttkrpError(2, "ttm", "the tensor-core mode-n product does not take this shape")
    if need > 0:
        ws = torch.empty(need, dtype=torch.uint8, device=X.device)
        _check(lib.mttkrp_ttm_ws(X.dim(), dims, ctypes.c_void_p(X.data_ptr()), mode, ctypes.c_void_p(M.data_ptr()),
                                 int(M.shape[0]), ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                                 need, _stream_handle(X.device, stream)), "mttkrp_ttm_ws")
        return out
    _check(lib.mttkrp_ttm(X.dim(), dims, ctypes.c_void_p(X.data_ptr()), mode, ctypes.c_void_p(M.data_ptr()),
                          int(M.shape[0]), ctypes.c_void_p(out.data_ptr()), _stream_handle(X.device, stream)),
           "mttkrp_ttm")
    return out


def ttm_multi_workspace_bytes(shape, modes, Js) -> int:
    """Workspace bytes of several tensor-core mode-n products of one tensor (the
    images of X once plus the largest per-product region; 0: none is taken)."""
    n = len(modes)
    dims = (ctypes.c_int64 * len(shape))(*shape)
    cm = (ctypes.c_int * n)(*[int(m) for m in modes])
    cj = (ctypes.c_int64 * n)(*[int(j) for j in Js])
    return int(load_library().mttkrp_ttm_multi_workspace_bytes(len(shape), dims, n, cm, cj))


def ttm_multi(X, modes, Ms, outs=None, stream=None, path: str = "auto", workspace=None):
    """T_t = X x_{modes[t]} Ms[t] for every t (mttkrp_ttm_multi): the products a
    Tucker form takes of one tensor, the tensor-core ones sharing one pass that
    writes X's fp16 images.  Ms: float32 CUDA matrices J_t x X.shape[modes[t]];
    returns the list of results (written into `outs` when given).  path "simt":
    every product on the CUDA cores; "auto": the tensor cores for every product
    they take when some J_t >= 64, else the CUDA cores; "tc": the tensor cores
    for every product or an error.  workspace: a uint8 CUDA tensor of at least
    ttm_multi_workspace_bytes() bytes to use instead of a fresh allocation."""
    import torch
    lib = load_library()
    modes = [int(m) for m in modes]
    Ms = list(Ms)
    n = len(modes)
    if n < 1 or len(Ms) != n:
        raise ValueError("modes and Ms must be non-empty and of the same length")
    if not isinstance(X, torch.Tensor) or not X.is_cuda or X.dtype != torch.float32 or not X.is_contiguous():
        raise TypeError("X must be a contiguous float32 CUDA tensor")
    shapes = []
    for t, (m, M) in enumerate(zip(modes, Ms)):
        if not isinstance(M, torch.Tensor) or not M.is_cuda or M.dtype != torch.float32 or not M.is_contiguous():
            raise TypeError(f"Ms[{t}] must be a contiguous float32 CUDA tensor")
        if M.device != X.device or M.dim() != 2 or not 0 <= m < X.dim() or M.shape[1] != X.shape[m]:
            raise ValueError(f"Ms[{t}] must be J x X.shape[{m}] on X's device")
        shape = list(X.shape)
        shape[m] = int(M.shape[0])
        shapes.append(shape)
    if outs is None:
        outs = [torch.empty(sh, dtype=torch.float32, device=X.device) for sh in shapes]
    else:
        outs = list(outs)
        if len(outs) != n:
            raise ValueError("outs must hold one tensor per product")
        for t, (o, sh) in enumerate(zip(outs, shapes)):
            if (not isinstance(o, torch.Tensor) or o.device != X.device or o.dtype != torch.float32
                    or not o.is_contiguous() or list(o.shape) != sh):
                raise ValueError(f"outs[{t}] must be a contiguous float32 CUDA tensor of shape {sh}")
    if path not in ("auto", "simt", "tc"):
        raise ValueError(f"unknown path {path!r}")
    Js = [int(M.shape[0]) for M in Ms]
    dims = (ctypes.c_int64 * X.dim())(*X.shape)
    cm = (ctypes.c_int * n)(*modes)
    cj = (ctypes.c_int64 * n)(*Js)
    cM = (ctypes.c_void_p * n)(*[M.data_ptr() for M in Ms])
    cT = (ctypes.c_void_p * n)(*[o.data_ptr() for o in outs])
    use_tc = path == "tc" or (path == "auto" and max(Js) >= 64)
    need = int(lib.mttkrp_ttm_multi_workspace_bytes(X.dim(), dims, n, cm, cj)) if use_tc else 0
    if path == "tc":
        for t in range(n):
            if int(lib.mttkrp_ttm_workspace_bytes(X.dim(), dims, modes[t], Js[t])) == 0:
                raise MttkrpError(2, "ttm_multi", f"the tensor-core mode-n product does not take product {t}")
    if need > 0 and workspace is not None:
        if (not isinstance(workspace, torch.Tensor) or workspace.device != X.device
                or workspace.dtype != torch.uint8 or not workspace.is_contiguous()):
            raise TypeError("workspace must be a contiguous uint8 CUDA tensor on X's device")
        ws, ws_bytes = workspace, workspace.numel()
    else:
        ws = torch.empty(need, dtype=torch.uint8, device=X.device) if need > 0 else None
        ws_bytes = need
    _check(lib.mttkrp_ttm_multi(X.dim(), dims, ctypes.c_void_p(X.data_ptr()), n, cm, cM, cj, cT,
                                ctypes.c_void_p(ws.data_ptr()) if ws is not None else None, ws_bytes,
                                _stream_handle(X.device, stream)), "mttkrp_ttm_multi")
    return outs


def probe_fma(blocks: int, iters: int, out, stream=None):
    """Enqueue the fp32 FMA peak probe (mttkrp_probe_fma); out: float32 CUDA
    tensor of blocks * 256 elements.  flops = 16 * iters * blocks * 256."""
    _check(load_library().mttkrp_probe_fma(int(blocks), int(iters), ctypes.c_void_p(out.data_ptr()),
                                           _stream_handle(out.device, stream)), "mttkrp_probe_fma")


def probe_mma(kind: str, blocks: int, iters: int, device=None, stream=None):
    """Enqueue the tensor-pipe peak probe (mttkrp_probe_mma) for kind "tf32" (K = 8)
    or "f16" (K = 16).  flops = 2 * 128 * 256 * K * iters * blocks."""
    import torch
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    k = {"tf32": 0, "f16": 1}[kind]
    _check(load_library().mttkrp_probe_mma(k, int(blocks), int(iters), _stream_handle(device, stream)),
           "mttkrp_probe_mma")


def device_status() -> int:
    """Read and clear the kernels' device-side error word (synchronises)."""
    w = ctypes.c_uint32(0)
    _check(load_library().mttkrp_device_status(ctypes.byref(w)), "mttkrp_device_status")
    return int(w.value)
