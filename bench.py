#!/usr/bin/env python3
"""Benchmark: dense matrix-free MTTKRP, every mode of one workload, on GB300.

One step = M_k for every mode k of the workload (one mttkrp_all_modes call),
inputs resident in HBM.  Prints one JSON line (rank 0):

  value        MTTKRP GFLOP/s over all ranks, 2*R*prod(I_n) flops per mode
  ms_per_step  milliseconds for all modes (device time, CUDA events, max over ranks)
  e2e          the same metric through the public API from pinned host memory,
               host->device copies of Y and the factors and device->host copies
               of the outputs inside the timed region, every step; the copy in
               of step t + 1 overlaps the computation of step t
               (serial_ms_per_step: one after another)
  roofline     the main contraction kernel: algorithmic flops per launch over its
               average CUDA-event duration, against the pipe's peak; call_frac:
               the whole all-modes call against the same roofline
  peaks_probe  fp32 FMA, tcgen05 kind::tf32 and kind::f16 rates measured in this
               run by the library's probe kernels, with the SM clock seen
  per_workload all five workloads (and the largest on the 3xTF32 kernels): per
               mode the kernel, its time, GFLOP/s and roofline fraction
               (t_roof = max(flops / that kernel's pipe peak, algorithmic bytes /
               HBM bandwidth)), and the all-modes time and fraction
  cpu_baseline the fp64 oracle on a bounded sample, on this host's cores

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 4] [--path auto|simt|tc|tc_tf32]
  python bench.py --impl reference ...   # the oracle on the host cores, same metric

N > 1 (torchrun): every rank runs the whole workload on its own GPU (replicas;
the path needs no exchange between GPUs); value counts all ranks' work over
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
SM_MAX_MHZ_FALLBACK = 2070.0
# nominal dense tensor rates relative to bf16 (2.25 PFLOP/s): tf32 1.1 PFLOP/s
# (used only when the tf32 probe could not run)
TF32_OVER_BF16 = 1.1 / 2.25


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="4")
    ap.add_argument("--path", default="auto", choices=["auto", "simt", "tc", "tc_tf32"])
    ap.add_argument("--no-workload-sweep", action="store_true",
                    help="skip the per-workload block (all five workloads, per mode)")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cp-als", type=int, default=0, metavar="SWEEPS",
                    help="instead: time SWEEPS CP-ALS sweeps (mttkrp_cp_als_sweep) on the workload's tensor")
    ap.add_argument("--cp-rank", type=int, default=32, help="rank of the CP-ALS model (--cp-als)")
    ap.add_argument("--ttm", type=int, default=-1, metavar="J",
                    help="instead: time the dense mode-n product X x_k M_k along every mode with J x I_k "
                         "matrices (J = 0: square, J = I_k)")
    ap.add_argument("--explicit-krp", action="store_true",
                    help="instead: the matrix-based variant (explicit Khatri-Rao product) against the "
                         "matrix-free one on several workloads: time per mode and workspace bytes")
    ap.add_argument("--rotations", action="store_true",
                    help="instead: time Givens rotations (a full group of disjoint pairs) along every mode")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target length of the oracle CPU-baseline sample")
    return ap.parse_args()


def workload_from_arg(s):
    return synth.workload(int(s)) if s.isdigit() else synth.workload(s)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": SM_MAX_MHZ_FALLBACK}, "fallback"


# the files the main contraction kernel of each path is compiled and launched
# from (kernel, shared declarations, planner); a DRAM traffic record stays valid
# while these are unchanged, whatever happens to the other kernels
MAIN_KERNEL_SOURCES = {"tc": ("api.cu", "internal.h", "tc.cu", "tc.h"),
                       "simt": ("api.cu", "internal.h", "simt.cu")}


def kernel_source_hash(names=None):
    """Hash of the CUDA sources: all of them, or only the files in `names`."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_tensor_decomposition_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if names is not None and name not in names:
            continue
        if name.endswith((".cu", ".h", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, path, src_hash):
    """DRAM bytes per launch of the main kernel from an ncu capture summary, if it
    was taken on the current kernel sources (else None)."""
    fn = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(fn):
        return None
    for line in open(fn):
        if line.startswith("#") or not line.strip():
            continue
        kv = dict(tok.split("=", 1) for tok in line.split() if "=" in tok)
        if kv.get("workload") == workload and kv.get("path") == path and kv.get("src") == src_hash:
            return float(kv["bytes_per_launch"])
    return None


def max_over_ranks(x: float, device=None) -> float:
    """Largest value of x over all ranks (x itself without torch.distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(flops_per_rank_step: float, world: int, ms_per_step_max: float) -> float:
    """Whole-job GFLOP/s: every rank's work over the slowest rank's step time."""
    return world * flops_per_rank_step / (ms_per_step_max * 1e-3) / 1e9


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.device_index = device_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.device_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [l.strip().split(",") for l in self.file.read().splitlines() if l.strip()]
        self.file.close()
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() in ("active", "1"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# CPU side: the oracle (test infrastructure; used only for the baseline legs)
# ---------------------------------------------------------------------------

def oracle_sample(w, Y, A, seconds):
    """Time the fp64 oracle on sampled output rows of mode 0, sized to ~seconds."""
    import oracle
    k = 0
    ncols = w.numel // w.dims[k]
    t0 = time.perf_counter()
    oracle.mttkrp(Y, A, k, rows=[0])
    t1 = time.perf_counter() - t0
    rows = int(max(1, min(w.dims[k], seconds / max(t1, 1e-3))))
    rows_list = list(range(rows))
    t0 = time.perf_counter()
    oracle.mttkrp(Y, A, k, rows=rows_list)
    dt = time.perf_counter() - t0
    flops = 2.0 * w.R * ncols * rows
    return {"value": flops / dt / 1e9, "unit": "GFLOP/s", "cores": oracle.threads(),
            "kind": "oracle",
            "sample": f"mode 0, output rows 0..{rows - 1} of {w.dims[k]} "
                      f"({rows}/{w.dims[k]} of one mode), {dt:.1f} s, fp64"}


def _mode_sample(Yh, k, elems):
    """Y cut to its first s indices along one mode other than k (mode 0, or
    mode 1 when k == 0) so that it holds about `elems` elements; a view."""
    d = Yh.ndim
    if d == 1:
        return Yh
    m = 0 if k != 0 else 1
    per = Yh.size // Yh.shape[m]
    s = int(max(1, min(Yh.shape[m], elems // max(per, 1))))
    return Yh[(slice(None),) * m + (slice(0, s),)]


def _timed_samples(Yh, seconds, run_mode, units_of):
    """Grow a per-mode sample until one pass over all modes takes about
    `seconds`; returns (units processed, seconds, elements per mode sample)."""
    elems = 1 << 18
    while True:
        t0 = time.perf_counter()
        units = 0.0
        for k in range(Yh.ndim):
            sample = _mode_sample(Yh, k, elems)
            run_mode(sample, k)
            units += units_of(sample, k)
        dt = time.perf_counter() - t0
        if dt >= seconds / 4 or elems >= Yh.size:
            return units, dt, elems
        elems = int(min(Yh.size, elems * max(2.0, min(16.0, seconds / 2 / max(dt, 1e-3)))))


def rotations_cpu_baseline(Yh, groups, seconds):
    """The fp64 rotation oracle on slices of the tensor (one mode at a time,
    a full group per mode), GB/s of rotated rows read and written."""
    from oracle import rotations as orot

    def run(sample, k):
        orot.apply_rotations(sample, k, *groups[k])

    def units(sample, k):
        return 2.0 * 4 * (sample.size // sample.shape[k]) * 2 * len(groups[k][0])

    moved, dt, elems = _timed_samples(Yh, seconds, run, units)
    return {"value": moved / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"every mode on a slice of about {elems} elements (cut along another mode), "
                      f"{dt:.1f} s, numpy fp64, one thread"}


def ttm_cpu_baseline(Xh, Ms, seconds):
    """The fp64 mode-n product oracle on slices of the tensor, TFLOP/s."""
    from oracle import ttm as ottm

    def run(sample, k):
        ottm.ttm(sample, k, Ms[k])

    def units(sample, k):
        return 2.0 * Ms[k].shape[0] * sample.size

    flops, dt, elems = _timed_samples(Xh, seconds, run, units)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"every mode on a slice of about {elems} elements (cut along another mode), "
                      f"{dt:.1f} s, numpy fp64 matrix products (BLAS threads)"}


def cp_als_cpu_baseline(Yh, A0):
    """One fp64 oracle sweep on the whole tensor, ms per sweep."""
    import numpy as np
    import oracle
    from oracle import cp_als as ocp
    norm = float(np.sum(np.asarray(Yh, dtype=np.float64) ** 2))
    t0 = time.perf_counter()
    ocp.cp_als_sweep(Yh, A0, norm_y2=norm)
    dt = time.perf_counter() - t0
    return {"value": dt * 1e3, "unit": "ms", "cores": oracle.threads(), "kind": "oracle",
            "sample": f"one sweep on the whole tensor ({dt:.1f} s; ||Y||^2 precomputed), "
                      f"MTTKRP in the C oracle (OpenMP), the rest numpy fp64"}


def run_reference(args, w):
    """--impl reference: the oracle on this host's cores, same metric and workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    Y = synth.make_tensor(w)
    A = synth.make_factors(w)
    # one step = one sampled output row of every mode
    rows = [[w.dims[k] // 2] for k in range(w.d)]
    flops = sum(2.0 * w.R * (w.numel // w.dims[k]) for k in range(w.d))

    def step():
        for k in range(w.d):
            oracle.mttkrp(Y, A, k, rows=rows[k])

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = flops / dt / 1e9
    line = {
        "impl": "reference",
        "metric": "MTTKRP GFLOP/s (2*R*prod(I_n) per mode), all modes",
        "value": round(value, 4), "unit": "GFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "dims": list(w.dims), "R": w.R,
                   "step": "one sampled output row of every mode (bounded sample)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GFLOP/s", "cores": oracle.threads(),
                         "kind": "oracle",
                         "sample": f"output row I_k/2 of each of the {w.d} modes per step"},
        "e2e": {"value": round(value, 4), "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU side
# ---------------------------------------------------------------------------

def kernel_name(plan, k):
    """The planner's kernel for mode k (family.layout[.small].bn<columns>)."""
    for tok in plan.describe(k).split():
        if tok.startswith("kernel="):
            return tok[len("kernel="):]
    return "unknown"


def kernel_kind(name):
    """Arithmetic of a kernel: fp16x2 (two-term fp16 split on the tensor cores),
    tf32x3 (3xTF32 on the tensor cores) or f32 (fp32 FMA on the CUDA cores)."""
    return {"img": "fp16x2", "h2": "fp16x2", "tf32": "tf32x3", "tf32tm": "tf32x3"}.get(name.split(".")[0], "f32")


def probe_peaks(device, sms):
    """Rates of the library's probe kernels in this run (TFLOP/s), with the SM
    clock sampled while they run: an fp32 FMA chain on every SM, and one CTA
    per SM issuing tcgen05 MMAs (M128 N256) of kind::tf32 and kind::f16."""
    import torch
    import dense_tensor_decomposition_gb300 as mk
    stream = torch.cuda.current_stream(device)
    out = torch.empty(sms * 8 * 256, device=device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def rate(launch, flops, seconds=0.3):
        launch()
        torch.cuda.synchronize(device)
        n = 1
        while True:
            e0.record(stream)
            for _ in range(n):
                launch()
            e1.record(stream)
            torch.cuda.synchronize(device)
            ms = e0.elapsed_time(e1)
            if ms >= seconds * 1e3 or n >= 1 << 14:
                return flops * n / (ms * 1e-3) / 1e12
            n = int(min(1 << 14, n * max(2.0, seconds * 1e3 / max(ms, 1e-3))))

    clocks = ClockSampler(device.index)
    clocks.start()
    time.sleep(0.3)
    fma_iters, mma_iters = 16384, 8192
    res = {
        "fp32_fma_tflops": rate(lambda: mk.probe_fma(sms * 8, fma_iters, out),
                                16.0 * fma_iters * sms * 8 * 256),
        "tf32_mma_tflops": rate(lambda: mk.probe_mma("tf32", sms, mma_iters, device),
                                2.0 * 128 * 256 * 8 * mma_iters * sms),
        "f16_mma_tflops": rate(lambda: mk.probe_mma("f16", sms, mma_iters, device),
                               2.0 * 128 * 256 * 16 * mma_iters * sms),
    }
    res = {k: round(v, 2) for k, v in res.items()}
    res["clocks"] = clocks.stop()
    res["status"] = mk.device_status()
    res["how"] = (f"fp32: {sms * 8} blocks x 256 threads x {fma_iters} iterations of 8 FMA chains; "
                  f"tensor: {sms} CTAs (one per SM) x {mma_iters} back-to-back tcgen05.mma M128 N256 "
                  f"(tf32 K8, f16 K16); CUDA events, about 0.3 s each")
    return res


def kind_peaks(peaks, probe, sms):
    """TFLOP/s of one fp32-accurate product per kind: fp16x2 = the driver-measured
    bf16 dense burst / 3 (fp16 and bf16 share the rate), tf32x3 = the tf32 probe
    / 3, f32 = the FMA probe (fallbacks: bf16 x nominal 1.1/2.25 / 3, and
    SMs x 128 x 2 x max clock)."""
    fp16 = peaks["bf16_tflops"] / 3.0
    tf32 = (probe["tf32_mma_tflops"] if probe else peaks["bf16_tflops"] * TF32_OVER_BF16) / 3.0
    f32 = probe["fp32_fma_tflops"] if probe else sms * 128 * 2 * peaks.get("sm_max_mhz", SM_MAX_MHZ_FALLBACK) / 1e6
    return {"fp16x2": fp16, "tf32x3": tf32, "f32": f32}


def roofline_ms(w, k, kind, kpk, hbm_gbs):
    """t_roof of mode k: the slower of its flops at its pipe's peak and its
    algorithmic bytes at the HBM bandwidth; and which one it is."""
    t_flop = w.flops_per_mode() / (kpk[kind] * 1e12) * 1e3
    t_hbm = w.bytes_per_mode(k) / (hbm_gbs * 1e9) * 1e3
    return max(t_flop, t_hbm), ("hbm" if t_hbm > t_flop else ("alu" if kind == "f32" else "tensor"))


def workload_sweep(device, kpk, hbm_gbs, cases):
    """Every mode of each (workload, path) in `cases`: the main kernel's CUDA-event
    time (median over calls), GFLOP/s and roofline fraction per mode, and the
    whole all-modes call (median of per-call events; workloads that fit in L2
    get a 512 MiB L2 flush before every call)."""
    import torch
    import dense_tensor_decomposition_gb300 as mk
    stream = torch.cuda.current_stream(device)
    out = []
    for idx, path in cases:
        w = synth.workload(idx)
        Y = torch.from_numpy(synth.make_tensor(w)).to(device)
        A = [torch.from_numpy(a).to(device) for a in synth.make_factors(w)]
        M = [torch.empty(n, w.R, device=device) for n in w.dims]
        plan = mk.Plan(w.dims, w.R, path)
        plan.attach_workspace(device)
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=device) if Y.numel() * 4 <= L2_BYTES else None
        for _ in range(3):
            plan.all_modes(Y, A, outs=M)
        torch.cuda.synchronize(device)
        reps = 20 if w.numel <= 1 << 24 else 5
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        plan.set_timing(True)
        for r in range(reps):
            if flush is not None:
                flush.fill_(r & 255)
            evs[r][0].record(stream)
            plan.all_modes(Y, A, outs=M)
            evs[r][1].record(stream)
        torch.cuda.synchronize(device)
        ms_all = statistics.median(a.elapsed_time(b) for a, b in evs)
        modes, roof_sum, kern_sum = [], 0.0, 0.0
        for k in range(w.d):
            kt = statistics.median(plan.kernel_times(k))
            name = kernel_name(plan, k)
            kind = kernel_kind(name)
            t_roof, bound = roofline_ms(w, k, kind, kpk, hbm_gbs)
            roof_sum += t_roof
            kern_sum += kt
            modes.append({"mode": k, "kernel": name, "ms": round(kt, 4),
                          "gflops": round(w.flops_per_mode() / (kt * 1e-3) / 1e9, 1),
                          "t_roof_ms": round(t_roof, 4), "bound": bound, "frac": round(t_roof / kt, 3)})
        plan.set_timing(False)
        out.append({"workload": w.name, "path": path, "dims": list(w.dims), "R": w.R,
                    "ms_all_modes": round(ms_all, 4),
                    "gflops_all_modes": round(w.d * w.flops_per_mode() / (ms_all * 1e-3) / 1e9, 1),
                    "frac_all_modes": round(roof_sum / ms_all, 3),
                    "ms_main_kernels": round(kern_sum, 4),
                    "l2": "flushed before every call" if flush is not None else "Y larger than L2",
                    "modes": modes})
        del Y, A, M, plan, flush
        torch.cuda.empty_cache()
    return out


def run_ours(args, w):
    import torch
    import torch.distributed as dist
    import dense_tensor_decomposition_gb300 as mk

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)

    def barrier():
        if world > 1:
            dist.barrier()

    Y = synth.make_tensor(w)
    A = synth.make_factors(w)
    Yd = torch.from_numpy(Y).to(device)
    Ad = [torch.from_numpy(a).to(device) for a in A]
    Md = [torch.empty(w.dims[k], w.R, device=device) for k in range(w.d)]
    plan = mk.Plan(w.dims, w.R, args.path)
    plan.attach_workspace(device)
    stream = torch.cuda.current_stream(device)

    # inputs that fit in L2 get an L2 flush (a 512 MiB write) before every timed
    # step; each step is then timed with its own events, flush excluded
    flush = None
    if Y.nbytes <= L2_BYTES:
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)

    for _ in range(args.warmup):
        plan.all_modes(Yd, Ad, outs=Md)
    torch.cuda.synchronize(device)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    plan.set_timing(True)
    launches0 = plan.launch_count()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps if flush is not None else 1)]
    barrier()
    torch.cuda.synchronize(device)
    w0 = time.perf_counter()
    if flush is None:
        evs[0][0].record(stream)
        for _ in range(args.steps):
            plan.all_modes(Yd, Ad, outs=Md)
        evs[0][1].record(stream)
    else:
        for s in range(args.steps):
            flush.fill_(s & 255)
            evs[s][0].record(stream)
            plan.all_modes(Yd, Ad, outs=Md)
            evs[s][1].record(stream)
    torch.cuda.synchronize(device)
    barrier()
    wall = time.perf_counter() - w0
    clk = clocks.stop()
    launches = plan.launch_count() - launches0
    ms_total = sum(a.elapsed_time(b) for a, b in evs)
    kern = [t for k in range(w.d) for t in plan.kernel_times(k)]
    plan.set_timing(False)

    ms_max = max_over_ranks(ms_total, device)
    ms_per_step = ms_max / args.steps
    flops_step = w.d * w.flops_per_mode()
    value = aggregate_throughput(flops_step, world, ms_per_step)

    # ---- end to end through the public API, from pinned host memory ----
    Yh = torch.from_numpy(Y).pin_memory()
    Ah = [torch.from_numpy(a).pin_memory() for a in A]
    Mh = [torch.empty(w.dims[k], w.R).pin_memory() for k in range(w.d)]
    h2d = Yh.numel() * 4 + sum(a.numel() * 4 for a in Ah)
    d2h = sum(m.numel() * 4 for m in Mh)
    plan.all_modes_from_host(Yh, Ah, (Yd, Ad, Md), Mh)
    torch.cuda.synchronize(device)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # one problem after another: copy in, compute, copy out, serialised
    e0.record(stream)
    for _ in range(args.e2e_steps):
        plan.all_modes_from_host(Yh, Ah, (Yd, Ad, Md), Mh)
    e1.record(stream)
    torch.cuda.synchronize(device)
    serial_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, device)
    # a stream of problems: the copy in of problem t + 1 overlaps the computation
    # of problem t (two device buffer sets); every step still copies its own
    # inputs in and its outputs out
    bufs = ((Yd, Ad, Md), (torch.empty_like(Yd), [torch.empty_like(a) for a in Ad],
                           [torch.empty_like(m) for m in Md]))
    batches = [(Yh, Ah, Mh)] * args.e2e_steps
    plan.all_modes_pipelined(batches[:2], bufs, stream=stream)
    torch.cuda.synchronize(device)
    barrier()
    e0.record(stream)
    plan.all_modes_pipelined(batches, bufs, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, device)
    e2e_value = aggregate_throughput(flops_step, world, e2e_ms)
    checksum = float(sum(float(m.double().abs().sum()) for m in Mh))

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    # ---- peaks measured in this run, roofline of the main contraction kernel ----
    peaks, peak_src = measured_peaks()
    props = torch.cuda.get_device_properties(device)
    sms = props.multi_processor_count
    try:
        probe = probe_peaks(device, sms)
    except Exception as e:  # the probes are context; the bench line stands without them
        probe = {"error": str(e)[:200]}
    kpk = kind_peaks(peaks, probe if "error" not in probe else None, sms)
    path = plan.mode_path(0)
    names = [kernel_name(plan, k) for k in range(w.d)]
    kinds = [kernel_kind(n) for n in names]
    kern_ms = statistics.mean(kern) if kern else None
    achieved_tflops = (w.flops_per_mode() / (kern_ms * 1e-3) / 1e12) if kern_ms else None
    # the modes' pipes, flop-weighted (every mode has the same flops): the time
    # all modes would take at their pipes' peaks, per mode
    flops = w.flops_per_mode()
    t_peak = sum(flops / (kpk[kd] * 1e12) for kd in kinds)
    peak = w.d * flops / t_peak / 1e12
    bound = "alu" if set(kinds) == {"f32"} else "tensor"
    roof_ms = [roofline_ms(w, k, kinds[k], kpk, peaks["hbm_gbs"])[0] for k in range(w.d)]
    call_frac = sum(roof_ms) / ms_per_step
    frac_sustained = None
    if "fp16x2" in kinds and achieved_tflops:
        sus = dict(kpk, fp16x2=peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) / 3.0)
        frac_sustained = round(achieved_tflops / (w.d * flops / sum(flops / (sus[kd] * 1e12) for kd in kinds)
                                                  / 1e12), 4)
    peak_note = ("per mode " + ", ".join(f"{n} ({kd})" for n, kd in zip(names, kinds))
                 + f"; fp16x2 = bf16 dense burst ({peak_src}) / 3 products; tf32x3 = tcgen05 kind::tf32 probe"
                   f" / 3 products; f32 = fp32 FMA probe (peaks_probe; nominal fallbacks if it failed)")
    main_src = kernel_source_hash(MAIN_KERNEL_SOURCES.get(path, ()))
    traffic = recorded_traffic(w.name, path, main_src)
    roofline = {"bound": bound, "achieved": round(achieved_tflops, 3) if achieved_tflops else None,
                "peak": round(peak, 3), "unit": "TFLOP/s",
                "frac": round(achieved_tflops / peak, 4) if achieved_tflops else None,
                "traffic": traffic, "peak_source": peak_note,
                "call_frac": round(call_frac, 4),
                "call_frac_note": "all-modes call (every kernel of the step) against the same roofline: "
                                  "sum over modes of max(flops / pipe peak, algorithmic bytes / HBM) "
                                  "over ms_per_step",
                "frac_vs_sustained_peak": frac_sustained,
                "kernel_ms_mean": round(kern_ms, 4) if kern_ms else None,
                "kernel_launches_timed": len(kern),
                "algorithmic_bytes_per_launch": max(w.bytes_per_mode(k) for k in range(w.d)),
                "hbm_gbs_at_algorithmic_bytes":
                    round(max(w.bytes_per_mode(k) for k in range(w.d)) / (kern_ms * 1e-3) / 1e9, 1)
                    if kern_ms else None}
    sweep = None
    if not args.no_workload_sweep:
        sweep = workload_sweep(device, kpk, peaks["hbm_gbs"],
                               [(i, "auto") for i in (1, 2, 3, 4, 5)] + [(w.index, "tc_tf32")])

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = oracle_sample(w, Y, A, args.cpu_seconds)

    line = {
        "metric": "MTTKRP GFLOP/s (2*R*prod(I_n) per mode), all modes",
        "value": round(value, 2), "unit": "GFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "+".join(sorted(set(kinds))), "data": "synthetic",
        "config": {"workload": w.name, "dims": list(w.dims), "R": w.R, "modes": w.d,
                   "path": path, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2 (Y {Y.nbytes >> 20} MiB > 129 MB)"
                         if flush is None else "L2 flushed (512 MiB write) before every step",
                   "ms_per_mode": round(ms_per_step / w.d, 4), "wall_s_timed": round(wall, 3)},
        "e2e": {"value": round(e2e_value, 2), "unit": "GFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
                "steps": args.e2e_steps, "copies": "overlapped with the previous step's compute",
                "serial_ms_per_step": round(serial_ms, 3)},
        "roofline": roofline,
        "peaks_probe": probe,
        "per_workload": sweep,
        "cpu_baseline": cpu,
        "clocks": clk,
        "gpu_launches": launches,
        "kernel_src": kernel_source_hash(), "main_kernel_src": main_src,
        "checksum": checksum,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_cp_als(args, w):
    """CP-ALS sweeps on the workload's tensor at rank --cp-rank from a seeded
    random start: one JSON line with the time per sweep, the MTTKRP share of it
    (CUDA events around the main kernels) and the fit reached."""
    import numpy as np
    import torch
    import dense_tensor_decomposition_gb300 as mk
    device = torch.device("cuda", 0)
    Yh = synth.make_tensor(w)
    Y = torch.from_numpy(Yh).to(device)
    R = args.cp_rank
    rng = np.random.default_rng(20261202)
    A0 = [rng.standard_normal((n, R)).astype(np.float32) for n in w.dims]
    plan = mk.Plan(w.dims, R, args.path)
    A = [torch.from_numpy(a).to(device) for a in A0]
    plan.cp_als(Y, A, sweeps=max(args.warmup, 1))          # warm-up (and first ||Y||^2)
    A = [torch.from_numpy(a).to(device) for a in A0]
    torch.cuda.synchronize(device)
    plan.set_timing(True)
    stream = torch.cuda.current_stream(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    lam, fits = plan.cp_als(Y, A, sweeps=args.cp_als)
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / args.cp_als
    mttkrp_ms = sum(sum(plan.kernel_times(k)) for k in range(w.d)) / args.cp_als
    plan.set_timing(False)
    cpu = None if args.no_cpu_baseline else cp_als_cpu_baseline(Yh, A0)
    # MTTKRP arithmetic, then the R x R algebra: compensated fp32 (Gram, Cholesky
    # with refinement) up to rank 1024, fp64 above
    cp_dtype = ("fp16x2" if plan.mode_path(0) == "tc" else "f32") + ("+f32c" if R <= 1024 else "+f64")
    print(json.dumps({
        "metric": "CP-ALS time per sweep (every factor updated once, fit included)",
        "value": round(ms, 4), "unit": "ms", "higher_is_better": False, "n_gpus": 1,
        "steps": args.cp_als, "dtype": cp_dtype,
        "data": "synthetic", "impl": "ours",
        "config": {"workload": w.name, "dims": list(w.dims), "R": R, "start": "seeded N(0,1) factors"},
        "mttkrp_kernel_ms_per_sweep": round(mttkrp_ms, 4),
        "mttkrp_share": round(mttkrp_ms / ms, 4),
        "fit_first_last": [round(float(fits[0]), 6), round(float(fits[-1]), 6)],
        "cpu_baseline": cpu,
        "kernel_src": kernel_source_hash(),
    }))


def run_rotations(args, w):
    """A full group of N/2 disjoint Givens pairs along every mode of the workload's
    tensor per step (mttkrp_apply_rotations): each step reads and writes the
    tensor once per mode.  One JSON line: GB/s against the measured HBM peak."""
    import numpy as np
    import torch
    import dense_tensor_decomposition_gb300 as mk
    device = torch.device("cuda", 0)
    Yh = synth.make_tensor(w)
    Y = torch.from_numpy(Yh).to(device)
    rng = np.random.default_rng(20261202)
    groups, groups_h = [], []
    for n in w.dims:
        G = n // 2
        pairs = rng.permutation(n)[: 2 * G].reshape(G, 2).astype(np.int32)
        phi = rng.uniform(-np.pi, np.pi, G)
        groups_h.append((pairs, np.cos(phi).astype(np.float32), np.sin(phi).astype(np.float32)))
        groups.append(tuple(torch.from_numpy(x).to(device) for x in groups_h[-1]))

    def step():
        for k in range(w.d):
            mk.apply_rotations(Y, k, *groups[k])

    for _ in range(max(args.warmup, 3)):
        step()
    stream = torch.cuda.current_stream(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / args.steps
    per_mode = []
    for k in range(w.d):
        e0.record(stream)
        for _ in range(args.steps):
            mk.apply_rotations(Y, k, *groups[k])
        e1.record(stream)
        torch.cuda.synchronize(device)
        per_mode.append(round(e0.elapsed_time(e1) / args.steps, 4))
    moved = 0
    for k, n in enumerate(w.dims):
        moved += 2 * 4 * (int(np.prod(w.dims)) // n) * 2 * (n // 2)   # rotated rows read + written
    gbs = moved / (ms * 1e-3) / 1e9
    peaks, src = measured_peaks()
    cpu = None if args.no_cpu_baseline else rotations_cpu_baseline(Yh, groups_h, args.cpu_seconds)
    print(json.dumps({
        "metric": "Givens rotations along every mode: GB/s of rotated rows read and written",
        "value": round(gbs, 1), "unit": "GB/s", "higher_is_better": True, "n_gpus": 1,
        "steps": args.steps, "ms_per_step": round(ms, 4), "dtype": "f32", "data": "synthetic", "impl": "ours",
        "config": {"workload": w.name, "dims": list(w.dims), "group": "N/2 disjoint pairs per mode",
                   "l2": "tensor larger than L2" if 4 * int(np.prod(w.dims)) > 129e6 else "fits L2"},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": src},
        "ms_per_mode": per_mode,
        "cpu_baseline": cpu,
        "kernel_src": kernel_source_hash(),
    }))


def ttm_roofline(flops, nbytes, kinds, kind_peak, hbm_gbs, ms):
    """Roofline of a step of mode-n products: per product the slower of its flops
    at the pipe it runs on (kind_peak[kind], TFLOP/s) and its algorithmic bytes
    at HBM (hbm_gbs).  When the HBM times of the step add up to more than the
    pipe times the line is reported as HBM-bound (GB/s, bytes over the step's
    time), else against the flop-weighted pipe peak (TFLOP/s); t_roof_ms sums
    the per-product maxima."""
    t_pipe = [f / (kind_peak[k] * 1e12) for f, k in zip(flops, kinds)]
    t_hbm = [b / (hbm_gbs * 1e9) for b in nbytes]
    t_roof = sum(max(a, b) for a, b in zip(t_pipe, t_hbm))
    if sum(t_hbm) > sum(t_pipe):
        achieved = sum(nbytes) / (ms * 1e-3) / 1e9
        out = {"bound": "hbm", "achieved": round(achieved, 1), "peak": round(hbm_gbs, 1), "unit": "GB/s",
               "frac": round(achieved / hbm_gbs, 4)}
    else:
        achieved = sum(flops) / (ms * 1e-3) / 1e12
        peak = sum(flops) / sum(t_pipe) / 1e12
        out = {"bound": "alu" if set(kinds) == {"f32"} else "tensor", "achieved": round(achieved, 3),
               "peak": round(peak, 3), "unit": "TFLOP/s", "frac": round(achieved / peak, 4)}
    out["t_roof_ms"] = round(t_roof * 1e3, 4)
    out["frac_of_t_roof"] = round(t_roof * 1e3 / ms, 4)
    return out


def run_ttm(args, w):
    """The dense mode-n product along every mode of the workload's tensor per
    step, one mttkrp_ttm_multi call (the tensor-core products share one pass
    that writes the fp16 images of X), each mode into its own preallocated
    result.  One JSON line: TFLOP/s (2 J I_1..I_d flops per mode); the
    roofline against the flop-weighted peak of the pipes the products run on,
    or against HBM when the algorithmic bytes take longer (ttm_roofline);
    ms_per_mode times each product alone (mttkrp_ttm_ws, its own image pass
    included)."""
    import numpy as np
    import torch
    import dense_tensor_decomposition_gb300 as mk
    device = torch.device("cuda", 0)
    Xh = synth.make_tensor(w)
    X = torch.from_numpy(Xh).to(device)
    rng = np.random.default_rng(20261203)
    numel = int(np.prod(w.dims))
    Js = [n if args.ttm == 0 else args.ttm for n in w.dims]
    Ms_h = [rng.standard_normal((J, n)).astype(np.float32) for J, n in zip(Js, w.dims)]
    Ms = [torch.from_numpy(m).to(device) for m in Ms_h]
    outs = [torch.empty(list(w.dims[:k]) + [Js[k]] + list(w.dims[k + 1:]), device=device) for k in range(w.d)]

    modes = list(range(w.d))
    need = mk.ttm_multi_workspace_bytes(w.dims, modes, Js) if max(Js) >= 64 else 0
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)

    def step():
        mk.ttm_multi(X, modes, Ms, outs=outs, workspace=ws if need else None)

    for _ in range(max(args.warmup, 3)):
        step()
    stream = torch.cuda.current_stream(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / args.steps
    per_mode = []
    for k in range(w.d):
        e0.record(stream)
        for _ in range(args.steps):
            mk.ttm(X, k, Ms[k], out=outs[k])
        e1.record(stream)
        torch.cuda.synchronize(device)
        per_mode.append(round(e0.elapsed_time(e1) / args.steps, 4))
    flops = sum(2.0 * J * numel for J in Js)
    moved = sum(4.0 * (numel + J * numel // n + J * n) for J, n in zip(Js, w.dims))
    tflops = flops / (ms * 1e-3) / 1e12
    peaks, src = measured_peaks()
    props = torch.cuda.get_device_properties(device)
    try:
        probe = probe_peaks(device, props.multi_processor_count)
    except Exception as e:
        probe = {"error": str(e)[:200]}
    kpk = kind_peaks(peaks, probe if "error" not in probe else None, props.multi_processor_count)
    # per mode: the tensor cores (fp16 split) where they take the shape, else the
    # FMA pipe; ttm_multi(path="auto") takes them for every product they take
    # once some J >= 64
    kinds = ["fp16x2" if need and mk.ttm_workspace_bytes(w.dims, k, Js[k]) > 0 else "f32"
             for k in range(w.d)]
    roof = ttm_roofline([2.0 * J * numel for J in Js],
                        [4.0 * (numel + J * numel // n + J * n) for J, n in zip(Js, w.dims)],
                        kinds, kpk, peaks["hbm_gbs"], ms)
    roof.update({"peak_source": "per mode: fp16x2 = bf16 dense burst (" + src + ") / 3 products, "
                                "f32 = fp32 FMA probe; flop-weighted; HBM: measured copy bandwidth",
                 "hbm_ms_at_algorithmic_bytes": round(moved / (peaks["hbm_gbs"] * 1e9) * 1e3, 4),
                 "hbm_peak_source": src})
    cpu = None if args.no_cpu_baseline else ttm_cpu_baseline(Xh, Ms_h, args.cpu_seconds)
    print(json.dumps({
        "metric": "dense mode-n product along every mode: TFLOP/s (2 J prod(I_n) per mode)",
        "value": round(tflops, 3), "unit": "TFLOP/s", "higher_is_better": True, "n_gpus": 1,
        "steps": args.steps, "ms_per_step": round(ms, 4), "dtype": "+".join(sorted(set(kinds))), "data": "synthetic",
        "impl": "ours",
        "config": {"workload": w.name, "dims": list(w.dims), "J": Js, "kinds": kinds,
                   "l2": "tensor larger than L2" if 4 * numel > 129e6 else "fits L2"},
        "roofline": roof,
        "ms_per_mode": per_mode,
        "peaks_probe": probe,
        "cpu_baseline": cpu,
        "kernel_src": kernel_source_hash(),
    }))


def run_explicit_krp(args):
    """The matrix-based variant (MTTKRP_PATH_TC_EXPLICIT_KRP: the Khatri-Rao
    product of every mode but k formed in the workspace, then multiplied on the
    tensor cores) against the matrix-free planner choice, on 256^3, 128^4, 20^6
    and 512^3: all-modes time, per-mode main-kernel time and workspace bytes by
    purpose.  One JSON line."""
    import torch
    import dense_tensor_decomposition_gb300 as mk
    device = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(device)
    out = []
    for idx in (2, 3, 5, 4):
        w = synth.workload(idx)
        Y = torch.from_numpy(synth.make_tensor(w)).to(device)
        A = [torch.from_numpy(a).to(device) for a in synth.make_factors(w)]
        M = [torch.empty(n, w.R, device=device) for n in w.dims]
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=device) if Y.numel() * 4 <= L2_BYTES else None
        entry = {"workload": w.name, "dims": list(w.dims), "R": w.R,
                 "krp_bytes_per_mode": [4 * w.R * (w.numel // n) for n in w.dims]}
        for variant, path in (("matrix_free", "auto"), ("explicit_krp", "tc_explicit_krp")):
            plan = mk.Plan(w.dims, w.R, path)
            plan.attach_workspace(device)
            for _ in range(max(args.warmup, 2)):
                plan.all_modes(Y, A, outs=M)
            torch.cuda.synchronize(device)
            plan.set_timing(True)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(5)]
            for r, (e0, e1) in enumerate(evs):
                if flush is not None:
                    flush.fill_(r & 255)
                e0.record(stream)
                plan.all_modes(Y, A, outs=M)
                e1.record(stream)
            torch.cuda.synchronize(device)
            fs = [dict(t.split("=", 1) for t in plan.describe(k).split() if "=" in t) for k in range(w.d)]
            entry[variant] = {
                "ms_all_modes": round(statistics.median(a.elapsed_time(b) for a, b in evs), 4),
                "ms_main_kernel": [round(statistics.median(plan.kernel_times(k)), 4) for k in range(w.d)],
                "kernels": [f["kernel"] for f in fs],
                "workspace_bytes": plan.workspace_bytes(-1),
                "ws_tables_max": max(int(f["ws_tables"]) for f in fs),
                "ws_partials_max": max(int(f["ws_partials"]) for f in fs),
                "ws_images": max(int(f["ws_images"]) for f in fs)}
            plan.set_timing(False)
            assert mk.device_status() == 0
            del plan
            torch.cuda.empty_cache()
        mf, ex = entry["matrix_free"], entry["explicit_krp"]
        entry["explicit_over_free_time"] = round(ex["ms_all_modes"] / mf["ms_all_modes"], 3)
        entry["explicit_product_over_free_tables"] = round(max(entry["krp_bytes_per_mode"]) / mf["ws_tables_max"], 1)
        out.append(entry)
        del Y, A, M, flush
        torch.cuda.empty_cache()
    print(json.dumps({
        "metric": "matrix-based (explicit Khatri-Rao product) vs matrix-free MTTKRP: ms per all-modes call "
                  "and workspace bytes",
        "unit": "ms", "higher_is_better": False, "n_gpus": 1, "data": "synthetic", "impl": "ours",
        "dtype": "fp16x2 (tf32x3 where the fp16 images do not apply)",
        "workloads": out, "kernel_src": kernel_source_hash()}))


def main():
    args = parse_args()
    w = workload_from_arg(args.workload)
    if args.impl == "reference":
        run_reference(args, w)
    elif args.explicit_krp:
        run_explicit_krp(args)
    elif args.rotations:
        run_rotations(args, w)
    elif args.ttm >= 0:
        run_ttm(args, w)
    elif args.cp_als > 0:
        run_cp_als(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
