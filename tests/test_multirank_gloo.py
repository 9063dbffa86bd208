"""Multi-process paths on the CPU (gloo, world size 2).

* bench.py's rank aggregation: the timed value is the maximum over ranks and
  the throughput counts every rank's work (replicas, weak scaling).
* The slab decomposition of MTTKRP across processes, checked with the fp64
  oracle: each rank holds a slab of Y along mode 0 and the matching rows of
  A_0; for k != 0 the per-rank results add up (one all-reduce of I_k x R) to
  the full M_k, and for k = 0 the row blocks concatenate (an all-gather).
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _bench_worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    _init(rank, world, port)
    import bench
    ms = 10.0 + 5.0 * rank
    q.put((rank, bench.max_over_ranks(ms), bench.aggregate_throughput(2e9, world, 15.0)))
    dist.destroy_process_group()


def _slab_worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    _init(rank, world, port)
    import oracle
    import synth
    dims, R = (10, 7, 6, 5), 4
    Y, A = synth.random_case(5150, dims, R, dtype=np.float64)
    lo, hi = dims[0] * rank // world, dims[0] * (rank + 1) // world
    Ys = np.ascontiguousarray(Y[lo:hi])
    As = [A[0][lo:hi]] + A[1:]
    out = {}
    for k in range(1, 4):
        part = torch.from_numpy(oracle.mttkrp(Ys, As, k))
        dist.all_reduce(part)
        out[k] = part.numpy()
    block = torch.from_numpy(oracle.mttkrp(Ys, As, 0))
    sizes = [dims[0] * (r + 1) // world - dims[0] * r // world for r in range(world)]
    gathered = [torch.zeros(s, R, dtype=torch.float64) for s in sizes]
    dist.all_gather(gathered, block)
    out[0] = torch.cat(gathered).numpy()
    if rank == 0:
        full = {k: oracle.mttkrp(Y, A, k) for k in range(4)}
        errs = {k: float(np.linalg.norm(out[k] - full[k]) / np.linalg.norm(full[k])) for k in range(4)}
        q.put(errs)
    dist.destroy_process_group()


def _run(fn, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=fn, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    return q


def test_bench_max_over_ranks_gloo():
    q = _run(_bench_worker)
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [15.0, 15.0]
    assert abs(got[0][2] - 2 * 2e9 / 15e-3 / 1e9) < 1e-9


def test_slab_sharding_matches_full_oracle():
    q = _run(_slab_worker)
    errs = q.get(timeout=10)
    assert all(e <= 1e-13 for e in errs.values()), errs
