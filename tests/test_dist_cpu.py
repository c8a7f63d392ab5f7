"""The multi-process path of bench.py on CPU (gloo, world size 2): the
rank helpers it times with (barrier, max and sum over ranks), the per-rank
seeding of the replicas, and a whole torchrun launch of the reference arm
(rank 0 prints the one JSON line, the other rank exits 0 without work)."""

import json
import os
import socket
import subprocess
import sys

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    r, w, pg = bench.dist_setup(world)
    assert (r, w) == (rank, world) and pg is not None
    bench.barrier(pg)
    mx = bench.max_over_ranks(pg, 10.0 + rank)           # the slowest rank's time is the job's time
    sm = bench.sum_over_ranks(pg, 1000.0 * (rank + 1))   # every rank's bytes count in the job's value
    # replicas: each rank draws its own batch from its own seed
    q = workloads.tiny_decode(seed=1 + rank).q.float().sum().item()
    t = torch.tensor([q], dtype=torch.float64)
    gathered = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
    pg.all_gather(gathered, t)
    qs = [float(g.item()) for g in gathered]
    bench.barrier(pg)
    pg.destroy_process_group()
    out_q.put((rank, mx, sm, qs))


def test_rank_helpers_world_size_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, sm, qs in res:
        assert mx == 11.0
        assert sm == 3000.0
        assert qs[0] != qs[1]  # different replicas


def test_reference_arm_under_torchrun_world_size_2():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", "--master-port=%d" % port, os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env={**os.environ, "OMP_NUM_THREADS": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout  # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
