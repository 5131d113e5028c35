"""The benchmark's multi-rank host logic on CPU ranks (gloo / torchrun, two
ranks): the slowest rank's time sets the job's time, the job's throughput is
every rank's work over it, and the reference arm prints its one line from
rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [0.25, 0.4][rank]
    bench.barrier(world)
    ms = bench.max_over_ranks(local_ms, world)
    out.put((rank, ms, bench.whole_job_tflops(1e12, ms, world)))
    bench.barrier(world)
    dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # 2 ranks x 1e12 flops in 0.4 ms (the slower rank) = 5000 TFLOP/s on both ranks
    assert [g[1] for g in got] == [0.4, 0.4]
    assert [round(g[2], 6) for g in got] == [5000.0, 5000.0]


def test_reference_arm_under_torchrun_prints_from_rank0_only():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--cpu-budget", "1"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.lstrip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
