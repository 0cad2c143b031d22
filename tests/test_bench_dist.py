"""The multi-process side of bench.py on CPU: the replicas-only run (one
process per GPU, no data-path collective) keeps a barrier and takes the
max of the ranks' step times and the sum of their work. These tests run
world size 2 over gloo, and the oracle arm under torchrun, where rank 0
alone prints its line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, local = bench.dist_setup()
    bench.barrier(w)
    mx = bench.allreduce(float(r + 1) * 10.0, "max", w)
    sm = bench.allreduce(float(r + 1), "sum", w)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    out.put((r, w, local, mx, sm))


def test_replica_timing_reduces_max_time_and_sum_work_over_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(out.get(timeout=5) for _ in range(world))
    assert [g[0] for g in got] == [0, 1]
    for r, w, local, mx, sm in got:
        assert w == world and local == r
        assert mx == 20.0          # the slowest rank's time
        assert sm == 3.0           # the work of all ranks


def test_reference_arm_prints_one_line_from_rank_zero_under_torchrun():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "1", "--config", "tiny"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
