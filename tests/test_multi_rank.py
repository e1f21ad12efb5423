"""The benchmark's multi-rank host logic on CPU (gloo, world size 2).

The attention path has no exchange step: ranks are independent replicas, each
with its own batch, and only the timing is combined (max of the ranks' times,
sum of their work). These tests run that combination and the reference arm's
rank handling as real two-process jobs over gloo.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    w, r, _ = bench.dist_setup()
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # per-rank time and work: the job's time is the slowest rank's, its work the sum
    t = bench.reduce_max(10.0 + 5.0 * r, w)
    units = bench.reduce_sum(100.0 * (r + 1), w)
    bench.barrier(w)
    out.put((r, w, t, units))
    dist.destroy_process_group()


def test_two_ranks_combine_time_by_max_and_work_by_sum():
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(out.get() for _ in range(2))
    assert [g[0] for g in got] == [0, 1]
    for _, world, t, units in got:
        assert world == 2 and t == 15.0 and units == 300.0


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5 and bench.reduce_sum(3.5, 1) == 3.5
    bench.barrier(1)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    """`bench.py --impl reference` launched as the driver launches N = 2: rank 0
    alone times the oracle and prints one JSON line; rank 1 exits 0 without work."""
    import oracle
    oracle.build()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--cpu-seconds", "1",
           "--workload", "tiny"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


if __name__ == "__main__":
    pytest.main([__file__, "-q"])
