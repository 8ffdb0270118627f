"""The N > 1 path of bench.py, run as world-size-2 gloo process groups on CPU.

The decode SpMV does not shard: every GPU runs an independent replica of the
decode-token stack and no data crosses ranks. What the multi-rank bench adds
is host logic only: rendezvous, a barrier on both sides of the timed region,
the maximum of the per-rank step time, and the whole-job aggregation
(``world`` tokens per slowest step). These tests check that logic with real
process groups and check that the reference arm prints exactly one line, from
rank 0, under torchrun.
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


def _rank_main(rank, world, port, step_ms, out_q):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    r, w, local = bench.dist_init()
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    ms_max = bench.max_over_ranks(step_ms[rank], w)
    out_q.put((rank, ms_max, bench.job_us_per_token(ms_max, w)))
    bench.barrier(w)
    dist.destroy_process_group()


def test_max_over_ranks_and_job_aggregate_gloo():
    world = 2
    step_ms = [1.75, 2.5]  # rank 1 is the slower replica
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, step_ms, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, ms_max, us in got:
        assert ms_max == max(step_ms)  # every rank sees the slowest rank's time
        assert us == pytest.approx(max(step_ms) * 1e3 / world)  # two tokens per slowest step


def test_job_aggregate_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_us_per_token(2.0, 1) == pytest.approx(2000.0)
    assert bench.job_us_per_token(2.0, 4) == pytest.approx(500.0)


def test_reference_arm_two_ranks_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env={**os.environ, "OMP_NUM_THREADS": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["n_gpus"] == 2
    assert out["cpu_baseline"]["kind"] == "oracle"
    assert out["e2e"]["h2d_bytes_per_step"] == 0 and out["e2e"]["value"] == out["value"]
    assert out["higher_is_better"] is False and out["value"] > 0
