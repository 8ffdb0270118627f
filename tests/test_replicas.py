"""The N > 1 paths, run as world-size-2 gloo process groups on CPU.

The decode SpMV does not shard: every GPU runs an independent replica of the
decode-token stack and no data crosses ranks. What the multi-rank bench adds
is host logic only: rendezvous, a barrier on both sides of the timed region,
the maximum of the per-rank step time, and the whole-job aggregation
(``world`` tokens per slowest step). These tests check that logic with real
process groups and check that the reference arm prints exactly one line, from
rank 0, under torchrun. The path itself would shard by rows (x replicated,
y gathered) or by K (partial sums added): ranks that pack and multiply their
row shards, gathered, give the unsharded bits, and K shards give the
unsharded packing and a sum within the fp64 bound.
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


def _shard_main(rank, world, port, out_q):
    try:
        _shard_rank(rank, world, port, out_q)
    except Exception as e:  # reported to the test instead of a silent exit
        out_q.put({"error": f"rank {rank}: {e!r}"})
        raise


def _shard_rank(rank, world, port, out_q):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import torch.distributed as dist

    import oracle
    import sparse_decoding_gb300 as nm
    import synth
    from tests.bits import to_bits
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rows, K, N, M = 96, 256, 4, 8
    W = synth.nm_structured(rows, K, N, M, seed=5)
    x = synth.activations(2, K, seed=6)
    r0, r1 = rank * rows // world, (rank + 1) * rows // world      # row shard (a multiple of 32)
    k0, k1 = rank * K // world, (rank + 1) * K // world            # K shard (a multiple of 32)

    def gather(t):
        parts = [torch.empty_like(t) for _ in range(world)]
        dist.all_gather(parts, t)
        return parts

    m_r, v_r = nm.pack_host(W[r0:r1].contiguous(), N, M)           # the product's host packer
    m_k, v_k = nm.pack_host(W[:, k0:k1].contiguous(), N, M)
    y_r, _ = oracle.spmv_f64(to_bits(W[r0:r1].contiguous()), to_bits(x))
    y_k, _ = oracle.spmv_f64(to_bits(W[:, k0:k1].contiguous()), to_bits(x[:, k0:k1].contiguous()))
    out = {
        # bf16 values travel as pairs of 16-bit words in int32 (gloo has no 16-bit types)
        "m_rows": torch.cat(gather(m_r), 0), "v_rows": torch.cat(gather(v_r.view(torch.int32)), 0),
        "m_k": torch.cat(gather(m_k), 1), "v_k": torch.cat(gather(v_k.view(torch.int32)), 1),
        "y_rows": torch.cat(gather(torch.from_numpy(np.ascontiguousarray(y_r))), 1),
        "y_k": sum(gather(torch.from_numpy(np.ascontiguousarray(y_k)))),
    }
    if rank == 0:
        out_q.put({k: v.numpy() for k, v in out.items()})
    dist.barrier()
    dist.destroy_process_group()


def test_row_and_k_shards_gloo():
    sys.path.insert(0, ROOT)
    import numpy as np

    import oracle
    import sparse_decoding_gb300 as nm
    import synth
    from tests.bits import to_bits
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = q.get(timeout=300)
    assert "error" not in got, got.get("error")
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    W = synth.nm_structured(96, 256, 4, 8, seed=5)
    x = synth.activations(2, 256, seed=6)
    m, v = nm.pack_host(W, 4, 8)
    y, S = oracle.spmv_f64(to_bits(W), to_bits(x))
    # row shards: the gathered masks, values and products are the unsharded bits
    assert np.array_equal(got["m_rows"], m.numpy())
    assert np.array_equal(got["v_rows"], v.view(__import__("torch").int32).numpy())
    assert np.array_equal(got["y_rows"], y)
    # K shards: the per-row concatenation of the shards' words and values is
    # the unsharded packing (32-column words never straddle a shard), and the
    # shards' partial products add up to the unsharded one within the fp64 bound
    assert np.array_equal(got["m_k"], m.numpy())
    assert np.array_equal(got["v_k"], v.view(__import__("torch").int32).numpy())
    assert np.all(np.abs(got["y_k"] - y) <= 1e-12 * S)
