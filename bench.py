#!/usr/bin/env python
"""Benchmark of the bitmask N:M decode SpMV on one decode token's linear stack.

A step is one decode token through every pruned linear of a Llama-3.1-8B-shaped
model: 32 layers x {qkv 6144x4096, o 4096x4096, gate_up 28672x4096,
down 4096x14336}, batch 1, pattern 2:4, i.e. 128 nm_spmv launches chained with
programmatic dependent launch and replayed as one CUDA graph. Weights are
synthetic (bf16 N(0, 0.02^2), Wanda-selected with a synthetic column norm,
packed on the GPU); the step reads 7.85 GB, far more than L2, so no flush is
needed between steps.

Prints one JSON line. ``value`` is microseconds per decode token (lower is
better) over the whole job. Extra keys: the same-GPU dense references (the
hand-written dense GEMV and cuBLAS), the roofline of the SpMV kernel, the CPU
oracle as a timed baseline, an end-to-end figure with host buffers, and the SM
clocks seen during the timed region.

``--impl reference`` times the CPU oracle instead (the only reference
implementation this method has), on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "bitmask N:M SpMV µs/decode-token (8B shapes), HBM GB/s vs peak, × vs dense GEMV"
UNIT = "us/token"
CONFIG_ID = 2  # stream-id namespace of the decode-token stack inputs
FALLBACK_HBM_GBS = 6800.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "nm_spmv_llama8b_stack.txt")
KERNEL_SOURCES = [os.path.join(ROOT, "sparse_decoding_gb300", "csrc", f) for f in ("spmv.cu", "streamk.cuh")]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--model", default="llama3.1-8b", choices=sorted(synth.MODELS))
    ap.add_argument("--pattern", default="2:4")
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (0 = the model's)")
    ap.add_argument("--no-variants", action="store_true", help="skip the extra pattern/batch lines")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-pruning", action="store_true", help="skip the OBS pruning measurement")
    ap.add_argument("--only-pruning", action="store_true",
                    help="run only the OBS pruning measurement and print its JSON object")
    ap.add_argument("--prune-linears", default="qkv,o,gate_up,down", help="linears to prune (comma list)")
    ap.add_argument("--prune-repeats", type=int, default=2, help="timed repeats per linear (after one untimed)")
    ap.add_argument("--suite", action="store_true",
                    help="run the larger model stacks instead (Qwen3-14B/32B at 4:8 and 8:16, batch 1; "
                         "Llama-3.3-70B at 2:4 and 16:32, batch 1/2/4/8) and print their JSON object")
    return ap.parse_args()


def parse_pattern(s: str):
    n, m = s.split(":")
    return int(n), int(m)


# --- multi-process (one process per GPU; replicas) ------------------------------------

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    """Max of a per-rank float over all ranks (the job is as slow as its slowest rank)."""
    if world == 1:
        return v
    import torch.distributed as dist
    dev = torch.device("cuda") if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_us_per_token(ms_per_step_max: float, world: int) -> float:
    """Whole-job time per decode token: every rank decodes one token per step
    (independent replicas), so `world` tokens finish in the slowest rank's step."""
    return ms_per_step_max * 1e3 / world


# --- bytes -------------------------------------------------------------------------------

def sparse_bytes(rows, K, batch):
    """Algorithmic bytes of one SpMV: kept values + masks + x + bf16 y."""
    return rows * (K // 2 * 2 + K // 8) + batch * K * 2 + batch * rows * 2


def dense_bytes(rows, K, batch):
    return rows * K * 2 + batch * K * 2 + batch * rows * 2


# --- clocks (NVML through ctypes; reading only) --------------------------------------------

class ClockSampler:
    """Samples SM clock and clock-event reasons of this process's GPU every ~2 ms."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int):
        self.ok = False
        self.samples = []
        self.max_mhz = None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            self.h = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._reasons = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(self.nvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
        except Exception:
            self.ok = False
        self._stop = threading.Event()

    def _run(self):
        mhz = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0 and \
                    self._reasons(self.h, ctypes.byref(rs)) == 0:
                self.samples.append((mhz.value, rs.value))
            time.sleep(0.002)

    def __enter__(self):
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"], "samples": 0}
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s for s, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(self.samples), "source": "nvml"}


# --- workload ---------------------------------------------------------------------------------

class Stack:
    """All linears of one decode token: weights packed per pattern, x/y per batch size.

    Each linear's W and column norms a are drawn on the GPU; every pattern is
    selected and packed from the same W in one pass (nm_select_pack). The dense
    references keep W itself (the dense model's weights). With swiglu, the
    gate_up linears of the first pattern are also packed in the gate/up pair
    layout of the SwiGLU epilogue."""

    def __init__(self, nm, model: str, patterns, batches, layers: int, keep_dense: bool, seed: int = 0,
                 swiglu: bool = True):
        shapes = synth.MODELS[model]
        self.model = model
        self.layers = layers or shapes["layers"]
        self.shapes = [(name, shapes[name][0], shapes[name][1]) for name in synth.MATRICES]
        self.patterns = list(patterns)
        self.packed = {p: [] for p in patterns}
        self.dense = []
        self.swiglu = []  # gate_up of the first pattern in the gate/up pair layout
        for layer in range(self.layers):
            for mi, (name, rows, K) in enumerate(self.shapes):
                W = synth.weights(rows, K, seed, synth.stream_id(CONFIG_ID, layer, mi, 0), device="cuda")
                a = synth.col_norms(K, seed, synth.stream_id(CONFIG_ID, layer, mi, 1), device="cuda")
                for pi, (N, M) in enumerate(patterns):
                    self.packed[(N, M)].append(nm.select_pack(W, a, N, M))
                    if swiglu and pi == 0 and name == "gate_up":
                        Wp = nm.select(W, a, N, M)
                        self.swiglu.append(nm.pack_swiglu(Wp[:rows // 2], Wp[rows // 2:], N, M))
                        del Wp
                if keep_dense:
                    self.dense.append(W)
                del W, a
        self.io = {}
        for b in batches:
            ktot = sum(K for _, _, K in self.shapes) * self.layers
            rtot = sum(r for _, r, _ in self.shapes) * self.layers
            x_all = torch.empty(b * ktot, dtype=torch.bfloat16, device="cuda")
            y_all = torch.empty(b * rtot, dtype=torch.bfloat16, device="cuda")
            xs, ys = [], []
            xo = yo = 0
            for layer in range(self.layers):
                for mi, (name, rows, K) in enumerate(self.shapes):
                    x = x_all[xo:xo + b * K].view(b, K)
                    x.copy_(synth.activations(b, K, seed, synth.stream_id(CONFIG_ID, layer, mi, 2), device="cuda"))
                    xs.append(x)
                    ys.append(y_all[yo:yo + b * rows].view(b, rows))
                    xo += b * K
                    yo += b * rows
            self.io[b] = (x_all, y_all, xs, ys)
        torch.cuda.synchronize()

    def linears(self):
        for layer in range(self.layers):
            for name, rows, K in self.shapes:
                yield name, rows, K

    def sparse_ops(self, pattern, batch, only=None):
        _, _, xs, ys = self.io[batch]
        ops = []
        for i, (name, rows, K) in enumerate(self.linears()):
            if only and name != only:
                continue
            m, v = self.packed[pattern][i]
            ops.append(dict(masks=m, values=v, x=xs[i], y=ys[i], rows=rows, K=K))
        return ops

    def mlp_ops(self, batch):
        """The stack with each layer's MLP chained: gate_up with the SwiGLU epilogue writes h, and
        down reads h as its x (qkv and o keep their own x)."""
        _, _, xs, ys = self.io[batch]
        ops, i = [], 0
        for layer in range(self.layers):
            h = None
            for name, rows, K in self.shapes:
                if name == "gate_up":
                    m, v = self.swiglu[layer]
                    h = torch.empty(batch, rows // 2, dtype=torch.bfloat16, device="cuda")
                    ops.append(dict(masks=m, values=v, x=xs[i], y=h, rows=rows, K=K, flags=1))
                elif name == "down":
                    m, v = self.packed[self.patterns[0]][i]
                    ops.append(dict(masks=m, values=v, x=h, y=ys[i], rows=rows, K=K))
                else:
                    m, v = self.packed[self.patterns[0]][i]
                    ops.append(dict(masks=m, values=v, x=xs[i], y=ys[i], rows=rows, K=K))
                i += 1
        return ops

    def qkv_ops(self, batch, pattern, rows_q, rows_k):
        """The stack with every qkv linear storing q, k and v in three buffers of their own."""
        _, _, xs, ys = self.io[batch]
        ops = []
        for i, (name, rows, K) in enumerate(self.linears()):
            m, v = self.packed[pattern][i]
            if name == "qkv":
                y = ys[i]
                rows_v = rows - rows_q - rows_k
                flat = y.view(-1)
                q = flat[:batch * rows_q].view(batch, rows_q)
                k = flat[batch * rows_q:batch * (rows_q + rows_k)].view(batch, rows_k)
                vv = flat[batch * (rows_q + rows_k):].view(batch, rows_v)
                ops.append(dict(masks=m, values=v, x=xs[i], y=q, y_k=k, y_v=vv, rows=rows, K=K, flags=2,
                                rows_q=rows_q, rows_k=rows_k))
            else:
                ops.append(dict(masks=m, values=v, x=xs[i], y=ys[i], rows=rows, K=K))
        return ops

    def dense_ops(self, batch):
        _, _, xs, ys = self.io[batch]
        return [dict(W=self.dense[i], x=xs[i], y=ys[i], rows=rows, K=K)
                for i, (name, rows, K) in enumerate(self.linears())]

    def bytes(self, batch, dense=False, only=None):
        f = dense_bytes if dense else sparse_bytes
        return sum(f(rows, K, batch) for name, rows, K in self.linears() if not only or name == only)


def capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_graph(g, steps, warmup, world=1, sampler=None):
    """Device time of `steps` replays (CUDA events on the replay stream); returns (mean_ms, median_ms)."""
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        ev[0].record()
        for i in range(steps):
            g.replay()
            ev[i + 1].record()
        torch.cuda.synchronize()
    barrier(world)
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    time_graph.last = sorted(per)
    return ev[0].elapsed_time(ev[-1]) / steps, statistics.median(per)


def pct(sorted_vals, q):
    """q-quantile of an ascending list (nearest rank)."""
    return sorted_vals[min(len(sorted_vals) - 1, max(0, round(q * (len(sorted_vals) - 1))))]


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_peak():
    """Dense bf16 tensor TFLOP/s: the burst figure of MEASURED_PEAKS.json, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def recorded_traffic():
    """dram bytes per launch from the committed ncu summary, if the kernel is unchanged since."""
    try:
        fields = {}
        for line in open(PROFILE_SUMMARY):
            if ":" in line:
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
        sha = hashlib.sha256(b"".join(open(f, "rb").read() for f in KERNEL_SOURCES)).hexdigest()
        if fields.get("kernel_source_sha256") != sha:
            return None
        return float(fields["dram_bytes_per_launch"])
    except Exception:
        return None


# --- CPU oracle baseline -------------------------------------------------------------------------

def _bits(t: torch.Tensor):
    import numpy as np
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def build_oracle_sample(model, N, M, batch, row_frac, seed=0):
    import oracle
    shapes = synth.MODELS[model]
    sample = []
    for mi, name in enumerate(synth.MATRICES):
        rows, K = shapes[name]
        r = max(32, int(rows * row_frac))
        W = _bits(synth.weights(r, K, seed, synth.stream_id(CONFIG_ID, 0, mi, 0)))
        a = synth.col_norms(K, seed, synth.stream_id(CONFIG_ID, 0, mi, 1)).numpy()
        masks, values = oracle.pack(oracle.select(W, a, N, M), N, M)
        x = _bits(synth.activations(batch, K, seed, synth.stream_id(CONFIG_ID, 0, mi, 2)))
        sample.append((name, rows, r, K, masks, values, x))
    return sample


def time_oracle_token(sample, layers):
    """One oracle pass over the sample; returns (seconds, estimated seconds per decode token)."""
    import oracle
    t_sample = 0.0
    t_token = 0.0
    for name, rows, r, K, masks, values, x in sample:
        t0 = time.perf_counter()
        oracle.spmv_packed_f64(masks, values, x, K)
        dt = time.perf_counter() - t0
        t_sample += dt
        t_token += dt * (rows / r) * layers
    return t_sample, t_token


def time_oracle_token_threads(sample, layers, threads):
    """The same pass with each linear's sample rows split over `threads` threads (the
    oracle's C calls run without the GIL); returns estimated seconds per decode token."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    t_token = 0.0
    with ThreadPoolExecutor(threads) as ex:
        for name, rows, r, K, masks, values, x in sample:
            cuts = [r * i // threads for i in range(threads + 1)]
            parts = [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
            t0 = time.perf_counter()
            list(ex.map(lambda ab: oracle.spmv_packed_f64(masks[ab[0]:ab[1]], values[ab[0]:ab[1]], x, K), parts))
            t_token += (time.perf_counter() - t0) * (rows / r) * layers
    return t_token


def sample_desc(sample, layers, N, M, batch):
    parts = ", ".join(f"{name} {r}/{rows} rows x K={K}" for name, rows, r, K, *_ in sample)
    return (f"oracle (plain C, fp64, decode + dense product, 1 thread) on layer 0 of the stack: {parts}; "
            f"{N}:{M}, batch {batch}; time scaled by rows and by {layers} layers to one decode token")


def cpu_cores_available():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


# --- arms -------------------------------------------------------------------------------------------

def run_reference(args):
    """The CPU oracle as the reference arm: each step one bounded sample of the decode-token stack."""
    rank, world, _ = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), 0
    if rank != 0:
        return
    N, M = parse_pattern(args.pattern)
    layers = args.layers or synth.MODELS[args.model]["layers"]
    sample = build_oracle_sample(args.model, N, M, args.batch, row_frac=1 / 64)
    for _ in range(args.warmup):
        time_oracle_token(sample, layers)
    tokens = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        _, t_tok = time_oracle_token(sample, layers)
        tokens.append(t_tok)
    wall = time.perf_counter() - t_all
    us = statistics.mean(tokens) * 1e6
    desc = sample_desc(sample, layers, N, M, args.batch)
    out = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(args.model, N, M, args.batch, layers),
        "cpu_baseline": {"kind": "oracle", "value": us, "unit": UNIT, "cores": 1, "sample": desc},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def workload_config(model, N, M, batch, layers):
    shapes = synth.MODELS[model]
    lin = ", ".join(f"{n} {shapes[n][0]}x{shapes[n][1]}" for n in synth.MATRICES)
    return {"workload": f"{model}-shaped decode-token linear stack: {layers} layers x ({lin}), "
                        f"{N}:{M}, batch {batch}",
            "pattern": f"{N}:{M}", "batch": batch, "layers": layers, "launches_per_step": 4 * layers,
            "l2": "inputs larger than L2 (every step streams all weights of all layers)",
            "weights": "bf16 N(0,0.02^2), Wanda N:M selection with a=|N(1,0.3^2)|, packed on the GPU",
            "x": "bf16 N(0,1), independent per linear",
            "launch": "CUDA graph of PDL-chained launches (a prepared nm_stack_plan)"}


def obs_flops(rows, K):
    """Algorithmic fp32 flops of OBS N:M pruning of one 50% linear: Cholesky
    factorisation K^3/3 and triangular inverse K^3/3 of the (reversed) Hessian,
    and the compensations, 2 (K - 1 - j) flops for each of the rows K / 2
    removed weights, rows K^2 / 2 in all."""
    return 2 * K ** 3 / 3 + rows * K ** 2 / 2


def run_obs_pruning(nm, model, N, M, tokens=2048, repeats=2, cpu=True, linears=synth.MATRICES):
    """Prune one decoder layer by the OBS rule and pack it: for each linear the
    calibration Hessian H = 2 X^T X of its own synthetic inputs, the pruning,
    and the bitmask pack. nm_obs_prune is synchronous, so event and wall time
    agree; each linear takes the best of `repeats` after one untimed run."""
    shapes = [(mi, n, synth.MODELS[model][n]) for mi, n in enumerate(synth.MATRICES) if n in linears]
    per, hess_ms, total_flops = {}, 0.0, 0.0
    for mi, name, (rows, K) in shapes:
        W = synth.weights(rows, K, seed=7, stream=synth.stream_id(9, 0, mi, 0), device="cuda")
        X = synth.calibration(tokens, K, seed=7, stream=synth.stream_id(9, 0, mi, 3), device="cuda")
        H = nm.obs_hessian(X)
        best = None
        for it in range(repeats + 1):
            torch.cuda.synchronize()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            e[0].record()
            nm.obs_hessian(X, H)
            e[1].record()
            Wp, _, _ = nm.obs_prune(W, H, N, M, masks=False)
            e[2].record()
            masks, values = nm.pack(Wp, N, M)
            e[3].record()
            torch.cuda.synchronize()
            t = [e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2]), e[2].elapsed_time(e[3])]
            if it > 0 and (best is None or sum(t) < sum(best)):
                best = t
        f = obs_flops(rows, K)
        total_flops += f
        hess_ms += best[0]
        per[name] = {"rows": rows, "K": K, "hessian_ms": round(best[0], 3), "prune_ms": round(best[1], 3),
                     "pack_ms": round(best[2], 3),
                     "fp32_tflops_effective": round(f / (best[1] * 1e-3) / 1e12, 2)}
        del W, X, H, Wp, masks, values
    total_ms = sum(v["hessian_ms"] + v["prune_ms"] + v["pack_ms"] for v in per.values())
    bf16, bf16_kind = measured_bf16_peak()
    emu_peak = bf16 / 6.0  # six bf16 products per emulated fp32 product (tc_gemm.cu)
    achieved = total_flops / (sum(v["prune_ms"] for v in per.values()) * 1e-3) / 1e12
    out = {"workload": f"{'one ' + model + ' decoder layer' if len(per) == 4 else model + ' ' + ', '.join(per)} "
                       f"pruned {N}:{M} by the OBS rule, each linear against the "
                       f"Hessian of {tokens} synthetic calibration tokens, then packed",
           "ms_per_layer": round(total_ms, 2), "hessian_ms": round(hess_ms, 3),
           "fp32_tflops_effective": round(total_flops / (sum(v["prune_ms"] for v in per.values()) * 1e-3) / 1e12, 2),
           "algorithmic_flops": f"{total_flops:.4g} (2 K^3 / 3 + rows K^2 / 2 per linear)",
           "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(emu_peak, 1),
                        "unit": "TFLOP/s", "frac": round(achieved / emu_peak, 4),
                        "frac_of_9_product_ceiling": round(achieved / (bf16 / 9.0), 4),
                        "peak_basis": f"{bf16_kind} bf16 {bf16} TFLOP/s / 6 (fp32 emulated on the bf16 tensor "
                                      "cores, six bf16 products per fp32 product); frac_of_9_product_ceiling: "
                                      "against bf16 / 9, the ceiling of the nine-product emulation; achieved = "
                                      "algorithmic fp32 flops / event-timed prune time"},
           "per_linear": per}
    if cpu:
        sys.path.insert(0, ROOT)
        from oracle import obs
        rows, K = synth.MODELS[model]["o"]
        Wc = synth.weights(64, K, seed=7).float().numpy().astype("float64")
        Xc = _bits(synth.calibration(tokens, K, seed=7))
        t0 = time.perf_counter()
        Hc = obs.hessian_f64(Xc)
        t1 = time.perf_counter()
        obs.obs_prune_f64(Wc, Hc, N, M)
        t2 = time.perf_counter()
        out["cpu_oracle"] = {"hessian_s": round(t1 - t0, 2), "prune_s": round(t2 - t1, 2),
                             "sample": f"o linear ({rows}x{K}): 64 of its {rows} rows, fp64 numpy "
                                       f"(factorisation of the whole {K}x{K} Hessian included)",
                             "cores": cpu_cores_available()}
    return out


def time_select_pack(nm, model, pattern, world, layers=1, reps=5):
    """nm_select_pack (Wanda selection and bitmask pack in one pass) on `layers` decoder
    layers' linears: ms per layer and the bytes it moves (W read, masks and values written)."""
    N, M = pattern
    shapes = [(synth.MODELS[model][n]) for n in synth.MATRICES]
    Ws, As = [], []
    for li in range(layers):
        for mi, (rows, K) in enumerate(shapes):
            Ws.append(synth.weights(rows, K, 5, synth.stream_id(11, li, mi, 0), device="cuda"))
            As.append(synth.col_norms(K, 5, synth.stream_id(11, li, mi, 1), device="cuda"))
    outs = [(torch.empty(W.shape[0], W.shape[1] // 32, dtype=torch.int32, device="cuda"),
             torch.empty(W.shape[0], W.shape[1] // 2, dtype=torch.bfloat16, device="cuda")) for W in Ws]
    L = nm.lib()

    def run():
        s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        for W, a, (m, v) in zip(Ws, As, outs):
            assert L.nm_select_pack(W.data_ptr(), a.data_ptr(), W.shape[0], W.shape[1], N, M, m.data_ptr(),
                                    v.data_ptr(), s) == 0
    g = capture(run)
    t, _ = time_graph(g, reps, 2, world)
    by = sum(W.numel() * 2 + W.numel() // 8 + W.numel() for W in Ws) + sum(a.numel() * 4 for a in As)
    peak = measured_peak()[0]
    del g, Ws, As, outs
    return {"workload": f"{layers} {model} decoder layer(s): qkv, o, gate_up, down, {N}:{M}",
            "ms_per_layer": round(t / layers, 4), "GB_s": round(by / (t * 1e-3) / 1e9, 1),
            "frac_of_measured_peak": round(by / (t * 1e-3) / 1e9 / peak, 4),
            "bytes": f"{by} (W read once; masks and values written)"}


def splitk_compare(nm, stack, pattern, world, steps, warmup):
    """The two ways to combine a row block split over CTAs, fp32 output: the
    default deterministic fix-up (the last CTA adds the parts in CTA order) and
    the split reduction with atomicAdd (every CTA of the layer's split adds its
    part into the zeroed y). Each timing runs the layers' own weights of one
    shape in one graph."""
    out = {}
    for name in ("o", "down"):
        idx = [i for i, (n, _, _) in enumerate(stack.linears()) if n == name]
        rows, K = synth.MODELS[stack.model][name]
        for b in (1, 8):
            xs = [synth.activations(b, K, 3, synth.stream_id(CONFIG_ID, li, 9, 2), device="cuda")
                  for li in range(len(idx))]
            ys = [torch.empty(b, rows, dtype=torch.float32, device="cuda") for _ in idx]
            res = {}
            for atomic in (False, True):
                def run(atomic=atomic):
                    for j, i in enumerate(idx):
                        m, v = stack.packed[pattern][i]
                        nm.spmv(m, v, xs[j], out=ys[j], f32=True, atomic=atomic)
                g = capture(run)
                t, _ = time_graph(g, steps, warmup, world)
                res["atomic" if atomic else "deterministic"] = t * 1e3 / len(idx)
                del g
            by = sparse_bytes(rows, K, b) + 2 * rows * b  # fp32 y: 2 more bytes per output than bf16
            peak = measured_peak()[0]
            out[f"{name} {rows}x{K} batch {b}"] = {
                "deterministic_us": round(res["deterministic"], 3), "atomic_us": round(res["atomic"], 3),
                "deterministic_GB_s": round(by / (res["deterministic"] * 1e-6) / 1e9, 1),
                "atomic_GB_s": round(by / (res["atomic"] * 1e-6) / 1e9, 1),
                "frac_of_measured_peak": {"deterministic": round(by / (res["deterministic"] * 1e-6) / 1e9 / peak, 4),
                                          "atomic": round(by / (res["atomic"] * 1e-6) / 1e9 / peak, 4)}}
            del xs, ys
    return out


SUITE = [("qwen3-14b", ((4, 8), (8, 16)), (1,)), ("qwen3-32b", ((4, 8), (8, 16)), (1,)),
         ("llama3.3-70b", ((2, 4), (16, 32)), (1, 2, 4, 8))]


def run_suite(args):
    """The larger stacks of the pages' Table 3 models, each against its dense references
    at the same batch. One pattern's packed weights are resident at a time (with the
    dense weights, the 70B stack needs 137 + 77 GB)."""
    torch.cuda.set_device(0)
    import sparse_decoding_gb300 as nm
    nm.init()
    peak, peak_kind = measured_peak()
    steps, warm = args.steps, min(args.warmup, 10)
    sampler = ClockSampler(0)
    out = {"metric": METRIC, "unit": UNIT, "peak": {"GB_s": peak, "source": f"{peak_kind} hbm_gbs"}, "models": {}}

    def time_plan(ops, b, dense=False):
        pl = nm.StackPlan(ops, b, dense=dense)
        g = capture(pl.run)
        t, _ = time_graph(g, steps, warm)
        del g
        pl.close()
        return t

    with sampler:
        for model, pats, batches in SUITE:
            stack = Stack(nm, model, [pats[0]], batches, args.layers, keep_dense=True, swiglu=False)
            res = {"layers": stack.layers, "dense": {}, "patterns": {}}
            for b in batches:
                dops = stack.dense_ops(b)

                def cublas(dops=dops):
                    for op in dops:
                        torch.mm(op["x"], op["W"].t(), out=op["y"])
                g = capture(cublas)
                tc, _ = time_graph(g, steps, warm)
                del g
                td = time_plan(dops, b, dense=True)
                res["dense"][f"batch {b}"] = {"hand_written_us": round(td * 1e3, 2), "cublas_us": round(tc * 1e3, 2),
                                              "GB_s": round(stack.bytes(b, dense=True) / (min(td, tc) * 1e-3) / 1e9, 1)}
            for pi, pat in enumerate(pats):
                if pi > 0:  # the next pattern, packed from the same W after the previous one is freed
                    stack.packed = {pat: []}
                    torch.cuda.empty_cache()
                    for i, (name, rows, K) in enumerate(stack.linears()):
                        layer, mi = divmod(i, 4)
                        a = synth.col_norms(K, 0, synth.stream_id(CONFIG_ID, layer, mi, 1), device="cuda")
                        stack.packed[pat].append(nm.select_pack(stack.dense[i], a, *pat))
                # selection + pack of the whole stack in one pass per linear
                As = [synth.col_norms(K, 0, synth.stream_id(CONFIG_ID, i // 4, i % 4, 1), device="cuda")
                      for i, (_, _, K) in enumerate(stack.linears())]
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for i, W in enumerate(stack.dense):
                    m, v = stack.packed[pat][i]
                    assert nm.lib().nm_select_pack(W.data_ptr(), As[i].data_ptr(), W.shape[0], W.shape[1], *pat,
                                                   m.data_ptr(), v.data_ptr(),
                                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
                e1.record()
                torch.cuda.synchronize()
                del As
                sp_ms = e0.elapsed_time(e1)
                entry = {"select_pack_ms_whole_stack": round(sp_ms, 2)}
                for b in batches:
                    t = time_plan(stack.sparse_ops(pat, b), b)
                    by = stack.bytes(b)
                    d = res["dense"][f"batch {b}"]
                    best = min(d["hand_written_us"], d["cublas_us"])
                    entry[f"batch {b}"] = {"us_per_token": round(t * 1e3, 2), "GB_s": round(by / (t * 1e-3) / 1e9, 1),
                                           "frac_of_measured_peak": round(by / (t * 1e-3) / 1e9 / peak, 4),
                                           "ratio_vs_best_dense": round(best / (t * 1e3), 4)}
                res["patterns"][f"{pat[0]}:{pat[1]}"] = entry
            shp = synth.MODELS[model]
            res["workload"] = (f"{model}-shaped decode-token linear stack: {stack.layers} layers x ("
                               + ", ".join(f"{n} {shp[n][0]}x{shp[n][1]}" for n in synth.MATRICES) + ")")
            # the CPU oracle beside it: one layer's sampled rows, scaled to the stack (extrapolated)
            N0, M0 = pats[0]
            sample = build_oracle_sample(model, N0, M0, 1, row_frac=1 / 64)
            t_tok = min(time_oracle_token(sample, stack.layers)[1] for _ in range(2))
            cores = cpu_cores_available()
            t_all = time_oracle_token_threads(sample, stack.layers, cores)
            res["cpu_oracle_extrapolated"] = {
                "us_per_token": round(t_tok * 1e6, 1), "cores": 1,
                "all_cores_us_per_token": round(t_all * 1e6, 1), "all_cores": cores,
                "sample": sample_desc(sample, stack.layers, N0, M0, 1) + " (extrapolated from one layer)"}
            out["models"][model] = res
            del stack
            torch.cuda.empty_cache()
    out["clocks"] = sampler.summary()
    out["device_status"] = nm.status_str(nm.device_status())
    out["data"] = "synthetic"
    print(json.dumps(out), flush=True)


def run_ours(args):
    rank, world, local = dist_init()
    torch.cuda.set_device(local)
    import sparse_decoding_gb300 as nm
    nm.init()
    N, M = parse_pattern(args.pattern)
    head = (N, M)
    patterns = [head]
    if not args.no_variants:
        patterns += [p for p in synth.PATTERNS if p != head]
    batches = [args.batch] + ([] if args.no_variants else [b for b in (2, 4, 8) if b != args.batch])
    stack = Stack(nm, args.model, patterns, batches, args.layers, keep_dense=True)
    layers = stack.layers
    B = args.batch

    # headline: the sparse stack, 4*layers kernels chained with programmatic
    # dependent launch (a prepared plan), replayed from a CUDA graph
    sparse_ops = stack.sparse_ops(head, B)
    plan = nm.StackPlan(sparse_ops, B)
    g_sparse = capture(plan.run)
    sampler = ClockSampler(local)
    ms_mean, ms_med = time_graph(g_sparse, args.steps, args.warmup, world, sampler)
    per_step = time_graph.last
    ms_max = max_over_ranks(ms_mean, world)
    value = job_us_per_token(ms_max, world)

    step_bytes = stack.bytes(B)
    achieved = step_bytes / (ms_mean * 1e-3) / 1e9
    peak, peak_kind = measured_peak()

    # the same stack as one persistent launch (grid barrier between ops)
    pplan = nm.StackPlan(sparse_ops, B, persistent=True)
    g_pers = capture(pplan.run)
    pers_ms, _ = time_graph(g_pers, args.steps, args.warmup, world)
    del g_pers
    pplan.close()

    # dense references: the hand-written GEMV (PDL chain and persistent) and cuBLAS
    dense_ops = stack.dense_ops(B)
    dense_plan = nm.StackPlan(dense_ops, B, dense=True)
    g_dense = capture(dense_plan.run)
    dense_ms, _ = time_graph(g_dense, args.steps, args.warmup, world)
    del g_dense
    dense_plan.close()
    dense_pplan = nm.StackPlan(dense_ops, B, dense=True, persistent=True)
    g_dpers = capture(dense_pplan.run)
    dense_pers_ms, _ = time_graph(g_dpers, args.steps, args.warmup, world)
    del g_dpers
    dense_pplan.close()

    def cublas_stack():
        for op in dense_ops:
            torch.mm(op["x"], op["W"].t(), out=op["y"])
    g_cublas = capture(cublas_stack)
    cublas_ms, _ = time_graph(g_cublas, args.steps, args.warmup, world)
    del g_cublas
    best_dense = min(dense_ms, dense_pers_ms, cublas_ms)

    # per-shape kernel bandwidth (one chained plan per shape, over all layers)
    per_shape = {}
    for name, rows, K in stack.shapes:
        ops = stack.sparse_ops(head, B, only=name)
        pl = nm.StackPlan(ops, B)
        g = capture(pl.run)
        t, _ = time_graph(g, max(5, args.steps // 5), 3, world)
        per_op_us = t * 1e3 / len(ops)
        per_shape[name] = {"rows": rows, "K": K, "us_per_op": round(per_op_us, 3),
                           "GB_s": round(sparse_bytes(rows, K, B) / (per_op_us * 1e-6) / 1e9, 1)}
        del g
        pl.close()

    def time_plan(ops, b, dense=False):
        pl = nm.StackPlan(ops, b, dense=dense)
        g = capture(pl.run)
        t, _ = time_graph(g, args.steps, min(args.warmup, 10), world)
        del g
        pl.close()
        return t

    def variant_entry(t, b, dense_t=None):
        by = stack.bytes(b)
        e = {"us_per_token": round(t * 1e3, 2), "GB_s": round(by / (t * 1e-3) / 1e9, 1),
             "frac_of_measured_peak": round(by / (t * 1e-3) / 1e9 / peak, 4)}
        if dense_t is not None:
            e["dense_us_per_token"] = {k: round(v * 1e3, 2) for k, v in dense_t.items()}
            e["ratio_vs_best_dense"] = round(min(dense_t.values()) / t, 4)
        return e

    variants = {}
    if not args.no_variants:
        # every pattern at the headline batch (the pages: the same traffic for all four)
        for pat in patterns[1:]:
            variants[f"{pat[0]}:{pat[1]} batch {B}"] = variant_entry(time_plan(stack.sparse_ops(pat, B), B), B)
        # batch 2, 4 and 8, each with the dense references at that batch
        for bb in (2, 4, 8):
            if bb not in stack.io or bb == B:
                continue
            tb = time_plan(stack.sparse_ops(head, bb), bb)
            dense_ops = stack.dense_ops(bb)
            db = {"hand_written": time_plan(dense_ops, bb, dense=True)}

            def cublas_b(dense_ops=dense_ops):
                for op in dense_ops:
                    torch.mm(op["x"], op["W"].t(), out=op["y"])
            g = capture(cublas_b)
            db["cublas"], _ = time_graph(g, args.steps, min(args.warmup, 10), world)
            del g
            variants[f"{head[0]}:{head[1]} batch {bb}"] = variant_entry(tb, bb, db)
        # q, k and v stored apart (three buffers per qkv linear)
        rq, rk = synth.QKV_SPLIT[args.model]
        for b in sorted({B} | ({4} if 4 in stack.io else set())):
            variants[f"{head[0]}:{head[1]} batch {b}, qkv stored as q, k, v ({rq}/{rk}/{rk} rows)"] = \
                variant_entry(time_plan(stack.qkv_ops(b, head, rq, rk), b), b)
        # the MLP chained as in a decode layer: gate_up + SwiGLU epilogue -> h -> down
        ops = stack.mlp_ops(B)
        pl = nm.StackPlan(ops, B)
        g = capture(pl.run)
        t, _ = time_graph(g, args.steps, min(args.warmup, 10), world)
        by = stack.bytes(B)
        variants[f"{head[0]}:{head[1]} batch {B}, gate_up with SwiGLU epilogue feeding down"] = {
            "us_per_token": round(t * 1e3, 2), "GB_s": round(by / (t * 1e-3) / 1e9, 1),
            "frac_of_measured_peak": round(by / (t * 1e-3) / 1e9 / peak, 4)}
        del g
        pl.close()

    split_k = None
    if not args.no_variants:
        split_k = splitk_compare(nm, stack, head, world, max(5, args.steps // 2), min(args.warmup, 5))

    # Wanda selection + pack fused in one pass, for one decoder layer's four linears
    select_pack = time_select_pack(nm, args.model, head, world)

    pruning = None
    if world == 1 and not args.no_pruning:
        pruning = run_obs_pruning(nm, args.model, N, M, cpu=(world == 1 and not args.no_cpu_baseline))

    # end to end through the public API: pinned host x in, stack, host y out, every step
    x_all, y_all, _, _ = stack.io[B]
    x_host = torch.empty(x_all.shape, dtype=x_all.dtype, pin_memory=True)
    x_host.copy_(x_all)
    y_host = torch.empty(y_all.shape, dtype=y_all.dtype, pin_memory=True)

    def e2e_step():
        x_all.copy_(x_host, non_blocking=True)
        plan.run()
        y_host.copy_(y_all, non_blocking=True)
    for _ in range(min(args.warmup, 10)):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record()
    for _ in range(args.steps):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    e2e_wall = (time.perf_counter() - t0) / args.steps * 1e3
    e2e_ms = max_over_ranks(max(e0.elapsed_time(e1) / args.steps, e2e_wall), world)

    status = nm.device_status()

    out = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max, 5), "median_ms_per_step": round(ms_med, 5),
        "p10_ms_per_step": round(pct(per_step, 0.1), 5), "p90_ms_per_step": round(pct(per_step, 0.9), 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_config(args.model, N, M, B, layers),
        "hbm_GB_s": round(achieved, 1),
        "persistent_us_per_token": round(pers_ms * 1e3, 2),
        "x_vs_dense": {"hand_written_dense_us": round(dense_ms * 1e3, 2),
                       "hand_written_dense_persistent_us": round(dense_pers_ms * 1e3, 2),
                       "cublas_dense_us": round(cublas_ms * 1e3, 2),
                       "ratio_vs_best_dense": round(best_dense / ms_mean, 4),
                       "dense_GB_s": round(stack.bytes(B, dense=True) / (best_dense * 1e-3) / 1e9, 1)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": recorded_traffic(),
                     "kernel": "streamk_kernel<SparseUnit>",
                     "achieved_basis": f"{step_bytes} algorithmic bytes per step / {4 * layers} launches, "
                                       "over the event-timed step (gaps between launches included)"},
        "per_shape": per_shape,
        "variants": variants,
        "split_k_combine": split_k,
        "select_pack": select_pack,
        "obs_pruning": pruning,
        "e2e": {"value": round(job_us_per_token(e2e_ms, world), 3), "unit": UNIT,
                "h2d_bytes_per_step": x_all.numel() * 2, "d2h_bytes_per_step": y_all.numel() * 2,
                "path": "pinned host x -> device, nm_stack_plan_run through the C ABI (the plan launches the CUDA graph of its chain captured at creation), y -> pinned host"},
        "gpu_launches": 4 * layers * args.steps,
        "clocks": sampler.summary(),
        "device_status": nm.status_str(status),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = build_oracle_sample(args.model, N, M, B, row_frac=1 / 8)
        ts = []
        t_all = time.perf_counter()
        while True:
            t_sample, t_tok = time_oracle_token(sample, layers)
            ts.append(t_tok)
            if len(ts) >= 3 or time.perf_counter() - t_all > 20:
                break
        cores = cpu_cores_available()
        t_all_cores = min(time_oracle_token_threads(sample, layers, cores) for _ in range(2))
        out["cpu_baseline"] = {"value": round(statistics.median(ts) * 1e6, 1), "unit": UNIT, "cores": 1,
                               "kind": "oracle", "sample": sample_desc(sample, layers, N, M, B),
                               "host_cores_available": cores, "repeats": len(ts),
                               "all_cores": {"value": round(t_all_cores * 1e6, 1), "unit": UNIT, "cores": cores,
                                             "how": "the same sample, each linear's rows split over one thread "
                                                    "per core (best of 2)"}}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.only_pruning:
        import sparse_decoding_gb300 as nm
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        nm.init()
        N, M = parse_pattern(args.pattern)
        out = run_obs_pruning(nm, args.model, N, M, repeats=args.prune_repeats, cpu=not args.no_cpu_baseline,
                              linears=tuple(args.prune_linears.split(",")))
        print(json.dumps({"obs_pruning": out}), flush=True)
        return
    if args.suite:
        run_suite(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
