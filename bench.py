#!/usr/bin/env python3
"""Benchmark of the GB300 W4A16 layer (one JSON line on stdout, rank 0).

Headline step: one decode pass of the LLaMA-3-8B projections -- (K, N) = (4096, 6144)
fused QKV, (4096, 4096) O, (4096, 28672) fused gate+up, (14336, 4096) down -- at each of
M = 1, 4, 16, INT4 group-128 weights, through the dispatching entry point wq_gemm_w4a16
(12 layer calls).  Metric: algorithmic bytes (0.53125 B/weight + 2MK + 2MN per call) per
second.  Inputs are synthetic and seeded; three copies of the packed weights rotate so
that every step streams 348 MB (> the 129 MB L2).  The step is replayed from a CUDA graph
and timed with CUDA events on its stream.

Secondary measurements in the same run (same JSON line): prefill GEMM TFLOP/s on the
Qwen2.5-72B shapes at M = 2048 and M = 8192, MXFP4 decode, the fused gate+up projection with
its SwiGLU epilogue and the fused QKV projection with its Q/K/V split (decode and prefill,
each beside the plain projection), the quantize kernels, GPTQ (sweep, on-device factor, end
to end from calibration activations), AWQ, and the GEMV/GEMM crossover on K = N = 8192 plus
the decode shapes, whose crossover points become the dispatch thresholds of the run.

--impl reference times the CPU oracle (test infrastructure, float64) on a bounded sample
of the same workload on all host cores (the BLAS thread pool of the matmul).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A16 decode GEMV HBM GB/s (% of peak); prefill GEMM TFLOPS (% bf16 peak)"
DECODE_SHAPES = [(4096, 6144), (4096, 4096), (4096, 28672), (14336, 4096)]   # (K, N)
DECODE_M = (1, 4, 16)
PREFILL_SHAPES = [(8192, 10240), (8192, 8192), (8192, 59136), (29568, 8192)]
PREFILL_M = 2048
PREFILL_M_LARGE = 8192
CROSS_M = (1, 2, 4, 8, 16, 24, 32, 48, 64, 128, 256, 512, 1024, 2048)
DECODE_MAX_M = 64          # activation rows the decode kernel accepts
THRESH_M = (16, 24, 32, 48, 64)   # the crossover points measured on each decode shape
COPIES = 3
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0


def decode_bytes(M, K, N):
    return 0.53125 * N * K + 2.0 * M * K + 2.0 * M * N


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def src_hash(name):
    p = os.path.join(ROOT, "bit_weight_quantized_wq_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profile_traffic(kernel_file, key):
    """Per-launch DRAM bytes recorded from an ncu capture (profiles/traffic.json), or None
    when the kernel source changed since the capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        e = d[key]
        if e.get("src_sha256_16") != src_hash(kernel_file):
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ----------------------------------------------------------------------------------- ranks
def max_over_ranks(value, device=None):
    """The largest of every rank's value (a no-op without an initialised process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, step_bytes, steps, ms_max):
    """Whole-job GB/s: every rank streams step_bytes per step; time is the slowest rank's."""
    return world * step_bytes * steps / (ms_max * 1e-3) / 1e9


# ----------------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", "wq_clocks_%d_%d.csv" % (os.getpid(), index))

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons, n = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 7:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx = float(parts[1])
                except ValueError:
                    continue
                n += 1
                for nm, v in zip(names, parts[3:7]):
                    if v.lower() in ("active", "1"):
                        reasons.add(nm)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": n}


# ----------------------------------------------------------------------------------- CPU oracle
def host_threads():
    """The host cores this process may run on, and the threads the BLAS pool of the oracle's
    matmul uses (threadpoolctl where installed, else the OpenMP/BLAS environment)."""
    cores = len(os.sched_getaffinity(0))
    used = None
    try:
        from threadpoolctl import threadpool_info
        used = max((d.get("num_threads", 0) for d in threadpool_info() if d.get("user_api") == "blas"), default=None)
    except Exception:
        pass
    if not used:
        used = int(os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS") or cores)
    return cores, used


def oracle_sample(seconds_budget, steps=1):
    """Times the float64 oracle on a bounded sample of the decode workload (all host cores:
    the matmul runs on the BLAS thread pool; the dequantization is numpy elementwise code).

    Returns (algorithmic bytes processed, seconds, description).  The sample: for each of the
    12 layer calls, the first R weight rows (output columns) -- dequantize them and multiply."""
    import numpy as np

    from bit_weight_quantized_wq_gb300 import inputs
    from oracle import int4_g128, linear

    rows = 64
    packs = []
    for i, (K, N) in enumerate(DECODE_SHAPES):
        W = inputs.weights(1000 + i, rows, K, 0.02)
        packs.append((K, N, int4_g128.quantize(W)))
    xs = {(M, K): inputs.activations(M * 100 + K, M, K)[1] for M in DECODE_M for K, _ in DECODE_SHAPES}

    def one_pass(r):
        b = 0.0
        for M in DECODE_M:
            for K, N, pk in packs:
                Wq, s, z = pk[0][:r], pk[1][:r], pk[2][:r]
                y = linear.linear_w4a16("int4_g128", xs[(M, K)], Wq, s, z)
                b += 0.53125 * r * K + 2.0 * M * K + 2.0 * M * r
                assert np.isfinite(y).all()
        return b

    t0 = time.perf_counter()
    one_pass(4)
    t_small = max(time.perf_counter() - t0, 1e-4)
    r = int(max(1, min(rows, 4 * seconds_budget / (t_small * steps))))
    total_b, t = 0.0, 0.0
    for _ in range(steps):
        t0 = time.perf_counter()
        total_b += one_pass(r)
        t += time.perf_counter() - t0
    desc = ("float64 oracle (dequantize + matmul) on the first %d weight rows of each of the 12 decode "
            "calls (LLaMA-3-8B projections x M in {1,4,16}), %d pass(es)" % (r, steps))
    return total_b, t, desc


def _all_core_env():
    n = str(len(os.sched_getaffinity(0)))
    return dict(os.environ, OMP_NUM_THREADS=n, OPENBLAS_NUM_THREADS=n, MKL_NUM_THREADS=n)


def cpu_baseline_subprocess(budget):
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample", str(budget)], env=_all_core_env(),
                       capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return {"value": None, "unit": "GB/s", "cores": None, "kind": "oracle", "sample": "failed: " + r.stderr[-300:]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": d["bytes"] / d["seconds"] / 1e9, "unit": "GB/s", "cores": d["threads"],
            "host_cores": d["cores"], "kind": "oracle", "sample": d["desc"]}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    if os.environ.get("WQ_BENCH_CPU_CHILD") != "1":
        # the BLAS pool sizes itself at import: run the timing in a child with all cores set
        env = dict(_all_core_env(), WQ_BENCH_CPU_CHILD="1")
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--impl", "reference", "--gpus", str(args.gpus),
                            "--steps", str(args.steps), "--warmup", str(args.warmup)], env=env)
        return r.returncode
    budget = 150.0 / max(1, args.steps + args.warmup)
    # warm-up passes (untimed), then K timed passes, each a bounded sample
    for _ in range(args.warmup):
        oracle_sample(budget, 1)
    tb, tt = 0.0, 0.0
    desc = ""
    for _ in range(args.steps):
        b, t, desc = oracle_sample(budget, 1)
        tb += b
        tt += t
    v = tb / tt / 1e9
    cores, threads = host_threads()
    out = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tt / max(1, args.steps),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded normal weights with 1% x10 outlier input columns; N(0,1) bf16 activations)",
           "config": {"workload": "decode: LLaMA-3-8B projections (K,N) in {(4096,6144),(4096,4096),(4096,28672),"
                                  "(14336,4096)} x M in {1,4,16}, INT4 g128 asym (bounded row sample on CPU)"},
           "cpu_baseline": {"value": v, "unit": "GB/s", "cores": threads, "host_cores": cores, "kind": "oracle",
                            "sample": desc},
           "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))
    return 0


# ----------------------------------------------------------------------------------- GPU arm
def run_ours(args):
    import numpy as np
    import torch

    from bit_weight_quantized_wq_gb300 import binding, inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    binding.check_device()
    hbm_peak, bf16_peak, bf16_sus, peak_kind = peaks()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    def dev_x(M, K, seed):
        xb, _ = inputs.activations(seed, M, K)
        return torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)

    # ---------------- headline workload: decode, INT4 g128, 3 weight copies
    layers = []        # per shape: list of COPIES (Wq, s, z)
    quant_t = []       # quantize timing (a1)
    for i, (K, N) in enumerate(DECODE_SHAPES):
        W = torch.from_numpy(inputs.weights(1000 + i, N, K, 0.02)).to(dev)
        Wq, s, z = binding.quantize_int4_g128(W)
        copies = [(Wq, s, z)] + [(Wq.clone(), s.clone(), z.clone()) for _ in range(COPIES - 1)]
        layers.append(copies)
        del W
    X = {(M, K): dev_x(M, K, M * 100 + K) for M in DECODE_M for K, _ in DECODE_SHAPES}
    Y = {(M, N): torch.empty((M, N), dtype=torch.bfloat16, device=dev) for M in DECODE_M for _, N in DECODE_SHAPES}
    ws = binding.Workspace(dev)
    ws_buf = ws.get(max(binding.gemm_workspace_bytes("int4_g128", M, K, N) for M in DECODE_M for K, N in DECODE_SHAPES))
    stream = torch.cuda.Stream(device=dev)

    def step():
        for ci, M in enumerate(DECODE_M):
            for li, (K, N) in enumerate(DECODE_SHAPES):
                Wq, s, z = layers[li][ci % COPIES]
                binding.gemm_w4a16("int4_g128", X[(M, K)], Wq, s, z, out=Y[(M, N)], workspace=ws_buf)

    step_bytes = sum(decode_bytes(M, K, N) for M in DECODE_M for K, N in DECODE_SHAPES)
    launches_per_step = len(DECODE_M) * len(DECODE_SHAPES)
    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        for _ in range(args.warmup):
            g.replay()
    torch.cuda.synchronize(dev)

    clk = ClockSampler(local)
    clk.start()
    barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clocks = clk.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), dev)
    value = replica_throughput(world, step_bytes, args.steps, ms)
    ms_step = ms / args.steps

    # ---------------- e2e through the public API with host buffers (no graph)
    # Every step: one copy of all twelve calls' activations from pinned host memory, the twelve
    # calls, one copy of all their outputs back to pinned host memory, then a host sync.  The
    # device buffers are 256-byte-aligned views into one input and one output block.
    def _pack_views(shapes):
        offs, total = [], 0
        for shp in shapes:
            offs.append(total)
            total += ((shp[0] * shp[1] * 2 + 255) // 256) * 256
        return offs, total

    x_keys = [(M, K) for M in DECODE_M for K, _ in DECODE_SHAPES]
    y_keys = [(M, N) for M in DECODE_M for _, N in DECODE_SHAPES]
    x_offs, x_total = _pack_views(x_keys)
    y_offs, y_total = _pack_views(y_keys)
    dx = torch.empty(x_total, dtype=torch.uint8, device=dev)
    dy = torch.empty(y_total, dtype=torch.uint8, device=dev)
    hx = torch.empty(x_total, dtype=torch.uint8).pin_memory()
    hy = torch.empty(y_total, dtype=torch.uint8).pin_memory()
    xv, yv = [], []
    for (M, K), o in zip(x_keys, x_offs):
        v = dx[o:o + 2 * M * K].view(torch.bfloat16).view(M, K)
        v.copy_(X[(M, K)])
        xv.append(v)
    for (M, N), o in zip(y_keys, y_offs):
        yv.append(dy[o:o + 2 * M * N].view(torch.bfloat16).view(M, N))
    hx.copy_(dx)
    e2e_steps = max(3, min(args.steps, 200))
    h2d = sum(2 * M * K for M, K in x_keys)
    d2h = sum(2 * M * N for M, N in y_keys)
    calls = []
    for ci, M in enumerate(DECODE_M):
        for li, (K, N) in enumerate(DECODE_SHAPES):
            Wq, s, z = layers[li][ci % COPIES]
            calls.append((xv[ci * len(DECODE_SHAPES) + li], Wq, s, z, yv[ci * len(DECODE_SHAPES) + li]))

    def e2e_step():
        dx.copy_(hx, non_blocking=True)
        for (xa, Wq, s, z, ya) in calls:
            binding.gemm_w4a16("int4_g128", xa, Wq, s, z, out=ya, workspace=ws_buf)
        hy.copy_(dy, non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()

    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
        barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        t_e2e = time.perf_counter() - t0
    e2e_value = world * step_bytes * e2e_steps / t_e2e / 1e9
    del hx, hy, dx, dy

    result = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded normal weights, sigma 0.02, 1% x10 outlier input columns; N(0,1) bf16 "
                "activations)",
        "config": {"workload": "decode: LLaMA-3-8B projections (K,N) in {(4096,6144),(4096,4096),(4096,28672),"
                               "(14336,4096)} x M in {1,4,16}, INT4 g128 asym, via wq_gemm_w4a16",
                   "global_batch": list(DECODE_M), "l2": "inputs larger than L2: 3 rotating weight copies, "
                   "%.0f MB streamed per step vs 129 MB L2" % (step_bytes / 1e6),
                   "graph": "CUDA graph of the 12 calls, replayed per step", "parallelism": "replicas" if world > 1 else "single GPU"},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"bound": "hbm", "achieved": value / world, "peak": hbm_peak, "unit": "GB/s",
                     "frac": value / world / hbm_peak,
                     "traffic": profile_traffic("gemv.cu", "gemv_decode_step_avg"),
                     "peak_kind": peak_kind + " (copy bandwidth, MEASURED_PEAKS.json hbm_gbs)",
                     "note": "dominant kernel = decode GEMV (all 12 launches); achieved = algorithmic bytes per "
                             "launch / average launch duration over the timed region"},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "public API (binding.gemm_w4a16) without graph capture; every step copies all twelve "
                       "calls' X in from pinned host memory (one copy) and all their Y out (one copy); "
                       "wall-clock over %d steps incl. the sync ending each step" % e2e_steps},
        "clocks": clocks,
    }

    # ---------------- secondary measurements (rank 0 only; each replays a graph)
    if rank == 0 and not args.headline_only:
        result["secondary"] = secondary(args, dev, stream, layers, X, hbm_peak, bf16_peak, bf16_sus)
        result["cpu_baseline"] = cpu_baseline_subprocess(12.0)
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def device_fp32_lane_ops_per_s(dev):
    """SM count x 128 fp32 lanes x the maximum SM clock, the fp32 ALU ceiling."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = 2070.0   # the part's maximum SM clock, unless nvidia-smi reports it
    try:
        r = subprocess.run(["nvidia-smi", "-i", str(dev.index or 0), "--query-gpu=clocks.max.sm",
                            "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=10)
        mhz = float(r.stdout.strip().splitlines()[0])
    except Exception:
        pass
    return sms * 128 * mhz * 1e6


def _graph_time(fn, stream, dev, reps, warm=3):
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        g.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / reps  # ms per replay


def secondary(args, dev, stream, layers, X, hbm_peak, bf16_peak, bf16_sus):
    import numpy as np
    import torch

    from bit_weight_quantized_wq_gb300 import binding, inputs

    out = {}
    reps = max(3, min(args.steps, 50))

    # prefill GEMM, Qwen2.5-72B shapes, M = 2048 and 8192, INT4 g128 (sigma 0.015)
    pre = []
    for i, (K, N) in enumerate(PREFILL_SHAPES):
        W = torch.from_numpy(inputs.weights(3000 + i, N, K, 0.015)).to(dev)
        pre.append(binding.quantize_int4_g128(W))
        del W
    torch.cuda.empty_cache()
    for Mp, key in ((PREFILL_M, "prefill"), (PREFILL_M_LARGE, "prefill_m%d" % PREFILL_M_LARGE)):
        Xp = {K: torch.from_numpy(inputs.activations(3100 + K, Mp, K)[0].view(np.int16)).to(dev).view(torch.bfloat16)
              for K in {k for k, _ in PREFILL_SHAPES}}
        Yp = [torch.empty((Mp, N), dtype=torch.bfloat16, device=dev) for _, N in PREFILL_SHAPES]
        wsp = binding.Workspace(dev).get(max(binding.gemm_workspace_bytes("int4_g128", Mp, K, N) for K, N in PREFILL_SHAPES))
        per_layer = []
        for i, (K, N) in enumerate(PREFILL_SHAPES):
            f = (lambda i=i, K=K: binding.gemm_w4a16("int4_g128", Xp[K], pre[i][0], pre[i][1], pre[i][2], out=Yp[i], workspace=wsp))
            ms = _graph_time(f, stream, dev, max(3, reps // (5 if Mp == PREFILL_M else 20)))
            fl = 2.0 * Mp * N * K
            per_layer.append({"K": K, "N": N, "M": Mp, "us": ms * 1e3, "tflops": fl / (ms * 1e-3) / 1e12})
        tot_fl = sum(2.0 * Mp * N * K for K, N in PREFILL_SHAPES)
        tot_ms = sum(q["us"] for q in per_layer) / 1e3
        tf = tot_fl / (tot_ms * 1e-3) / 1e12
        out[key] = {"metric": "prefill GEMM TFLOP/s (INT4 g128 W4A16, Qwen2.5-72B shapes, M=%d)" % Mp,
                    "value": tf, "unit": "TFLOP/s", "layers": per_layer,
                    "roofline": {"bound": "tensor", "achieved": tf, "peak": bf16_peak, "unit": "TFLOP/s",
                                 "frac": tf / bf16_peak,
                                 "traffic": profile_traffic("gemm_tc.cu", "gemm_tc_prefill") if Mp == PREFILL_M else None,
                                 "note": "fp16 operands (same dense rate as bf16); peak = measured cuBLAS bf16 burst"}}
        if Mp == PREFILL_M:
            # SwiGLU on the fused gate+up projection (K = 8192, 2F = 59136), beside the plain one
            gi = PREFILL_SHAPES.index((8192, 59136))
            ysw = torch.empty((Mp, 59136 // 2), dtype=torch.bfloat16, device=dev)
            fsw = (lambda: binding.gemm_w4a16_swiglu("int4_g128", Xp[8192], pre[gi][0], pre[gi][1], pre[gi][2],
                                                     out=ysw, workspace=wsp))
            ms = _graph_time(fsw, stream, dev, max(3, reps // 5))
            fl = 2.0 * Mp * 59136 * 8192
            out["swiglu_prefill"] = {"workload": "Qwen2.5-72B fused gate+up (K=8192, 2F=59136) with SiLU(gate)*up "
                                                 "in the epilogue, INT4 g128, M=%d" % Mp,
                                     "us": ms * 1e3, "tflops": fl / (ms * 1e-3) / 1e12,
                                     "plain_gate_up_us": per_layer[gi]["us"]}
            del ysw
            # QKV split on the fused QKV projection (GQA 64/8, d_head 128: Nq = 8192, Nkv = 1024)
            qi = PREFILL_SHAPES.index((8192, 10240))
            yq = (torch.empty((Mp, 8192), dtype=torch.bfloat16, device=dev),
                  torch.empty((Mp, 1024), dtype=torch.bfloat16, device=dev),
                  torch.empty((Mp, 1024), dtype=torch.bfloat16, device=dev))
            fq = (lambda: binding.gemm_w4a16_qkv("int4_g128", Xp[8192], pre[qi][0], pre[qi][1], pre[qi][2],
                                                 Nq=8192, Nkv=1024, out=yq, workspace=wsp))
            ms = _graph_time(fq, stream, dev, max(3, reps // 5))
            fl = 2.0 * Mp * 10240 * 8192
            out["qkv_prefill"] = {"workload": "Qwen2.5-72B fused QKV (K=8192, Nq=8192, Nkv=1024) written as Q, K, V "
                                              "by the epilogue, INT4 g128, M=%d" % Mp,
                                  "us": ms * 1e3, "tflops": fl / (ms * 1e-3) / 1e12,
                                  "plain_fused_us": per_layer[qi]["us"]}
            del yq
        del Xp, Yp
        torch.cuda.empty_cache()
    del pre
    torch.cuda.empty_cache()

    # W8A8 FP8 E4M3 and W4A4 MXFP4 (on the FP8 tensor-core path) on the same Qwen2.5-72B
    # shapes, M = 2048 and 8192: the GEMM alone and the layer from bf16 activations
    # (per-token quantization + GEMM).  Peak: the FP8 dense rate, 2x the measured bf16 burst
    # (the nominal fp8/bf16 ratio 4.5 / 2.25).
    fp8_peak = 2.0 * bf16_peak
    for key, wfmt in (("fp8_prefill", "fp8"), ("w4a4_prefill", "w4a4")):
        res = {}
        for Mp in (PREFILL_M, PREFILL_M_LARGE):
            per_layer = []
            for i, (K, N) in enumerate(PREFILL_SHAPES):
                W = torch.from_numpy(inputs.weights(3000 + i, N, K, 0.015)).to(dev)
                if wfmt == "fp8":
                    Wq8, sw = binding.quantize_fp8_weights(W)
                else:
                    Wq8, sw = binding.mxfp4_weights_to_e4m3(*binding.quantize_mxfp4(W))
                del W
                Xp = torch.from_numpy(inputs.activations(3100 + K, Mp, K)[0].view(np.int16)).to(dev).view(torch.bfloat16)
                Yp = torch.empty((Mp, N), dtype=torch.bfloat16, device=dev)
                wsf = binding.Workspace(dev).get(binding.load_library().wq_gemm_w8a8_fp8_workspace_bytes(Mp, K))
                qfn = binding.quantize_fp8_activations if wfmt == "fp8" else binding.quantize_w4a4_activations
                Xq, sx = qfn(Xp)
                lay = binding.gemm_w8a8_fp8 if wfmt == "fp8" else binding.gemm_w4a4_mxfp4
                nrep = max(3, reps // (5 if Mp == PREFILL_M else 20))
                ms_g = _graph_time(lambda: binding.gemm_fp8(Xq, sx, Wq8, sw, out=Yp), stream, dev, nrep)
                ms_l = _graph_time(lambda: lay(Xp, Wq8, sw, out=Yp, workspace=wsf), stream, dev, nrep)
                fl = 2.0 * Mp * N * K
                per_layer.append({"K": K, "N": N, "M": Mp, "gemm_us": ms_g * 1e3, "gemm_tflops": fl / (ms_g * 1e-3) / 1e12,
                                  "layer_us": ms_l * 1e3, "layer_tflops": fl / (ms_l * 1e-3) / 1e12})
                del Wq8, sw, Xp, Yp, Xq, sx
                torch.cuda.empty_cache()
            tot_fl = sum(2.0 * Mp * N * K for K, N in PREFILL_SHAPES)
            tg = tot_fl / (sum(q["gemm_us"] for q in per_layer) * 1e-6) / 1e12
            tl = tot_fl / (sum(q["layer_us"] for q in per_layer) * 1e-6) / 1e12
            res["m%d" % Mp] = {"gemm_tflops": tg, "layer_tflops": tl, "layers": per_layer,
                               "roofline": {"bound": "tensor", "achieved": tg, "peak": fp8_peak, "unit": "TFLOP/s",
                                            "frac": tg / fp8_peak,
                                            "note": "tcgen05 kind::f8f6f4 GEMM; peak = 2 x measured bf16 burst"}}
        res["workload"] = ("W8A8 FP8 E4M3 (per-channel weight, per-token activation scales)" if wfmt == "fp8" else
                           "W4A4 MXFP4 (weights and per-token activations in MXFP4, re-encoded exactly to E4M3)") + \
            ", Qwen2.5-72B shapes, M = 2048 and 8192"
        out[key] = res

    # MXFP4 decode (same four shapes, M in {1, 16})
    mx_layers = []
    for i, (K, N) in enumerate(DECODE_SHAPES):
        W = torch.from_numpy(inputs.weights(2000 + i, N, K, 0.02)).to(dev)
        pk = binding.quantize_mxfp4(W)
        mx_layers.append([pk] + [tuple(t.clone() for t in pk) for _ in range(COPIES - 1)])
        del W
    Ym = {(M, N): torch.empty((M, N), dtype=torch.bfloat16, device=dev) for M in (1, 16) for _, N in DECODE_SHAPES}
    wsm = binding.Workspace(dev).get(max(binding.gemm_workspace_bytes("mxfp4", 16, K, N) for K, N in DECODE_SHAPES))

    def mx_step():
        for ci, M in enumerate((1, 16)):
            for li, (K, N) in enumerate(DECODE_SHAPES):
                Wq, s = mx_layers[li][ci % COPIES]
                binding.gemm_w4a16("mxfp4", X[(M, K)], Wq, s, out=Ym[(M, N)], workspace=wsm)

    ms = _graph_time(mx_step, stream, dev, reps)
    b = sum(decode_bytes(M, K, N) for M in (1, 16) for K, N in DECODE_SHAPES)
    out["mxfp4_decode"] = {"value": b / (ms * 1e-3) / 1e9, "unit": "GB/s", "frac_of_hbm_peak": b / (ms * 1e-3) / 1e9 / hbm_peak,
                           "workload": "same four projections, M in {1,16}, OCP MXFP4"}
    del mx_layers
    torch.cuda.empty_cache()

    # per-(shape, M) decode timings (INT4), each layer on its own graph with 3 copies
    per = []
    for li, (K, N) in enumerate(DECODE_SHAPES):
        for M in DECODE_M:
            yb = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            wsb = binding.Workspace(dev).get(binding.gemm_workspace_bytes("int4_g128", M, K, N))

            def f(li=li, M=M, K=K, yb=yb, wsb=wsb):
                for c in range(COPIES):
                    Wq, s, z = layers[li][c]
                    binding.gemm_w4a16("int4_g128", X[(M, K)], Wq, s, z, out=yb, workspace=wsb)

            ms = _graph_time(f, stream, dev, reps) / COPIES
            gbs = decode_bytes(M, K, N) / (ms * 1e-3) / 1e9
            per.append({"K": K, "N": N, "M": M, "us": ms * 1e3, "GBps": gbs, "frac": gbs / hbm_peak})
    out["decode_layers"] = per

    # SwiGLU epilogue on the fused gate+up projection (LLaMA-3-8B: K = 4096, 2F = 28672), the
    # same packed weights read as the interleaved gate/up layout; beside the plain projection.
    gi = DECODE_SHAPES.index((4096, 28672))
    F = 28672 // 2
    sw = []
    for M in DECODE_M:
        ys = torch.empty((M, F), dtype=torch.bfloat16, device=dev)
        wss = binding.Workspace(dev).get(binding.gemm_workspace_bytes("int4_g128", M, 4096, 2 * F))

        def fs(M=M, ys=ys, wss=wss):
            for c in range(COPIES):
                Wq, s, z = layers[gi][c]
                binding.gemm_w4a16_swiglu("int4_g128", X[(M, 4096)], Wq, s, z, out=ys, workspace=wss)

        ms = _graph_time(fs, stream, dev, reps) / COPIES
        b = 0.53125 * 2 * F * 4096 + 2.0 * M * 4096 + 2.0 * M * F
        plain = next(q["us"] for q in per if q["K"] == 4096 and q["N"] == 2 * F and q["M"] == M)
        sw.append({"M": M, "us": ms * 1e3, "GBps": b / (ms * 1e-3) / 1e9, "frac": b / (ms * 1e-3) / 1e9 / hbm_peak,
                   "plain_gate_up_us": plain})
    out["swiglu_decode"] = {"workload": "LLaMA-3-8B fused gate+up (K=4096, 2F=28672) with SiLU(gate)*up "
                                        "in the epilogue, INT4 g128, Y [M, 14336]", "points": sw}

    # QKV split on the fused QKV projection (LLaMA-3-8B: GQA 32/8, d_head 128: Nq = 4096,
    # Nkv = 1024), beside the plain projection writing one [M, 6144] tensor.
    qi = DECODE_SHAPES.index((4096, 6144))
    qk = []
    for M in DECODE_M:
        yq = (torch.empty((M, 4096), dtype=torch.bfloat16, device=dev), torch.empty((M, 1024), dtype=torch.bfloat16, device=dev),
              torch.empty((M, 1024), dtype=torch.bfloat16, device=dev))
        wsq = binding.Workspace(dev).get(binding.gemm_workspace_bytes("int4_g128", M, 4096, 6144))

        def fq(M=M, yq=yq, wsq=wsq):
            for c in range(COPIES):
                Wq, s, z = layers[qi][c]
                binding.gemm_w4a16_qkv("int4_g128", X[(M, 4096)], Wq, s, z, Nq=4096, Nkv=1024, out=yq, workspace=wsq)

        ms = _graph_time(fq, stream, dev, reps) / COPIES
        b = decode_bytes(M, 4096, 6144)
        plain = next(q["us"] for q in per if q["K"] == 4096 and q["N"] == 6144 and q["M"] == M)
        qk.append({"M": M, "us": ms * 1e3, "GBps": b / (ms * 1e-3) / 1e9, "frac": b / (ms * 1e-3) / 1e9 / hbm_peak,
                   "plain_fused_us": plain})
    out["qkv_decode"] = {"workload": "LLaMA-3-8B fused QKV (K=4096, Nq=4096, Nkv=1024) written as Q, K, V by the "
                                     "epilogue, INT4 g128", "points": qk}

    # GPTQ sweep (INT4 g128) on a LLaMA-3-8B projection (N = K = 4096).  The factor is the
    # seeded stand-in (the sweep's work does not depend on its values).  Bound: fp32 ALU, one
    # multiply and one subtract per update, N K^2 / 2 updates.
    Wg = torch.from_numpy(inputs.weights(5100, 4096, 4096, 0.02)).to(dev)
    Ug = torch.from_numpy(inputs.upper_factor(5101, 4096)).to(dev)
    ms = _graph_time(lambda: binding.gptq_int4_g128(Wg, Ug), stream, dev, 2, warm=1)
    upd = 4096.0 * 4096 * 4096 / 2
    alu_peak = device_fp32_lane_ops_per_s(dev) / 2 / 1e12   # T updates/s
    out["gptq_int4_g128"] = {"workload": "GPTQ sweep, N = K = 4096 (LLaMA-3-8B o_proj), INT4 g128",
                             "ms": ms, "T_updates_per_s": upd / (ms * 1e-3) / 1e12,
                             "roofline": {"bound": "alu", "achieved": upd / (ms * 1e-3) / 1e12, "peak": alu_peak,
                                          "unit": "T updates/s", "frac": upd / (ms * 1e-3) / 1e12 / alu_peak,
                                          "note": "peak = SMs x 128 fp32 lanes x max SM clock / 2 ops per update"}}
    del Ug
    # GPTQ's inverse-Hessian factor on the device from 128 calibration samples (float64:
    # H = 2 X^T X + lambda I, blocked Cholesky, blocked triangular inverse), and GPTQ end to end
    # (factor + sweep).  Flop count 2 n K^2 + K^3 / 3 + K^3 / 3 against the nominal fp64 rate.
    Xg = torch.from_numpy(inputs.calibration(5102, 128, 4096)).to(dev)
    wsg = torch.empty(binding.load_library().wq_gptq_workspace_bytes(4096), dtype=torch.uint8, device=dev)
    ms_f = _graph_time(lambda: binding.gptq_factor(Xg, workspace=wsg), stream, dev, 3, warm=1)
    ms_e = _graph_time(lambda: binding.gptq_int4_g128_calib(Wg, Xg, workspace=wsg), stream, dev, 2, warm=1)
    flf = 2.0 * 128 * 4096 ** 2 + 2.0 * 4096 ** 3 / 3
    fp64_nominal = 1.25   # TFLOP/s, the part's nominal fp64 rate (no measured fp64 peak)
    out["gptq_factor"] = {"workload": "H = 2 X^T X + lambda I and the upper factor of H^-1, K = 4096, n = 128",
                          "ms": ms_f, "end_to_end_ms": ms_e,
                          "roofline": {"bound": "fp64", "achieved": flf / (ms_f * 1e-3) / 1e12, "peak": fp64_nominal,
                                       "unit": "TFLOP/s", "frac": flf / (ms_f * 1e-3) / 1e12 / fp64_nominal,
                                       "note": "peak = nominal fp64 rate (fallback, not measured)"}}
    del Wg, Xg, wsg
    torch.cuda.empty_cache()

    # AWQ search (21 exponents) + packing on the same projection, 128 calibration samples.
    # Bound: the fp32 error GEMM, 2 n N K per exponent.
    Wa = torch.from_numpy(inputs.weights(5200, 4096, 4096, 0.02)).to(dev)
    Xa = torch.from_numpy(inputs.calibration(5201, 128, 4096)).to(dev)
    wsa = torch.empty(binding.load_library().wq_awq_workspace_bytes(4096, 4096, 128), dtype=torch.uint8, device=dev)
    ms = _graph_time(lambda: binding.awq_int4_g128(Wa, Xa, workspace=wsa), stream, dev, 3, warm=1)
    fl = 21 * 2.0 * 128 * 4096 * 4096
    fp32_peak = device_fp32_lane_ops_per_s(dev) * 2 / 1e12    # TFLOP/s, FMA = 2
    out["awq_int4_g128"] = {"workload": "AWQ search (21 exponents) + packing, N = K = 4096, 128 calibration samples",
                            "ms": ms,
                            "roofline": {"bound": "alu", "achieved": fl / (ms * 1e-3) / 1e12, "peak": fp32_peak,
                                         "unit": "TFLOP/s", "frac": fl / (ms * 1e-3) / 1e12 / fp32_peak,
                                         "note": "error-GEMM flops over the whole search time; peak = fp32 FMA rate"}}
    del Wa, Xa, wsa
    torch.cuda.empty_cache()

    # quantize kernels on the decode shapes: fp32 read + packed write
    qres = {}
    for name, fn, ob in (("int4_g128", binding.quantize_int4_g128, 0.53125), ("mxfp4", binding.quantize_mxfp4, 0.53125)):
        Ws = [torch.from_numpy(inputs.weights(50 + i, N, K, 0.02)).to(dev) for i, (K, N) in enumerate(DECODE_SHAPES)]

        def qf(Ws=Ws, fn=fn):
            for W in Ws:
                fn(W)

        ms = _graph_time(qf, stream, dev, max(3, reps // 5))
        byts = sum((4 + ob) * K * N for K, N in DECODE_SHAPES)
        qres[name] = {"GBps": byts / (ms * 1e-3) / 1e9, "frac": byts / (ms * 1e-3) / 1e9 / hbm_peak}
        del Ws
    torch.cuda.empty_cache()
    out["quantize"] = qres

    # crossover sweep K = N = 8192: both kernels, both formats
    if not args.no_sweep:
        K = N = 8192
        sweep = {}
        for fmt in ("int4_g128", "mxfp4"):
            W = torch.from_numpy(inputs.weights(4000, N, K, 0.02)).to(dev)
            pk = binding.quantize_int4_g128(W) if fmt == "int4_g128" else binding.quantize_mxfp4(W)
            cps = [pk] + [tuple(t.clone() for t in pk) for _ in range(COPIES - 1)]
            del W
            pts = []
            best_T = 0
            for M in CROSS_M:
                Xs = torch.from_numpy(inputs.activations(4000 + M, M, K)[0].view(np.int16)).to(dev).view(torch.bfloat16)
                ys = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
                row = {"M": M}
                for kname, kfn in (("gemv", binding.gemv_w4a16), ("tc", binding.gemm_tc_w4a16)):
                    if kname == "gemv" and M > DECODE_MAX_M:
                        continue
                    wsx = binding.Workspace(dev).get(binding.gemm_workspace_bytes(fmt, M, K, N))

                    def f(kfn=kfn, Xs=Xs, ys=ys, wsx=wsx):
                        for c in cps:
                            kfn(fmt, Xs, c[0], c[1], c[2] if fmt == "int4_g128" else None, out=ys, workspace=wsx)

                    try:
                        ms = _graph_time(f, stream, dev, max(3, reps // 5)) / COPIES
                    except Exception as ex:  # a kernel that cannot run this shape
                        row[kname] = {"error": str(ex)[:120]}
                        continue
                    row[kname] = {"us": ms * 1e3, "GBps": decode_bytes(M, K, N) / (ms * 1e-3) / 1e9,
                                  "TFLOPs": 2.0 * M * N * K / (ms * 1e-3) / 1e12}
                pts.append(row)
            best_T = crossover_T(pts)
            binding.set_dispatch_threshold(fmt, K, N, best_T)
            sweep[fmt] = {"points": pts, "threshold_T": best_T, "applied": True}
        out["crossover_8192"] = sweep
        # the decode shapes: the crossover around the decode kernel's limit, per format
        th = {}
        for fmt in ("int4_g128", "mxfp4"):
            th[fmt] = {}
            for i, (K, N) in enumerate(DECODE_SHAPES):
                W = torch.from_numpy(inputs.weights(4100 + i, N, K, 0.02)).to(dev)
                pk = binding.quantize_int4_g128(W) if fmt == "int4_g128" else binding.quantize_mxfp4(W)
                cps = [pk] + [tuple(t.clone() for t in pk) for _ in range(COPIES - 1)]
                del W
                pts = []
                for M in THRESH_M:
                    Xs = torch.from_numpy(inputs.activations(4100 + M, M, K)[0].view(np.int16)).to(dev).view(torch.bfloat16)
                    ys = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
                    wsx = binding.Workspace(dev).get(binding.gemm_workspace_bytes(fmt, M, K, N))
                    row = {"M": M}
                    for kname, kfn in (("gemv", binding.gemv_w4a16), ("tc", binding.gemm_tc_w4a16)):
                        def f(kfn=kfn, Xs=Xs, ys=ys, wsx=wsx):
                            for c in cps:
                                kfn(fmt, Xs, c[0], c[1], c[2] if fmt == "int4_g128" else None, out=ys, workspace=wsx)
                        row[kname] = {"us": _graph_time(f, stream, dev, max(3, reps // 5)) / COPIES * 1e3}
                    pts.append(row)
                T = crossover_T(pts, lower=16)
                binding.set_dispatch_threshold(fmt, K, N, T)
                th[fmt]["%dx%d" % (K, N)] = {"T": T, "points": pts}
                del cps, pk
            torch.cuda.empty_cache()
        out["dispatch_thresholds"] = {"how": "per (fmt, K, N): the largest M of the measured points up to which the "
                                             "decode kernel is at least as fast as the tensor-core kernel at every "
                                             "point; applied with wq_set_dispatch_threshold", "table": th}
    return out


def crossover_T(pts, lower=0):
    """The largest M such that the decode kernel is no slower than the tensor-core kernel at
    every measured M up to it (points without a decode time end the run)."""
    T = lower
    for r in pts:
        g, c = r.get("gemv", {}), r.get("tc", {})
        if "us" not in g or "us" not in c or g["us"] > c["us"]:
            break
        T = r["M"]
    return T


def run_ncu_case(args):
    """A few plain launches of one kernel on one layer, for ncu captures (not a bench line).

    decode:  the (K, N) = (4096, 28672) layer at M = 1, INT4, 3 weight copies (189 MB > L2).
    decode_step: the headline step -- the 12 decode calls (4 shapes x M in {1, 4, 16}), INT4,
             3 weight copies; one step = 12 launches, run warmup + steps times without a graph.
    prefill: the (K, N) = (8192, 8192) layer at M = 2048, INT4 (37 MB weights, 32 MB X).
    mxfp4:   the decode layer in MXFP4.
    swiglu_decode: the decode layer read as the fused gate+up weight (2F = 28672) with the
             SwiGLU epilogue, M = 1, INT4.
    quant:   INT4 quantize of the (4096, 28672) weights (470 MB fp32).
    gptq:    the GPTQ sweep, N = K = 4096, seeded stand-in inverse-Hessian factor.
    fp8:     the FP8 E4M3 GEMM alone on the (8192, 8192) prefill layer, M = 2048.
    awq:     the AWQ search + packing, N = K = 4096, 128 calibration samples.
    """
    import numpy as np
    import torch

    from bit_weight_quantized_wq_gb300 import binding, inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    case = args.ncu_case
    if case == "decode_step":
        layers = []
        for i, (K, N) in enumerate(DECODE_SHAPES):
            W = torch.from_numpy(inputs.weights(1000 + i, N, K, 0.02)).to(dev)
            pk = binding.quantize_int4_g128(W)
            layers.append([pk] + [tuple(t.clone() for t in pk) for _ in range(COPIES - 1)])
            del W
        X = {(M, K): torch.from_numpy(inputs.activations(M * 100 + K, M, K)[0].view(np.int16)).to(dev).view(torch.bfloat16)
             for M in DECODE_M for K, _ in DECODE_SHAPES}
        Y = {(M, N): torch.empty((M, N), dtype=torch.bfloat16, device=dev) for M in DECODE_M for _, N in DECODE_SHAPES}
        ws = binding.Workspace(dev).get(max(binding.gemm_workspace_bytes("int4_g128", M, K, N)
                                            for M in DECODE_M for K, N in DECODE_SHAPES))
        n = 0
        for _ in range(args.warmup + args.steps):
            for ci, M in enumerate(DECODE_M):
                for li, (K, N) in enumerate(DECODE_SHAPES):
                    Wq, s, z = layers[li][ci % COPIES]
                    binding.gemm_w4a16("int4_g128", X[(M, K)], Wq, s, z, out=Y[(M, N)], workspace=ws)
                    n += 1
        torch.cuda.synchronize()
        print(json.dumps({"ncu_case": case, "launches": n, "launches_per_step": len(DECODE_M) * len(DECODE_SHAPES)}))
        return 0
    if case == "fp8":
        # the FP8 GEMM alone on the (8192, 8192) prefill layer at M = 2048
        K, N, M = 8192, 8192, 2048
        W = torch.from_numpy(inputs.weights(1002, N, K, 0.015)).to(dev)
        Wq8, sw = binding.quantize_fp8_weights(W)
        del W
        X = torch.from_numpy(inputs.activations(7, M, K)[0].view(np.int16)).to(dev).view(torch.bfloat16)
        Xq, sx = binding.quantize_fp8_activations(X)
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        for _ in range(args.warmup + args.steps):
            binding.gemm_fp8(Xq, sx, Wq8, sw, out=Y)
        torch.cuda.synchronize()
        print(json.dumps({"ncu_case": case, "launches": args.warmup + args.steps, "K": K, "N": N, "M": M}))
        return 0
    if case in ("gptq", "awq"):
        W = torch.from_numpy(inputs.weights(5100, 4096, 4096, 0.02)).to(dev)
        if case == "gptq":
            U = torch.from_numpy(inputs.upper_factor(5101, 4096)).to(dev)
            fn = lambda: binding.gptq_int4_g128(W, U)
        else:
            X = torch.from_numpy(inputs.calibration(5201, 128, 4096)).to(dev)
            wsa = torch.empty(binding.load_library().wq_awq_workspace_bytes(4096, 4096, 128), dtype=torch.uint8,
                              device=dev)
            fn = lambda: binding.awq_int4_g128(W, X, workspace=wsa)
        for _ in range(args.warmup + args.steps):
            fn()
        torch.cuda.synchronize()
        print(json.dumps({"ncu_case": case, "calls": args.warmup + args.steps}))
        return 0
    if case in ("decode", "mxfp4", "swiglu_decode"):
        K, N, M, fmt = 4096, 28672, 1, ("mxfp4" if case == "mxfp4" else "int4_g128")
    elif case == "prefill":
        K, N, M, fmt = 8192, 8192, 2048, "int4_g128"
    else:
        K, N, M, fmt = 4096, 28672, 1, "int4_g128"
    W = torch.from_numpy(inputs.weights(1002, N, K, 0.02)).to(dev)
    if case == "quant":
        for _ in range(args.warmup + args.steps):
            binding.quantize_int4_g128(W)
        torch.cuda.synchronize()
        print(json.dumps({"ncu_case": case, "launches": args.warmup + args.steps}))
        return 0
    pk = binding.quantize_int4_g128(W) if fmt == "int4_g128" else binding.quantize_mxfp4(W)
    del W
    copies = [pk] + [tuple(t.clone() for t in pk) for _ in range(COPIES - 1)]
    X = torch.from_numpy(inputs.activations(7, M, K)[0].view(np.int16)).to(dev).view(torch.bfloat16)
    sw = case == "swiglu_decode"
    Y = torch.empty((M, N // 2 if sw else N), dtype=torch.bfloat16, device=dev)
    ws = binding.Workspace(dev).get(binding.gemm_workspace_bytes(fmt, M, K, N))
    fn = binding.gemm_w4a16_swiglu if sw else binding.gemm_w4a16
    n = 0
    for i in range(args.warmup + args.steps):
        c = copies[i % COPIES]
        fn(fmt, X, c[0], c[1], c[2] if fmt == "int4_g128" else None, out=Y, workspace=ws)
        n += 1
    torch.cuda.synchronize()
    print(json.dumps({"ncu_case": case, "launches": n, "K": K, "N": N, "M": M, "fmt": fmt}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--cpu-sample", type=float, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--ncu-case", default=None, choices=["decode", "decode_step", "prefill", "mxfp4", "swiglu_decode", "quant", "gptq", "awq", "fp8"],
                    help="run a few plain launches of one kernel (for ncu captures) instead of the bench")
    args = ap.parse_args()
    if args.cpu_sample is not None:
        b, t, d = oracle_sample(args.cpu_sample, 1)
        cores, threads = host_threads()
        print(json.dumps({"bytes": b, "seconds": t, "desc": d, "cores": cores, "threads": threads}))
        return 0
    if args.warmup < 3:
        args.warmup = 3
    if args.ncu_case:
        return run_ncu_case(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
