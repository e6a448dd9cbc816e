"""Benchmark of the W4A16 linear layer on GB300 (one JSON line on stdout).

Workload (default, one GPU): the Llama-2-7B decode layers (K, N) = (4096,
12288) qkv, (4096, 4096) o_proj, (4096, 22016) gate_up, (11008, 4096) down,
AWQ group-128 4-bit asymmetric weights, bf16 activations, M in {1, 4, 16}.
One step runs the fused GEMM for every (layer, M) pair: 12 calls. Every call
reads its own copy of the repacked weights (12 copies, about 315 MB, well
above the 129 MB L2), so no call finds its weights in L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

value       = weight GB/s over the timed steps (algorithmic bytes: packed codes
              K*N/2 + scales G*N*2 + zeros G*N/2 per call), all ranks together.
tflops      = 2*M*N*K summed over the calls / time.
e2e         = the same metric through the public Python/C-ABI path with x
              copied from pinned host memory and y copied back inside the
              timed region, eager launches.
roofline    = the decode kernel's per-launch durations (CUDA events on the
              launch stream, launches front-loaded behind a long device copy
              so the host never starves the GPU), against the measured HBM
              copy bandwidth.
cpu_baseline = the CPU oracle (numpy: unpack, dequantise, fp64 matmul) on the
              o_proj layer at M = 1, 4 and 16.
dequant_cublas = the same step as w4_dequant to dense bf16 + cuBLAS (torch.matmul),
              graph-timed like `value`; fused_speedup = its time / ours.
prefill     = the Llama-2-7B prefill layers (M in {512, 2048, 4096}) on the
              tcgen05 kernel: TFLOP/s per call and, for M >= 2048, against the
              measured dense bf16 tensor-core peak.
--impl reference times that oracle as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = ("W4A16 GEMM TFLOP/s and weight GB/s vs M (1–4096), % of HBM / bf16 TC roofline")
WORKLOAD = synth.WORKLOADS[1]          # Llama-2-7B decode layers
FALLBACK_HBM_GBS = 6800.0
FALLBACK_TC_TFLOPS = 1900.0

# DRAM bytes per launch of the decode kernel from ncu (dram__bytes_read.sum +
# dram__bytes_write.sum), keyed by the sha1 of the kernel source they were
# taken on; see profiles/. A changed kernel source reports null.
TRAFFIC_RECORDS: dict = {
    "c33dd14b5051": 26437227,   # mean of the 12 launches of one step
}


def alg_bytes(K: int, N: int, group: int = 128) -> int:
    G = K // group
    return K * N // 2 + G * N * 2 + G * N // 2


def kernel_source_hash() -> str:
    p = os.path.join(ROOT, "int4_weight_only_repack_gb300", "csrc", "decode_kernel.cu")
    with open(p, "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()[:12]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_tc_peak():
    """Dense bf16 tensor-core peak (burst: the prefill calls are timed alone)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_TC_TFLOPS, "fallback"


# --------------------------------------------------------------------------- #
# Clock sampling during the timed region                                       #
# --------------------------------------------------------------------------- #
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.15)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- #
# Our arm                                                                       #
# --------------------------------------------------------------------------- #
def setup_dist():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int, device) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def build_calls(w4, torch, device):
    """Repack one weight copy per (layer, M) and allocate x / y for each call."""
    calls = []
    for li, (K, N, name) in enumerate(WORKLOAD.shapes):
        L = synth.make_workload_layer(WORKLOAD.index, li)
        qweight = torch.from_numpy(L.qweight).to(device)
        qzeros = torch.from_numpy(L.qzeros).to(device)
        scales = torch.from_numpy(L.scales.view(np.int16)).to(device).view(torch.bfloat16)
        for M in WORKLOAD.ms:
            layer = w4.repack_awq(qweight, qzeros, scales, K, N, WORKLOAD.group, torch.bfloat16)
            x_bits = synth.make_workload_x(WORKLOAD.index, li, M)
            x = torch.from_numpy(x_bits.view(np.int16)).to(device).view(torch.bfloat16)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
            calls.append(dict(name=name, K=K, N=N, M=M, layer=layer, x=x, y=y, x_bits=x_bits))
        del qweight, qzeros, scales
    # one workspace for the stream, as big as the largest call asks for (the
    # calls run in stream order, so they can share it)
    need = max(w4.w4a16_gemm_workspace_size(c["M"], c["N"], c["K"], WORKLOAD.group,
                                            torch.bfloat16, False) for c in calls)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
    for c in calls:
        c["ws"] = ws
    torch.cuda.synchronize()
    return calls


def run_step(w4, calls):
    for c in calls:
        L = c["layer"]
        w4.w4a16_gemm(c["x"], L.qw, L.scales, L.zeros, None, c["y"], c["M"], c["N"], c["K"],
                      L.group, L.dtype, c["ws"])


def per_launch_times(w4, torch, calls, reps: int, device):
    """Average duration of each call's kernel, CUDA events on the launch stream.

    A long device-side copy is enqueued first so that every launch and event
    below is queued before the GPU reaches them: the events then bracket the
    kernels alone, not host enqueue gaps.
    """
    stream = torch.cuda.current_stream()
    big = torch.empty(1 << 30, dtype=torch.uint8, device=device)
    big2 = torch.empty_like(big)
    totals = [0.0] * len(calls)
    for _ in range(reps):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in calls]
        for _ in range(6):
            big2.copy_(big)
        for c, (e0, e1) in zip(calls, evs):
            L = c["layer"]
            e0.record(stream)
            w4.w4a16_gemm(c["x"], L.qw, L.scales, L.zeros, None, c["y"], c["M"], c["N"], c["K"],
                          L.group, L.dtype, c["ws"])
            e1.record(stream)
        torch.cuda.synchronize()
        for i, (e0, e1) in enumerate(evs):
            totals[i] += e0.elapsed_time(e1) * 1e-3
    del big, big2
    return [t / reps for t in totals]


def graph_time(torch, fn, reps: int) -> float:
    """Seconds per call of `fn` (a sequence of launches), from a CUDA graph of it
    replayed `reps` times, CUDA events on the launch stream."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    del g
    return e0.elapsed_time(e1) * 1e-3 / reps


def dequant_cublas_measure(w4, torch, calls, reps: int, device):
    """The same step as dequantise-then-GEMM: w4_dequant of each call's layer to a
    dense bf16 [K, N] (one scratch per layer shape), then torch.matmul (cuBLAS)."""
    scratch = {}
    for c in calls:
        key = (c["K"], c["N"])
        if key not in scratch:
            scratch[key] = torch.empty((c["K"], c["N"]), dtype=torch.bfloat16, device=device)

    def step():
        for c in calls:
            L, W = c["layer"], scratch[(c["K"], c["N"])]
            w4.w4_dequant(L.qw, L.scales, L.zeros, c["K"], c["N"], L.group, L.dtype, L.layout,
                          False, W)
            torch.matmul(c["x"], W, out=c["y2"])

    for c in calls:
        c["y2"] = torch.empty_like(c["y"])
    t = graph_time(torch, step, reps)
    for c in calls:
        del c["y2"]
    del scratch
    return t


def prefill_measure(w4, torch, device, reps: int = 10):
    """The Llama-2-7B prefill layers (same shapes, M in {512, 2048, 4096}) on the
    tcgen05 kernel: TFLOP/s per (layer, M), two weight copies per layer; beside
    each, a dense bf16 GEMM of the same shape through torch.matmul (cuBLAS), the
    ceiling a weight-only kernel approaches at compute-bound sizes."""
    wl = synth.WORKLOADS[2]
    rows = []
    for li, (K, N, name) in enumerate(wl.shapes):
        L = synth.make_workload_layer(wl.index, li)
        qweight = torch.from_numpy(L.qweight).to(device)
        qzeros = torch.from_numpy(L.qzeros).to(device)
        scales = torch.from_numpy(L.scales.view(np.int16)).to(device).view(torch.bfloat16)
        layers = [w4.repack_awq(qweight, qzeros, scales, K, N, wl.group, torch.bfloat16)
                  for _ in range(2)]
        del qweight, qzeros, scales
        for M in wl.ms:
            x = torch.randn(M, K, device=device).to(torch.bfloat16)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=device)

            def fn():
                for l in layers:
                    w4.linear(x, l, y=y)

            t = graph_time(torch, fn, reps) / len(layers)
            wd = [torch.randn(K, N, device=device).to(torch.bfloat16) for _ in range(2)]
            yd = torch.empty((M, N), dtype=torch.bfloat16, device=device)

            def dense():
                for w in wd:
                    torch.matmul(x, w, out=yd)

            td = graph_time(torch, dense, reps) / len(wd)
            rows.append({"layer": name, "M": M, "us": round(t * 1e6, 2),
                         "tflops": round(2.0 * M * N * K / t / 1e12, 1),
                         "dense_bf16_cublas_us": round(td * 1e6, 2),
                         "dense_bf16_cublas_tflops": round(2.0 * M * N * K / td / 1e12, 1)})
            del x, y, wd, yd
        del layers
        torch.cuda.empty_cache()
    return rows


def cpu_baseline_measure(min_seconds: float = 10.0):
    """The oracle as it stands on this host: o_proj (4096 x 4096) at M = 1, 4, 16."""
    import oracle
    li = [s[2] for s in WORKLOAD.shapes].index("o_proj")
    K, N, _ = WORKLOAD.shapes[li]
    L = synth.make_workload_layer(WORKLOAD.index, li)
    xs = {M: synth.make_workload_x(WORKLOAD.index, li, M) for M in WORKLOAD.ms}
    t0 = time.perf_counter()
    done_bytes = 0
    calls = 0
    while True:
        for M in WORKLOAD.ms:
            oracle.reference_y(xs[M], L.qweight, L.qzeros, L.scales, WORKLOAD.group, "bf16", "awq")
            done_bytes += alg_bytes(K, N)
            calls += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            break
    return {"value": done_bytes / el / 1e9, "unit": "GB/s", "cores": blas_threads(),
            "kind": "oracle",
            "sample": f"o_proj K=4096 N=4096 at M=1,4,16: {calls} full oracle calls (AWQ unpack, "
                      f"fp32 dequantise, fp64 matmul) in {el:.1f} s"}


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def ours(args):
    import torch

    import int4_weight_only_repack_gb300 as w4

    world, rank, local = setup_dist()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    w4.lib()

    calls = build_calls(w4, torch, device)
    step_bytes = sum(alg_bytes(c["K"], c["N"]) for c in calls)
    step_flops = sum(2 * c["M"] * c["N"] * c["K"] for c in calls)

    # warm-up (eager), then capture one step as a CUDA graph
    for _ in range(max(args.warmup, 3)):
        run_step(w4, calls)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run_step(w4, calls)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()

    # ---- timed region ----------------------------------------------------------
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    elapsed = max_over_ranks(e0.elapsed_time(e1) * 1e-3, world, device)

    # ---- per-launch kernel durations (roofline) ---------------------------------
    t_launch = per_launch_times(w4, torch, calls, reps=5, device=device)
    kern_bytes = sum(alg_bytes(c["K"], c["N"]) for c in calls)
    kern_time = sum(t_launch)
    peak, peak_src = measured_peaks()
    achieved = kern_bytes / kern_time / 1e9
    per_call = [{"layer": c["name"], "M": c["M"], "us": round(t * 1e6, 2),
                 "gbs": round(alg_bytes(c["K"], c["N"]) / t / 1e9, 1),
                 "frac": round(alg_bytes(c["K"], c["N"]) / t / 1e9 / peak, 3)}
                for c, t in zip(calls, t_launch)]
    traffic = TRAFFIC_RECORDS.get(kernel_source_hash())

    # ---- end to end through the public API, host buffers ------------------------
    e2e_steps = min(args.steps, 200)
    hx = [torch.from_numpy(c["x_bits"].view(np.int16)).view(torch.bfloat16).pin_memory()
          for c in calls]
    hy = [torch.empty((c["M"], c["N"]), dtype=torch.bfloat16).pin_memory() for c in calls]
    h2d = sum(t.numel() * 2 for t in hx)
    d2h = sum(t.numel() * 2 for t in hy)
    for _ in range(2):
        for c, a, b in zip(calls, hx, hy):
            c["x"].copy_(a, non_blocking=True)
            w4.linear(c["x"], c["layer"], y=c["y"])
            b.copy_(c["y"], non_blocking=True)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        for c, a, b in zip(calls, hx, hy):
            c["x"].copy_(a, non_blocking=True)
            w4.linear(c["x"], c["layer"], y=c["y"])
            b.copy_(c["y"], non_blocking=True)
    torch.cuda.synchronize()
    e2e_el = max_over_ranks(time.perf_counter() - t0, world, device)

    # ---- comparison: dequantise then cuBLAS, same step, same timing ------------
    t_deq = dequant_cublas_measure(w4, torch, calls, reps=min(args.steps, 200), device=device)

    # ---- large-M (prefill) layers on the tensor cores -------------------------
    prefill = None
    if not args.no_prefill:
        rows = prefill_measure(w4, torch, device)
        big = [r for r in rows if r["M"] >= 2048]
        kn = {sh[2]: (sh[0], sh[1]) for sh in synth.WORKLOADS[2].shapes}
        flops = sum(2.0 * r["M"] * kn[r["layer"]][0] * kn[r["layer"]][1] for r in big)
        tsum = sum(r["us"] for r in big) * 1e-6
        tc_peak, tc_src = measured_tc_peak()
        prefill = {"workload": "llama2_7b_prefill: the four layers at M in {512, 2048, 4096}, "
                               "bf16, two weight copies per layer, CUDA graph of the calls",
                   "tflops_m_ge_2048": round(flops / tsum / 1e12, 1),
                   "roofline": {"bound": "tensor", "achieved": round(flops / tsum / 1e12, 1),
                                "peak": tc_peak, "unit": "TFLOP/s",
                                "frac": round(flops / tsum / 1e12 / tc_peak, 4),
                                "peak_source": tc_src, "kernel": "w4a16_prefill_kernel"},
                   "per_call": rows}

    # ---- grouped MoE GEMM (one GPU only: a side figure like the CPU baseline) --
    moe_part = None
    if world == 1 and not args.no_moe:
        moe_part = {"workload": "mixtral_8x7b_shaped experts (8; w13 4096->28672, w2 "
                                "14336->4096), 16 and 4096 tokens routed top-2, bf16, "
                                "one w4a16_moe_gemm call against one w4a16_gemm per expert",
                    "per_call": moe_measure((16, 4096))}

    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_base = cpu_baseline_measure(args.cpu_seconds)

    if rank == 0:
        value = step_bytes * args.steps * world / elapsed / 1e9
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(elapsed / args.steps * 1e3, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded N(0,0.02) weights quantised per group of 128, x ~ N(0,1))",
            "config": {
                "workload": "llama2_7b_decode: (K,N)=(4096,12288),(4096,4096),(4096,22016),"
                            "(11008,4096); M in {1,4,16}; AWQ g128; bf16",
                "calls_per_step": len(calls),
                "weight_bytes_per_step": step_bytes,
                "l2": "inputs larger than L2: 12 distinct weight copies (%.0f MB) per step"
                      % (step_bytes / 1e6),
                "timing": "CUDA graph of one step replayed; CUDA events on the launch stream",
                "parallelism": "replicas" if world > 1 else "single GPU",
            },
            "tflops": round(step_flops * args.steps * world / elapsed / 1e12, 4),
            "gpu_launches": len(calls) * args.steps,
            "clocks": clocks,
            "e2e": {"value": round(step_bytes * e2e_steps * world / e2e_el / 1e9, 2),
                    "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": traffic, "peak_source": peak_src,
                         "kernel": "w4a16_decode_kernel",
                         "per_launch": per_call},
            "cpu_baseline": cpu_base,
            "dequant_cublas": {"value": round(step_bytes / t_deq / 1e9, 2), "unit": "GB/s",
                               "ms_per_step": round(t_deq * 1e3, 5),
                               "fused_speedup": round(t_deq / (elapsed / args.steps), 2),
                               "how": "w4_dequant to dense bf16 [K,N] + torch.matmul (cuBLAS) "
                                      "per call, CUDA graph of the step"},
            "prefill": prefill,
            "moe": moe_part,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# --------------------------------------------------------------------------- #
# Reference arm: the CPU oracle                                                 #
# --------------------------------------------------------------------------- #
def reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    li = [s[2] for s in WORKLOAD.shapes].index("o_proj")
    K, N, _ = WORKLOAD.shapes[li]
    L = synth.make_workload_layer(WORKLOAD.index, li)
    Ms = list(WORKLOAD.ms)
    xs = {M: synth.make_workload_x(WORKLOAD.index, li, M) for M in Ms}

    def step(i):
        M = Ms[i % len(Ms)]
        oracle.reference_y(xs[M], L.qweight, L.qzeros, L.scales, WORKLOAD.group, "bf16", "awq")

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    el = time.perf_counter() - t0
    value = alg_bytes(K, N) * args.steps / el / 1e9
    sample = (f"each step: one full oracle call (AWQ unpack, fp32 dequantise, fp64 matmul) on "
              f"o_proj K=4096 N=4096, M cycling 1,4,16")
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": "llama2_7b_decode (o_proj sample of it on the host cores)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": blas_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def single(args):
    """One GEMM call shape repeated `--steps` times (for profiler captures)."""
    import torch

    import int4_weight_only_repack_gb300 as w4

    parts = args.single.split(",")
    K, N, M = int(parts[0]), int(parts[1]), int(parts[2])
    dtype = parts[3] if len(parts) > 3 else "bf16"
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    dev = torch.device("cuda")
    L = synth.make_custom_layer([5, K, N], K, N, group=128, dtype=dtype)
    layer = w4.repack_awq(torch.from_numpy(L.qweight).to(dev), torch.from_numpy(L.qzeros).to(dev),
                          torch.from_numpy(L.scales.view(np.int16)).to(dev).view(tdt), K, N, 128, tdt)
    x = torch.from_numpy(synth.make_custom_x([6, M, K], M, K, dtype).view(np.int16)).to(dev).view(tdt)
    y = torch.empty((M, N), dtype=tdt, device=dev)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        w4.linear(x, layer, y=y)
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) * 1e-3 / max(1, args.steps)
    print(json.dumps({"single": [K, N, M, dtype], "us_per_call": round(t * 1e6, 2),
                      "weight_gbs": round(alg_bytes(K, N) / t / 1e9, 1),
                      "tflops": round(2.0 * M * N * K / t / 1e12, 2),
                      "device_status": w4.w4_device_status()}), flush=True)


def sweep(args):
    """A layer sweep over M: one JSON line per (layer, M) with time, weight
    GB/s, TFLOP/s and the fraction of the matching roofline (HBM for M <= 16,
    dense bf16 tensor peak above). Default: the Llama-2-70B layers, M from 1 to
    4096 (--sweep-config 4); --sweep-config 3: the Llama-2-13B GPTQ act-order
    layers (fp16, M in {1, 16, 1024})."""
    import torch

    import int4_weight_only_repack_gb300 as w4

    dev = torch.device("cuda")
    wl = synth.WORKLOADS[args.sweep_config]
    hbm, _ = measured_peaks()
    tc, _ = measured_tc_peak()
    hdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
    for li, (K, N, name) in enumerate(wl.shapes):
        L = synth.make_workload_layer(wl.index, li)
        qweight = torch.from_numpy(L.qweight).to(dev)
        qzeros = torch.from_numpy(L.qzeros).to(dev)
        scales = torch.from_numpy(L.scales.view(np.int16)).to(dev).view(hdt)
        g_idx = torch.from_numpy(L.g_idx).to(dev) if L.g_idx is not None else None
        ncopy = max(2, int(400e6 // alg_bytes(K, N)) + 1)
        if wl.fmt == "gptq":
            layers = [w4.repack_gptq(qweight, qzeros, scales, g_idx, K, N, wl.group, hdt)
                      for _ in range(ncopy)]
        else:
            layers = [w4.repack_awq(qweight, qzeros, scales, K, N, wl.group, hdt)
                      for _ in range(ncopy)]
        del qweight, qzeros, scales
        for M in wl.ms:
            x = torch.randn(M, K, device=dev).to(hdt)
            y = torch.empty((M, N), dtype=hdt, device=dev)
            use = layers if M <= 256 else layers[:2]

            def fn():
                for l in use:
                    w4.linear(x, l, y=y)

            t = graph_time(torch, fn, 10) / len(use)
            gbs = alg_bytes(K, N) / t / 1e9
            tfl = 2.0 * M * N * K / t / 1e12
            print(json.dumps({"sweep": wl.name, "layer": name, "K": K, "N": N, "M": M,
                              "dtype": wl.dtype, "act_order": g_idx is not None,
                              "us": round(t * 1e6, 2), "weight_gbs": round(gbs, 1),
                              "tflops": round(tfl, 1),
                              "frac": round(gbs / hbm if M <= 16 else tfl / tc, 3),
                              "bound": "hbm" if M <= 16 else "tensor"}), flush=True)
            del x, y
        del layers
        torch.cuda.empty_cache()
    print(json.dumps({"sweep_done": wl.name, "device_status": w4.w4_device_status()}), flush=True)


def moe_measure(token_counts, proj="all"):
    """Grouped W4A16 GEMM over an MoE layer's experts (w4a16_moe_gemm): the two
    expert projections of a Mixtral-8x7B-shaped layer (8 experts; w13: K 4096 ->
    N 28672, w2: K 14336 -> N 4096), for batches of `token_counts` tokens, each
    routed top-2 by a seeded draw (rows sorted by expert). One record per
    projection and batch: time of the grouped call (CUDA graph); up to 16 rows
    an expert, weight GB/s over the routed experts' bytes (experts without rows
    are skipped by the kernel), above that TFLOP/s (2 * rows * K * N); and the
    same rows as one w4a16_gemm call per routed expert for comparison."""
    import torch

    import int4_weight_only_repack_gb300 as w4

    dev = torch.device("cuda")
    E, topk = 8, 2
    hbm, _ = measured_peaks()
    tc, _ = measured_tc_peak()
    out = []
    routes = []
    for T in token_counts:
        rng = np.random.default_rng([0, 17] if T == 16 else [0, 17, T])
        choice = np.stack([rng.choice(E, topk, replace=False) for _ in range(T)])
        counts = np.bincount(choice.reshape(-1), minlength=E)
        routes.append((T, counts, np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)))
    for name, K, N in (("w13", 4096, 28672), ("w2", 14336, 4096)):
        if proj not in ("all", name):
            continue
        qws, qzs, scs = [], [], []
        for e in range(E):
            L = synth.make_custom_layer([0, 17, e, K, N], K, N, group=128, dtype="bf16")
            qws.append(torch.from_numpy(L.qweight).to(dev))
            qzs.append(torch.from_numpy(L.qzeros).to(dev))
            scs.append(torch.from_numpy(L.scales.view(np.int16)).to(dev).view(torch.bfloat16))
        experts = w4.repack_awq_experts(qws, qzs, scs, K, N, 128, torch.bfloat16)
        del qws, qzs, scs
        qw_b, z_b, s_b = w4.w4_repack_sizes(K, N, 128, w4.W4_LAYOUT_TILE)
        for T, counts, off in routes:
            rows = int(off[-1])
            x = torch.randn(rows, K, device=dev).to(torch.bfloat16)
            y = torch.empty((rows, N), dtype=torch.bfloat16, device=dev)
            ws = torch.empty(max(1, max(w4.w4a16_gemm_workspace_size(int(c), N, K, 128,
                                                                    torch.bfloat16, False)
                                        for c in counts if c > 0)),
                             dtype=torch.uint8, device=dev)
            offd = torch.from_numpy(off).to(dev)
            mx = int(counts.max())
            reps = 50 if T == 16 else 10
            t_grouped = graph_time(torch, lambda: w4.moe_linear(x, experts, offd, mx, y=y), reps)

            def per_expert():
                for e in range(E):
                    r0, r1 = int(off[e]), int(off[e + 1])
                    if r1 > r0:
                        w4.w4a16_gemm(x[r0:r1], experts.qw[e * qw_b // 4:(e + 1) * qw_b // 4],
                                      experts.scales[e * s_b // 2:(e + 1) * s_b // 2],
                                      experts.zeros[e * z_b // 4:(e + 1) * z_b // 4], None,
                                      y[r0:r1], r1 - r0, N, K, 128, torch.bfloat16,
                                      workspace=ws)

            t_loop = graph_time(torch, per_expert, reps)
            active = int((counts > 0).sum())
            line = {"moe": "mixtral_8x7b_shaped", "proj": name, "K": K, "N": N,
                    "experts": E, "tokens": T, "topk": topk, "rows": rows,
                    "rows_per_expert": counts.tolist(), "routed_experts": active,
                    "kernel": "w4a16_decode_kernel" if mx <= 16 else "w4a16_prefill_kernel",
                    "us": round(t_grouped * 1e6, 2),
                    "per_expert_calls_us": round(t_loop * 1e6, 2)}
            if mx <= 16:
                wb = active * alg_bytes(K, N)
                line["weight_gbs"] = round(wb / t_grouped / 1e9, 1)
                line["frac_hbm"] = round(wb / t_grouped / 1e9 / hbm, 3)
            else:
                tfl = 2.0 * rows * K * N / t_grouped / 1e12
                line["tflops"] = round(tfl, 1)
                line["frac_tc"] = round(tfl / tc, 3)
            line["device_status"] = w4.w4_device_status()
            out.append(line)
            del x, y, ws
        del experts
        torch.cuda.empty_cache()
    return out


def moe(args):
    """--moe: one JSON line per projection and batch (see moe_measure)."""
    for line in moe_measure([int(t) for t in args.moe_tokens.split(",")], args.moe_proj):
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the large-M (prefill) layers")
    ap.add_argument("--no-moe", action="store_true",
                    help="skip the grouped MoE GEMM figures of the default run")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--sweep-config", type=int, default=4, choices=(3, 4),
                    help="workload of --sweep: 4 = Llama-2-70B, 3 = Llama-2-13B GPTQ act-order")
    ap.add_argument("--sweep", action="store_true",
                    help="every layer of --sweep-config at every M of that workload (one line each)")
    ap.add_argument("--moe", action="store_true",
                    help="the grouped MoE GEMM on a Mixtral-8x7B-shaped layer (one line per projection)")
    ap.add_argument("--moe-tokens", default="16,4096",
                    help="comma-separated token counts of --moe (routed top-2 over 8 experts)")
    ap.add_argument("--moe-proj", default="all", choices=("all", "w13", "w2"),
                    help="the projection(s) --moe runs")
    ap.add_argument("--single", default=None,
                    help="K,N,M[,dtype]: time one layer shape only (profiling aid)")
    args = ap.parse_args()
    if args.single:
        single(args)
    elif args.sweep:
        sweep(args)
    elif args.moe:
        moe(args)
    elif args.impl == "reference":
        reference(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
