"""Benchmark of the W4A16 linear layer on GB300 (one JSON line on stdout).

Headline workload (one GPU): the Llama-2-7B decode layers (K, N) = (4096,
12288) qkv, (4096, 4096) o_proj, (4096, 22016) gate_up, (11008, 4096) down,
AWQ group-128 4-bit asymmetric weights, bf16 activations, M in {1, 4, 16}.
One step runs the fused GEMM for every (layer, M) pair: 12 calls. Consecutive
steps alternate between two sets of weight copies (24 copies, about 630 MB,
4.9x the 129 MB L2), so no call finds its weights in L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

value        = weight GB/s of the timed steps (algorithmic bytes per call:
               packed codes K*N/2 + scales G*N*2 + zeros G*N/2), all ranks.
roofline     = the decode kernel in the regime `value` times: each of the 12
               (layer, M) calls timed as a CUDA graph of back-to-back calls over
               rotating weight copies totalling at least 3x L2; achieved = the
               12 calls' algorithmic bytes / the sum of their per-call times,
               against the measured HBM copy bandwidth. `step_frac` is `value`
               against the same peak.
configs      = every workload point, one record each: the 7B decode calls, the
               7B prefill layers (M 512..4096), the Llama-2-13B GPTQ act-order
               layers (fp16, M 1/16/1024) and the Llama-2-70B sweep (M 1..4096).
               Each record: time per call (CUDA graph over rotating copies),
               weight GB/s, TFLOP/s, the roofline the ridge picks (HBM when the
               call's bytes at the measured bandwidth take longer than its
               FLOPs at the measured bf16 tensor peak, else tensor) and the
               fraction of it; beside it the same call as dequantise-then-
               cuBLAS (w4_dequant to a dense [K, N] + torch.matmul) and the CPU
               oracle on a sample of the call (columns, and at most 64 rows),
               extrapolated to the whole call.
e2e          = the headline metric through the public Python API (linear())
               with each step's x copied from pinned host memory and its y
               copied back inside the timed region, eager launches.
cpu_baseline = the CPU oracle (numpy: unpack, dequantise, fp64 matmul) on the
               o_proj layer at M = 1, 4 and 16.
--impl reference times that oracle as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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
L2_ROTATION = 3.0                      # weight copies per timing loop: at least 3x L2

# DRAM bytes per launch of the small-M kernels from ncu (dram__bytes_read.sum +
# dram__bytes_write.sum, the mean over the 12 launches of one step), keyed by
# the sha1 of the kernels' sources they were taken on (kernel_source_hash);
# see profiles/. A changed kernel source reports null.
TRAFFIC_RECORDS: dict = {
    "a97423a79b59": 26429995,   # mean of the 12 launches of one step (10 clustered, 2 streaming)
}


def alg_bytes(K: int, N: int, group: int = 128) -> int:
    G = K // group
    return K * N // 2 + G * N * 2 + G * N // 2


def kernel_source_hash(names=("decode_kernel.cu", "decode_stream_kernel.cu")) -> str:
    """sha1 (first 12 hex digits) of the small-M kernels' sources, in order."""
    h = hashlib.sha1()
    for name in names:
        with open(os.path.join(ROOT, "int4_weight_only_repack_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return json.load(f)
    except Exception:
        return None


def measured_peaks():
    d = _peaks()
    try:
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_tc_peak():
    """Dense bf16 tensor-core peak (burst: every call is timed on its own)."""
    d = _peaks()
    try:
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_TC_TFLOPS, "fallback"


def roofline_point(K, N, M, t, hbm_gbs, tc_tflops):
    """The roofline of one call: its bytes at the HBM peak against its FLOPs at
    the tensor peak; the longer of the two is the bound, frac = ideal / t."""
    tb = alg_bytes(K, N) / (hbm_gbs * 1e9)
    tf = 2.0 * M * N * K / (tc_tflops * 1e12)
    bound = "hbm" if tb >= tf else "tensor"
    return bound, max(tb, tf) / t


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
# Replicas (N > 1)                                                              #
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


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


# --------------------------------------------------------------------------- #
# Layers, weight pools, timing                                                  #
# --------------------------------------------------------------------------- #
class LayerPool:
    """Repacked copies of one synthetic layer (TILE layout) plus a host sample of
    its checkpoint columns for the oracle."""

    def __init__(self, w4, torch, device, cfg, li, n_copies, sample_cols=256):
        wl = synth.WORKLOADS[cfg]
        K, N, name = wl.shapes[li]
        self.K, self.N, self.name, self.cfg = K, N, name, cfg
        self.dtype, self.fmt, self.group = wl.dtype, wl.fmt, wl.group
        self.tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
        seed = 1000 * cfg + li
        qweight, qzeros, scales, g_idx = synth.make_layer_torch(
            seed, K, N, wl.group, wl.dtype, wl.fmt, wl.act_order, device=device)
        nc = min(N, sample_cols)
        # host copy of the first nc columns of the checkpoint (a narrower layer)
        if wl.fmt == "awq":
            self.h_qweight = qweight[:, :nc // 8].cpu().numpy()
        else:
            self.h_qweight = qweight[:, :nc].cpu().numpy()
        self.h_qzeros = qzeros[:, :nc // 8].cpu().numpy()
        self.h_scales = scales[:, :nc].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        self.h_gidx = g_idx.cpu().numpy() if g_idx is not None else None
        self.sample_cols = nc
        self.copies = []
        for _ in range(n_copies):
            if wl.fmt == "gptq":
                self.copies.append(w4.repack_gptq(qweight, qzeros, scales, g_idx, K, N, wl.group,
                                                  self.tdt))
            else:
                self.copies.append(w4.repack_awq(qweight, qzeros, scales, K, N, wl.group,
                                                 self.tdt))
        torch.cuda.synchronize()
        for c in self.copies:
            if c.status is not None and int(c.status[0].item()) != 0:
                raise RuntimeError(f"{name}: act-order repack reported status {int(c.status[0])}")
        del qweight, qzeros, scales, g_idx

    @staticmethod
    def copies_for(K, N, torch, device, minimum=2):
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        return max(minimum, math.ceil(L2_ROTATION * l2 / alg_bytes(K, N)))


def graph_time_reps(torch, fn, reps: int) -> float:
    """Seconds per replay of a CUDA graph of `fn`, median of `reps` replays timed
    one by one with CUDA events on the launch stream (after two warm-up replays)."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for e0, e1 in ev:
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    del g
    return statistics.median(e0.elapsed_time(e1) * 1e-3 for e0, e1 in ev)


def call_time(w4, torch, pool, x, y, copies=None, reps=10):
    """Seconds per w4a16 call: a graph of one call per weight copy (back to back,
    so every call streams a copy that the others have pushed out of L2)."""
    use = pool.copies if copies is None else pool.copies[:copies]

    def fn():
        for l in use:
            w4.linear(x, l, y=y)

    return graph_time_reps(torch, fn, reps) / len(use)


def dequant_cublas_time(w4, torch, pool, x, dense, y2, copies=None, reps=5):
    """Seconds per call of the dequantise-then-cuBLAS path: w4_dequant of the
    call's copy to a dense [K, N] in the activation dtype, then torch.matmul (an
    act-order layer's dense rows come out sorted, so x is gathered by perm first)."""
    use = pool.copies if copies is None else pool.copies[:copies]
    perm = use[0].perm.long() if use[0].perm is not None else None

    def fn():
        for l in use:
            w4.w4_dequant(l.qw, l.scales, l.zeros, pool.K, pool.N, l.group, l.dtype, l.layout,
                          False, dense)
            xs = x if perm is None else torch.index_select(x, 1, perm)
            torch.matmul(xs, dense, out=y2)

    return graph_time_reps(torch, fn, reps) / len(use)


def oracle_sample_time(pool, M, min_seconds=0.05):
    """The CPU oracle on a sample of one call: the pool's first `sample_cols`
    output columns and min(M, 64) rows of x, repeated until `min_seconds`; the
    time is extrapolated to the whole call by N / columns x M / rows."""
    import oracle
    rows = min(M, 64)
    x = synth.make_custom_x([9, pool.cfg, pool.K, rows], rows, pool.K, pool.dtype)
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle.reference_y(x, pool.h_qweight, pool.h_qzeros, pool.h_scales, pool.group,
                           pool.dtype, pool.fmt, g_idx=pool.h_gidx)
        n += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            break
    t = el / n * (pool.N / pool.sample_cols) * (M / rows)
    return {"s_per_call": t, "weight_gbs": round(alg_bytes(pool.K, pool.N) / t / 1e9, 5),
            "sample": f"{pool.sample_cols} of {pool.N} columns x {rows} of {M} rows, "
                      f"extrapolated", "cores": blas_threads()}


def point_record(w4, torch, device, pool, M, hbm, tc, scratch, with_dense=False,
                 with_oracle=True, reps=10):
    """One (layer, M) record: our call, dequantise-then-cuBLAS and the oracle."""
    K, N = pool.K, pool.N
    x = torch.randn(M, K, device=device).to(pool.tdt)
    y = torch.empty((M, N), dtype=pool.tdt, device=device)
    copies = None if M <= 256 else 2
    t = call_time(w4, torch, pool, x, y, copies, reps)
    bound, frac = roofline_point(K, N, M, t, hbm, tc)
    rec = {"layer": pool.name, "K": K, "N": N, "M": M, "us": round(t * 1e6, 2),
           "weight_gbs": round(alg_bytes(K, N) / t / 1e9, 1),
           "tflops": round(2.0 * M * N * K / t / 1e12, 2), "bound": bound,
           "frac": round(frac, 4),
           "weight_copies": len(pool.copies) if copies is None else copies}
    key = (K, N, pool.tdt)
    if key not in scratch:
        scratch.clear()
        torch.cuda.empty_cache()
        scratch[key] = torch.empty((K, N), dtype=pool.tdt, device=device)
    y2 = torch.empty_like(y)
    td = dequant_cublas_time(w4, torch, pool, x, scratch[key], y2,
                             copies=min(len(pool.copies), 3 if M <= 256 else 2), reps=5)
    rec["dequant_cublas_us"] = round(td * 1e6, 2)
    rec["fused_speedup"] = round(td / t, 2)
    if with_dense:
        wd = [torch.randn(K, N, device=device).to(pool.tdt) for _ in range(2)]
        yd = torch.empty_like(y)

        def dense():
            for w in wd:
                torch.matmul(x, w, out=yd)

        tdn = graph_time_reps(torch, dense, 5) / len(wd)
        rec["dense_cublas_us"] = round(tdn * 1e6, 2)
        rec["dense_cublas_tflops"] = round(2.0 * M * N * K / tdn / 1e12, 1)
        del wd, yd
    if with_oracle:
        o = oracle_sample_time(pool, M)
        rec["oracle_weight_gbs"] = o["weight_gbs"]
        rec["oracle_sample"] = o["sample"]
    del x, y, y2
    return rec


def config_records(w4, torch, device, cfg, hbm, tc, with_dense_from=None, with_oracle=True):
    """Records for every (layer, M) of workload `cfg`."""
    wl = synth.WORKLOADS[cfg]
    out = []
    scratch = {}
    for li, (K, N, name) in enumerate(wl.shapes):
        n = LayerPool.copies_for(K, N, torch, device)
        pool = LayerPool(w4, torch, device, cfg, li, n)
        for M in wl.ms:
            dense = with_dense_from is not None and M >= with_dense_from
            out.append(point_record(w4, torch, device, pool, M, hbm, tc, scratch,
                                    with_dense=dense, with_oracle=with_oracle))
        del pool
        torch.cuda.empty_cache()
    scratch.clear()
    torch.cuda.empty_cache()
    return out


def w4a8_records(w4, torch, device, tc, with_oracle=True, reps=10):
    """INT4 weights x per-tensor FP8 activations (w4a8_gemm, tcgen05 kind::f8f6f4)
    on the Llama-2-7B prefill layers at M in {512, 2048, 4096}: TFLOP/s against
    the dense fp8 peak (the measured bf16 peak x 2, the nominal fp8 / bf16
    ratio), beside the W4A16 tcgen05 kernel on the same call and the FP8 oracle
    on a sample of the call."""
    import oracle
    from oracle import fp8_oracle as f8
    fp8_peak = 2.0 * tc
    out = []
    wl = synth.WORKLOADS[2]
    for li, (K, N, name) in enumerate(wl.shapes):
        pool = LayerPool(w4, torch, device, 2, li, 2)
        for M in wl.ms:
            x = torch.randn(M, K, device=device).to(torch.bfloat16)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
            ws = torch.empty(w4.w4a8_gemm_workspace_size(M, K), dtype=torch.uint8, device=device)

            def f8call():
                for l in pool.copies:
                    w4.linear_fp8(x, l, y=y, workspace=ws)

            t = graph_time_reps(torch, f8call, reps) / len(pool.copies)
            t16 = call_time(w4, torch, pool, x, y, None, reps)
            tfl = 2.0 * M * N * K / t / 1e12
            rec = {"layer": name, "K": K, "N": N, "M": M, "us": round(t * 1e6, 2),
                   "tflops": round(tfl, 1), "frac_fp8_peak": round(tfl / fp8_peak, 4),
                   "w4a16_us": round(t16 * 1e6, 2),
                   "note": "includes the two activation-quantisation kernels"}
            if with_oracle:
                rows = min(M, 64)
                xb = synth.make_custom_x([9, 2, K, rows], rows, K, "bf16")
                t0 = time.perf_counter()
                f8.reference_y_w4a8(xb, pool.h_qweight, pool.h_qzeros, pool.h_scales, 128, "bf16")
                el = time.perf_counter() - t0
                tor = el * (N / pool.sample_cols) * (M / rows)
                rec["oracle_tflops"] = round(2.0 * M * N * K / tor / 1e12, 6)
                rec["oracle_sample"] = f"{pool.sample_cols} of {N} columns x {rows} of {M} rows, extrapolated"
            out.append(rec)
            del x, y, ws
        del pool
        torch.cuda.empty_cache()
    return {"workload": "llama2_7b_prefill layers, bf16 activations quantised per tensor to e4m3",
            "peak": {"fp8_tflops": fp8_peak, "source": "measured bf16 dense peak x 2 (nominal fp8/bf16)"},
            "per_call": out}


def repack_measure(w4, torch, device, reps=5):
    """Throughput of the one-time AWQ -> TILE repack on the Llama-2-70B gate_up
    layer (K 8192, N 57344): bytes read (qweight, qzeros, scales) + written
    (TILE words, zeros, scales) per call / time (CUDA events around one call)."""
    K, N, g = 8192, 57344, 128
    qweight, qzeros, scales, _ = synth.make_layer_torch(4001, K, N, g, "bf16", device=device)
    qw_b, z_b, s_b = w4.w4_repack_sizes(K, N, g, w4.W4_LAYOUT_TILE)
    outs = [(torch.empty(qw_b // 4, dtype=torch.int32, device=device),
             torch.empty(z_b // 4, dtype=torch.int32, device=device),
             torch.empty(s_b // 2, dtype=torch.bfloat16, device=device)) for _ in range(2)]
    times = []
    for r in range(reps + 1):
        qw, zz, ss = outs[r % 2]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        w4.w4_repack_awq(qweight, qzeros, scales, K, N, g, torch.bfloat16, w4.W4_LAYOUT_TILE,
                         qw, zz, ss)
        e1.record()
        torch.cuda.synchronize()
        if r:
            times.append(e0.elapsed_time(e1) * 1e-3)
    t = statistics.median(times)
    moved = (K * N // 2 + z_b + s_b) * 2
    hbm, _ = measured_peaks()
    del qweight, qzeros, scales, outs
    torch.cuda.empty_cache()
    return {"layer": "llama2_70b gate_up (8192 x 57344), AWQ -> TILE", "us": round(t * 1e6, 1),
            "gbs": round(moved / t / 1e9, 1), "frac_hbm": round(moved / t / 1e9 / hbm, 4),
            "bytes": moved, "how": "w4_repack_awq (unpack + TILE words, zeros, scales + the "
                                   "stream-ordering kernel), CUDA events around one call, median"}


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


# --------------------------------------------------------------------------- #
# Our arm                                                                       #
# --------------------------------------------------------------------------- #
def ours(args):
    import torch

    import int4_weight_only_repack_gb300 as w4

    world, rank, local = setup_dist()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    w4.lib()
    hbm, hbm_src = measured_peaks()
    tc, tc_src = measured_tc_peak()

    # ---- the headline step: 12 calls, two sets of weight copies -----------------
    pools = []
    for li, (K, N, _) in enumerate(WORKLOAD.shapes):
        n = LayerPool.copies_for(K, N, torch, device, minimum=2 * len(WORKLOAD.ms))
        pools.append(LayerPool(w4, torch, device, WORKLOAD.index, li, n))
    calls = []
    for li, pool in enumerate(pools):
        for mi, M in enumerate(WORKLOAD.ms):
            x_bits = synth.make_workload_x(WORKLOAD.index, li, M)
            calls.append(dict(pool=pool, li=li, M=M, mi=mi, x_bits=x_bits))
    # every step's inputs live in one buffer (and its outputs in another) so the
    # end-to-end pass moves them with one copy each way
    x_elems = sum(c["M"] * c["pool"].K for c in calls)
    y_elems = sum(c["M"] * c["pool"].N for c in calls)
    x_all = torch.empty(x_elems, dtype=torch.bfloat16, device=device)
    y_all = torch.empty(y_elems, dtype=torch.bfloat16, device=device)
    hx_all = torch.empty(x_elems, dtype=torch.bfloat16).pin_memory()
    hy_all = torch.empty(y_elems, dtype=torch.bfloat16).pin_memory()
    xo = yo = 0
    for c in calls:
        K, N, M = c["pool"].K, c["pool"].N, c["M"]
        hx_all[xo:xo + M * K].copy_(torch.from_numpy(c["x_bits"].view(np.int16).reshape(-1))
                                    .view(torch.bfloat16))
        c["x"] = x_all[xo:xo + M * K].view(M, K)
        c["y"] = y_all[yo:yo + M * N].view(M, N)
        xo += M * K
        yo += M * N
    x_all.copy_(hx_all)
    nsets = 2

    def step_fn(s):
        def fn():
            for c in calls:
                layer = c["pool"].copies[(c["mi"] + len(WORKLOAD.ms) * s) % len(c["pool"].copies)]
                w4.linear(c["x"], layer, y=c["y"])
        return fn

    step_bytes = sum(alg_bytes(c["pool"].K, c["pool"].N) for c in calls)
    step_flops = sum(2 * c["M"] * c["pool"].N * c["pool"].K for c in calls)
    for _ in range(max(args.warmup, 3)):
        for s in range(nsets):
            step_fn(s)()
    torch.cuda.synchronize()
    graphs = []
    for s in range(nsets):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step_fn(s)()
        graphs.append(g)
    for _ in range(max(args.warmup, 3)):
        for g in graphs:
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
    for i in range(args.steps):
        graphs[i % nsets].replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    elapsed = max_over_ranks(e0.elapsed_time(e1) * 1e-3, world, device)
    del graphs

    # ---- the decode kernel per call, graph-timed over >= 3x L2 of copies --------
    scratch = {}
    per_call = []
    for c in calls:
        rec = point_record(w4, torch, device, c["pool"], c["M"], hbm, tc, scratch,
                           with_oracle=rank == 0 and not args.no_cpu_baseline, reps=20)
        per_call.append(rec)
    scratch.clear()
    kern_time = sum(r["us"] for r in per_call) * 1e-6
    achieved = step_bytes / kern_time / 1e9
    traffic = TRAFFIC_RECORDS.get(kernel_source_hash())

    # ---- end to end through the public API, host buffers ------------------------
    # Every step copies its inputs in from pinned host memory and its results
    # out to pinned host memory. The copies run on a copy stream with two sets
    # of device buffers, so that a step's copies overlap the neighbouring steps'
    # GEMMs, as a serving loop would arrange them; events order every copy
    # against the GEMMs that read or write its buffers.
    e2e_steps = min(args.steps, 200)
    comp = torch.cuda.current_stream()
    cps = torch.cuda.Stream(device=device)
    xsets = [x_all, torch.empty_like(x_all)]
    ysets = [y_all, torch.empty_like(y_all)]
    hys = [hy_all, torch.empty(y_elems, dtype=torch.bfloat16).pin_memory()]
    views = []
    for b in range(2):
        xo = yo = 0
        vs = []
        for c in calls:
            K, N, M = c["pool"].K, c["pool"].N, c["M"]
            vs.append((xsets[b][xo:xo + M * K].view(M, K), ysets[b][yo:yo + M * N].view(M, N)))
            xo += M * K
            yo += M * N
        views.append(vs)
    h2d_done = [torch.cuda.Event(), torch.cuda.Event()]
    comp_done = [torch.cuda.Event(), torch.cuda.Event()]
    d2h_done = [torch.cuda.Event(), torch.cuda.Event()]

    def issue_h2d(s):
        b = s % 2
        with torch.cuda.stream(cps):
            if s >= 2:
                cps.wait_event(comp_done[b])  # the GEMMs of step s - 2 have read set b
            xsets[b].copy_(hx_all, non_blocking=True)
            h2d_done[b].record(cps)

    def e2e_step(s, last):
        b = s % 2
        comp.wait_event(h2d_done[b])
        if s >= 2:
            comp.wait_event(d2h_done[b])  # step s - 2's results have left set b
        for c, (xv, yv) in zip(calls, views[b]):
            layer = c["pool"].copies[(c["mi"] + len(WORKLOAD.ms) * (s % nsets)) % len(c["pool"].copies)]
            w4.linear(xv, layer, y=yv)
        comp_done[b].record(comp)
        with torch.cuda.stream(cps):
            cps.wait_event(comp_done[b])
            hys[b].copy_(ysets[b], non_blocking=True)
            d2h_done[b].record(cps)
        if s + 2 < last:
            issue_h2d(s + 2)

    def e2e_run(n):
        issue_h2d(0)
        if n > 1:
            issue_h2d(1)
        for s in range(n):
            e2e_step(s, n)

    e2e_run(2 * nsets)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    e2e_run(e2e_steps)
    torch.cuda.synchronize()
    e2e_el = max_over_ranks(time.perf_counter() - t0, world, device)

    # ---- comparison: the same step as dequantise-then-cuBLAS ---------------------
    t_deq = sum(r["dequant_cublas_us"] for r in per_call) * 1e-6
    del pools, calls
    torch.cuda.empty_cache()

    # ---- the other workloads, one record per (layer, M) ---------------------------
    configs = {"llama2_7b_decode": per_call}
    prefill = None
    if not args.no_configs and world == 1:
        oracle_on = rank == 0 and not args.no_cpu_baseline
        configs["llama2_7b_prefill"] = config_records(w4, torch, device, 2, hbm, tc,
                                                      with_dense_from=512, with_oracle=oracle_on)
        configs["llama2_13b_gptq_act_order"] = config_records(w4, torch, device, 3, hbm, tc,
                                                              with_oracle=oracle_on)
        configs["llama2_70b_sweep"] = config_records(w4, torch, device, 4, hbm, tc,
                                                     with_dense_from=1024, with_oracle=oracle_on)
        big = [r for r in configs["llama2_7b_prefill"] if r["M"] >= 2048]
        flops = sum(2.0 * r["M"] * r["K"] * r["N"] for r in big)
        tsum = sum(r["us"] for r in big) * 1e-6
        dense = sum(r["dense_cublas_us"] for r in big) * 1e-6
        prefill = {"workload": "llama2_7b_prefill at M in {2048, 4096}, bf16",
                   "tflops_m_ge_2048": round(flops / tsum / 1e12, 1),
                   "vs_dense_bf16_cublas": round(dense / tsum, 3),
                   "roofline": {"bound": "tensor", "achieved": round(flops / tsum / 1e12, 1),
                                "peak": tc, "unit": "TFLOP/s",
                                "frac": round(flops / tsum / 1e12 / tc, 4),
                                "peak_source": tc_src, "kernel": "w4a16_prefill_kernel"}}

    w4a8 = None
    if world == 1 and not args.no_configs:
        w4a8 = w4a8_records(w4, torch, device, tc, with_oracle=rank == 0 and not args.no_cpu_baseline)

    moe_part = None
    if world == 1 and not args.no_moe:
        moe_part = {"workload": "mixtral_8x7b_shaped experts (8; w13 4096->28672, w2 "
                                "14336->4096), 16 and 4096 tokens routed top-2, bf16, "
                                "one w4a16_moe_gemm call against one w4a16_gemm per expert",
                    "per_call": moe_measure((16, 4096))}
    repack = repack_measure(w4, torch, device) if world == 1 else None

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
                "calls_per_step": len(per_call),
                "weight_bytes_per_step": step_bytes,
                "l2": "inputs larger than L2: consecutive steps alternate between two sets of "
                      "12 weight copies (%.0f MB per set, %.0f MB in all)"
                      % (step_bytes / 1e6, nsets * step_bytes / 1e6),
                "timing": "CUDA graph of one step per set, replayed alternately; CUDA events on "
                          "the launch stream",
                "parallelism": "replicas" if world > 1 else "single GPU",
            },
            "tflops": round(step_flops * args.steps * world / elapsed / 1e12, 4),
            "gpu_launches": len(per_call) * args.steps,
            "clocks": clocks,
            "e2e": {"value": round(step_bytes * e2e_steps * world / e2e_el / 1e9, 2),
                    "unit": "GB/s", "h2d_bytes_per_step": x_elems * 2,
                    "d2h_bytes_per_step": y_elems * 2, "steps": e2e_steps,
                    "how": "linear() per call, eager; each step's x in one pinned-host -> "
                           "device copy and its y in one device -> pinned-host copy, on a "
                           "copy stream with two sets of device buffers, so that a step's "
                           "copies overlap the neighbouring steps' GEMMs"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
                         "unit": "GB/s", "frac": round(achieved / hbm, 4),
                         "traffic": traffic, "peak_source": hbm_src,
                         "kernel": "w4a16_decode_kernel",
                         "step_frac": round(value / world / hbm, 4),
                         "how": "each (layer, M) call as a CUDA graph of back-to-back calls over "
                                ">= 3x L2 of weight copies; achieved = the step's bytes / the sum "
                                "of the 12 per-call times (records under configs)"},
            "cpu_baseline": cpu_base,
            "dequant_cublas": {"value": round(step_bytes / t_deq / 1e9, 2), "unit": "GB/s",
                               "ms_per_step": round(t_deq * 1e3, 5),
                               "fused_speedup": round(t_deq / (elapsed / args.steps), 2),
                               "how": "sum over the 12 calls of w4_dequant to dense bf16 [K,N] + "
                                      "torch.matmul (cuBLAS), each graph-timed over weight copies"},
            "prefill": prefill,
            "configs": configs,
            "roofline_peaks": {"hbm_gbs": hbm, "bf16_tflops": tc, "source": hbm_src,
                               "ridge_M": round(tc * 1e12 / (4 * hbm * 1e9), 1),
                               "note": "fp16 calls use the bf16 figure (the same dense rate)"},
            "w4a8": w4a8,
            "moe": moe_part,
            "repack": repack,
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
    """One call shape repeated `--steps` times (for profiler captures):
    --single K,N,M[,dtype[,fp8]]; fp8 runs w4a8_gemm instead of w4a16_gemm. The
    layer is repacked once (AWQ -> TILE) before the calls."""
    import torch

    import int4_weight_only_repack_gb300 as w4

    parts = args.single.split(",")
    K, N, M = int(parts[0]), int(parts[1]), int(parts[2])
    dtype = parts[3] if len(parts) > 3 else "bf16"
    fp8 = len(parts) > 4 and parts[4] == "fp8"
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    dev = torch.device("cuda")
    qweight, qzeros, scales, _ = synth.make_layer_torch(5, K, N, 128, dtype, device=dev)
    layer = w4.repack_awq(qweight, qzeros, scales, K, N, 128, tdt)
    x = torch.randn(M, K, device=dev).to(tdt)
    y = torch.empty((M, N), dtype=tdt, device=dev)
    fn = (lambda: w4.linear_fp8(x, layer, y=y)) if fp8 else (lambda: w4.linear(x, layer, y=y))
    fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) * 1e-3 / max(1, args.steps)
    print(json.dumps({"single": [K, N, M, dtype, "fp8" if fp8 else "w4a16"],
                      "us_per_call": round(t * 1e6, 2),
                      "weight_gbs": round(alg_bytes(K, N) / t / 1e9, 1),
                      "tflops": round(2.0 * M * N * K / t / 1e12, 2),
                      "device_status": w4.w4_device_status()}), flush=True)


def sweep(args):
    """Every (layer, M) record of one workload, one JSON line each (the same
    records the default line carries under `configs`)."""
    import torch

    import int4_weight_only_repack_gb300 as w4

    dev = torch.device("cuda")
    w4.lib()
    hbm, _ = measured_peaks()
    tc, _ = measured_tc_peak()
    wl = synth.WORKLOADS[args.sweep_config]
    for rec in config_records(w4, torch, dev, args.sweep_config, hbm, tc,
                              with_oracle=not args.no_cpu_baseline):
        print(json.dumps({"sweep": wl.name, **rec}), flush=True)
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
            qw_e, qz_e, sc_e, _ = synth.make_layer_torch(17000 + 100 * e + (K // 1024), K, N, 128,
                                                         "bf16", device=dev)
            qws.append(qw_e)
            qzs.append(qz_e)
            scs.append(sc_e)
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
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip every CPU oracle timing (the headline baseline and the samples)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the prefill, act-order and 70B records of the default run")
    ap.add_argument("--no-moe", action="store_true",
                    help="skip the grouped MoE GEMM figures of the default run")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--sweep-config", type=int, default=4, choices=(2, 3, 4),
                    help="workload of --sweep: 2 = Llama-2-7B prefill, 3 = Llama-2-13B GPTQ "
                         "act-order, 4 = Llama-2-70B")
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
