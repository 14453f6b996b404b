#!/usr/bin/env python
"""Benchmark of the k-quant prefill matmul on one GB300 (or N replicas).

One step = the whole hot path on one batch, one call (qgemm_q4k_f32): fp32
activations quantized to Q8_K, then the Q4_K x Q8_K GEMM.  Above the small-M
path the quantizer also writes the tile GEMM's fp16 operand planes and the
tcgen05 tile GEMM starts under it; for M <= 8 the small-M streaming kernel
runs, and for M <= 2 it quantizes the activations itself (one launch).
PTQ1_0 workloads call qgemm_ptq1_f32, routed ones quantize and then call the
routed GEMM.  Default workload: the
largest configuration, the Q4_K sweep point M = 8192 tokens, K = N = 5120,
X ~ N(0,1); synthetic, seeded (synth.py).  --workload picks another.

Metric: effective TOPS = 2*M*N*K / step time (the whole job over all ranks);
weight GB/s and the tile GEMM's roofline fraction are reported beside it.

Timing: W untimed warm-up steps, then exactly K steps, each bracketed by CUDA
events on the launching stream, with L2 flushed before every step (a 256 MiB
write and then a 256 MiB read of another buffer, outside the events, so that
the step starts with its inputs in DRAM and no dirty lines of the flush left
in L2 to write back); barrier + synchronize on both sides; the slowest
rank's mean is the step time.  A step is replayed as one CUDA graph captured
from the API calls (--no-graph: the eager calls), which removes the host-side
gaps between its kernels.  The same K steps then run once more as eager calls,
with the GEMM kernel alone timed by events the library records around its
launch (qgemm_set_profile_events).

End to end (the "e2e" key): the same steps through the same API calls, with X
(and a routed step's expert ids) starting in pinned host memory and Y ending
there.  The library's kernels read X and write Y across the host link
themselves (zero-copy).  The same step with cudaMemcpyAsync copies of X and Y
around the device step is reported beside it (e2e.copies).  Both count the
bytes that cross the link each step.

--impl reference times the CPU oracle (the parity authority) on bounded
samples of the same workload on the host cores (token rows partitioned over
all of them): the reference arm.  The GPU arm's cpu_baseline is the same
all-core oracle on a larger sample, with the single-core oracle beside it.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "k-quant GEMM effective TOPS and weight GB/s vs roofline at prefill M"
UNIT = "TOPS"
DEFAULT_WORKLOAD = synth.sweep(8192).name

# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the dominant
# kernel (the first GEMM launch of the run, after an L2 flush), from the ncu
# captures summarised in profiles/dram_traffic_by_workload.md (absent until
# measured, and removed whenever the kernel changes).
NCU_TRAFFIC_BYTES = {
    "q4k_sweep_m8192_k5120_n5120": 302274048,
    "q4k_sweep_m2048_k5120_n5120": 54499840,
    "q4k_sweep_m512_k5120_n5120": 27387904,
    "q4k_sweep_m64_k5120_n5120": 15517440,
    "q4k_sweep_m8_k5120_n5120": 14830080,
    "q4k_sweep_m4_k5120_n5120": 14810880,
    "q4k_sweep_m1_k5120_n5120": 14807552,
    "q4k_m64_k2048_n2048": 2709760,
    "q4k_m512_k2048_n11008_outliers": 20983040,
    "q6k_m512_k11008_n2048": 31299072,
    "q6k_fullscale_m512_k11008_n2048": 31300608,
    "q4k_m2048_k4096_n14336": 139535872,
    "q4k_moe_e8_top2_m512_k4096_n14336": 318473728,
    "ptq1_m2048_k5120_n5120": 32066560,
}


def quantize_report(M, K, us, with_planes, hbm_gbs):
    """The quantizer's own line: algorithmic bytes (fp32 X read, Q8_K written:
    (4 + 292/256) bytes per element) over its event time, against HBM."""
    if us is None:
        return {"kernel": "none: the small-M kernel quantizes X itself (one launch per step)"}
    algo = (4.0 + 292.0 / 256.0) * M * K
    planes = (2.0 + 2.0 / 16.0) * M * K + (K // 256) * ((M + 3) // 4 * 4) * 4.0 if with_planes else 0.0
    gbs = algo / (us * 1e-6) / 1e9
    return {"kernel": "quantize_q8k_kernel" + (" (also writes the tile GEMM's operand planes)" if with_planes else ""),
            "us": us, "algorithmic_bytes": algo, "achieved_gbs": gbs, "frac_hbm": gbs / float(hbm_gbs),
            "bytes_moved_incl_operand_planes": algo + planes,
            "gbs_incl_operand_planes": (algo + planes) / (us * 1e-6) / 1e9}


def workloads():
    return {w.name: w for w in synth.CONFIGS + synth.FULLSCALE_CONFIGS + synth.ROUTED_CONFIGS + synth.PTQ1_CONFIGS}


def routed(wl) -> bool:
    return isinstance(wl, synth.RoutedWorkload)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampled every 100 ms in the background."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_id}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [s.strip() for s in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        if not self.samples:
            return None
        win = [s for t, s in self.samples if t0 <= t <= t1]
        widened = False
        if len(win) < 3:
            win = [s for t, s in self.samples if t0 - 2.0 <= t <= t1 + 0.2]
            widened = True
        if not win:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm, smax = [], []
        for s in win:
            try:
                sm.append(float(s[1]))
                smax.append(float(s[2]))
            except (ValueError, IndexError):
                continue
            for i, n in enumerate(names):
                if len(s) > 5 + i and s[5 + i].lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
               "samples": len(sm)}
        if widened:
            out["window"] = "timed region plus the 2 s of warm-up before it (timed region shorter than 3 samples)"
        return out


def gpu_id_for_smi(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


# ------------------------------------------------------------------ CPU oracle
def oracle_sample(wl, rows, x=None, w=None):
    """Time the CPU oracle (quantize + GEMM) on `rows` token rows; returns (seconds, ops)."""
    import oracle
    orc = oracle.get()
    w = wl.weights() if w is None else w
    x = wl.x() if x is None else x
    xs = np.ascontiguousarray(x[:rows])
    if routed(wl):
        ids = np.ascontiguousarray(wl.ids()[:rows])
        t = time.perf_counter()
        qs, d, bs = orc.quantize_q8k(xs)
        orc.gemm_id(wl.wtype, w, wl.E, wl.K, qs, d, bs, ids)
        dt = time.perf_counter() - t
        return dt, 2.0 * rows * wl.top_k * wl.N * wl.K
    t = time.perf_counter()
    qs, d, bs = orc.quantize_q8k(xs)
    orc.gemm(wl.wtype, w, wl.K, qs, d, bs)
    dt = time.perf_counter() - t
    return dt, 2.0 * rows * wl.N * wl.K


# The oracle on all host cores: the token rows are partitioned over a pool of
# single-threaded oracle processes (started with spawn, so that no worker is
# forked from a process that holds a CUDA context).  Each worker builds the
# workload's weights once; a task is (X rows, their expert ids or None).
_POOL_W = None
_POOL_WL = None


def _pool_init(name):
    global _POOL_W, _POOL_WL
    _POOL_WL = workloads()[name]
    _POOL_W = _POOL_WL.weights()
    import oracle
    oracle.get()


def _pool_rows(task):
    import oracle
    orc = oracle.get()
    xs, ids = task
    qs, d, bs = orc.quantize_q8k(xs)
    if ids is not None:
        orc.gemm_id(_POOL_WL.wtype, _POOL_W, _POOL_WL.E, _POOL_WL.K, qs, d, bs, ids)
    else:
        orc.gemm(_POOL_WL.wtype, _POOL_W, _POOL_WL.K, qs, d, bs)
    return len(xs)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OraclePool:
    """`cores` oracle processes; run(rows) times quantize + GEMM of the first
    `rows` token rows, split evenly over the processes (wall clock)."""

    def __init__(self, wl, x, cores):
        import multiprocessing as mp
        self.wl, self.x, self.cores = wl, x, cores
        self.ids = wl.ids() if routed(wl) else None
        self.pool = mp.get_context("spawn").Pool(cores, initializer=_pool_init, initargs=(wl.name,))

    def run(self, rows):
        chunks = [c for c in np.array_split(np.arange(rows), self.cores) if len(c)]
        tasks = [(np.ascontiguousarray(self.x[c]), None if self.ids is None else np.ascontiguousarray(self.ids[c]))
                 for c in chunks]
        t = time.perf_counter()
        done = sum(self.pool.map(_pool_rows, tasks))
        dt = time.perf_counter() - t
        per_row = 2.0 * self.wl.N * self.wl.K * (self.wl.top_k if self.ids is not None else 1)
        return dt, done * per_row

    def close(self):
        self.pool.close()
        self.pool.join()


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    wl = workloads()[args.workload]
    x = wl.x()
    cores = host_cores()
    rows = min(wl.M, args.ref_rows * cores)
    pool = OraclePool(wl, x, cores)
    for _ in range(args.warmup):
        pool.run(rows)
    ts, ops = [], 0.0
    for _ in range(args.steps):
        dt, ops = pool.run(rows)
        ts.append(dt)
    pool.close()
    mean = sum(ts) / len(ts)
    value = ops / mean / 1e12
    sample = (f"{rows} of {wl.M} token rows per step, split over {cores} oracle processes "
              f"(quantize + GEMM over all N={wl.N}, K={wl.K})")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(wl):
    c = {"workload": wl.name, "weights": {4: "Q4_K", 6: "Q6_K", 1: "PTQ1_0"}[wl.wtype], "M": wl.M, "K": wl.K,
         "N": wl.N, "x": f"{wl.sigma}*N(0,1)" + (", 1% columns x8" if getattr(wl, "outlier_frac", 0) else ""),
         "l2": "flushed before every step, outside the timed events: a 256 MiB write, then a 256 MiB read of "
               "another buffer (L2 left holding clean lines the step never touches)"}
    if routed(wl):
        c.update({"experts": wl.E, "top_k": wl.top_k, "routing": f"synthetic top-{wl.top_k}, skew {wl.skew}",
                  "routed_rows": wl.M * wl.top_k})
    return c


def max_over_ranks(values, world, device):
    """Each rank's timings -> the slowest rank's, element by element (the job
    lasts as long as its slowest replica).  One all-reduce of the whole list."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def job_tops(world, ops_per_rank, ms):
    """Whole-job throughput under weak scaling: the work of all `world` ranks
    over the slowest rank's time per step (ms)."""
    return world * ops_per_rank / (ms * 1e-3) / 1e12


# ------------------------------------------------------------------ GPU arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads()))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=512,
                    help="token rows of the single-core CPU-baseline sample (the all-core one: this many per core)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline runs until this much time")
    ap.add_argument("--ref-rows", type=int, default=2, help="token rows per host core in a reference-arm step")
    ap.add_argument("--no-graph", action="store_true", help="time the eager API calls instead of a graph replay")
    ap.add_argument("--settle", type=float, default=0.5,
                    help="seconds of extra untimed steps after warm-up (clock settling); 0 = none")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch
    import torch.distributed as dist
    import block_quantized_matmul_quantize_gb300 as qg

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()

    wl = workloads()[args.workload]
    assert wl.wtype in (4, 6, 1)
    M, N, K = wl.M, wl.N, wl.K
    w_host, x_host = wl.weights(), wl.x()
    dev = torch.device("cuda", local)
    is_routed = routed(wl)
    rows_out = M * wl.top_k if is_routed else M           # output rows (routed: one per token and slot)
    w = torch.from_numpy(w_host).to(dev)
    if wl.wtype == 6:
        w = qg.qgemm_q6k_prepack(w, w_host.shape[0], K)
    elif wl.wtype == 1:
        w = qg.qgemm_ptq1_prepack(w, w_host.shape[0], K)
    x = torch.from_numpy(x_host).to(dev)
    q = qg.Q8K.empty(M, K, dev)
    y = torch.empty((rows_out, N), dtype=torch.float32, device=dev)
    if is_routed:
        ids = torch.from_numpy(wl.ids()).to(dev)
        ws = torch.empty(max(qg.qgemm_id_workspace_bytes(M, wl.top_k, wl.E, K), 256), dtype=torch.uint8, device=dev)
    else:
        ws = torch.empty(max(qg.qgemm_workspace_bytes(M, N, K), 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(64 << 20, dtype=torch.int32, device=dev)

    def flush_l2():
        # Outside the timed region: write a 256 MiB buffer, then read another
        # 256 MiB one.  L2 (129 MB) then holds only clean lines of a buffer
        # the step never touches, so the step's inputs come from DRAM and its
        # kernels do not pay for writing back the flush buffer's dirty lines.
        flush.zero_()
        flush_r.max()
    stream = torch.cuda.current_stream()

    def step_on(xin, yout, ids_in=None):
        if is_routed:
            # quantize, then route + gather + one tile GEMM over all experts
            qg.qgemm_quantize_q8k(xin, out=q)
            if wl.wtype == 4:
                qg.qgemm_q4k_id(w, wl.E, N, K, q, ids_in, y=yout, workspace=ws)
            else:
                qg.qgemm_q6k_id(w, wl.E, N, K, q, ids_in, y=yout, workspace=ws)
            return
        if wl.wtype == 1:
            qg.qgemm_ptq1_f32(w, N, K, xin, out=q, y=yout, workspace=ws)
            return
        # fp32 X in, Y out, one call: for M <= 2 one launch (the small-M kernel
        # quantizes X itself), else the quantizer (writing the GEMM's operand
        # planes in the same launch) and the GEMM started under it
        if wl.wtype == 4:
            qg.qgemm_q4k_f32(w, N, K, xin, out=q, y=yout, workspace=ws)
        else:
            qg.qgemm_q6k_f32(w, N, K, xin, out=q, y=yout, workspace=ws)

    def step():
        step_on(x, y, ids if is_routed else None)

    sampler = ClockSampler(gpu_id_for_smi(local))
    # warm-up, then about half a second more so that clocks settle
    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    t_end = time.time() + args.settle
    while time.time() < t_end:
        for _ in range(20):
            flush_l2()
            step()
        torch.cuda.synchronize()

    # The step's launches (quantize, operand preparation, GEMM) captured once as
    # a CUDA graph: the same kernels with the same arguments, replayed without
    # the host-side gaps between them.
    graph = None
    if not args.no_graph:
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(3):
                step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize()

    K_steps = args.steps
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(K_steps)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(K_steps)]
    ex_s = [torch.cuda.Event(enable_timing=True) for _ in range(K_steps)]
    ex_e = [torch.cuda.Event(enable_timing=True) for _ in range(K_steps)]
    gb = [torch.cuda.Event(enable_timing=True) for _ in range(K_steps)]
    ga = [torch.cuda.Event(enable_timing=True) for _ in range(K_steps)]
    for e in gb + ga:      # create the events (torch creates them lazily on first record)
        e.record()
    torch.cuda.synchronize()

    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    # timed steps (graph replay, or the eager calls with --no-graph)
    for i in range(K_steps):
        flush_l2()
        ev_s[i].record(stream)
        if graph is not None:
            graph.replay()
        else:
            step()
        ev_e[i].record(stream)
    torch.cuda.synchronize()
    # the same steps through the eager API calls, with the GEMM launch timed alone
    c0 = qg.qgemm_get_counters()
    for i in range(K_steps):
        flush_l2()
        qg.qgemm_set_profile_events(gb[i], ga[i])
        ex_s[i].record(stream)
        step()
        ex_e[i].record(stream)
    torch.cuda.synchronize()
    barrier()
    t1 = time.time()
    qg.qgemm_set_profile_events(None, None)
    c1 = qg.qgemm_get_counters()
    sampler.stop()

    step_ms = [ev_s[i].elapsed_time(ev_e[i]) for i in range(K_steps)]
    eager_ms = [ex_s[i].elapsed_time(ex_e[i]) for i in range(K_steps)]
    gemm_ms = [gb[i].elapsed_time(ga[i]) for i in range(K_steps)]
    mean_ms = sum(step_ms) / K_steps
    eager_mean_ms = sum(eager_ms) / K_steps
    gemm_mean_ms = sum(gemm_ms) / K_steps
    mean_ms, gemm_mean_ms, eager_mean_ms = max_over_ranks([mean_ms, gemm_mean_ms, eager_mean_ms], world, dev)

    ops = 2.0 * rows_out * N * K
    value = job_tops(world, ops, mean_ms)
    # library kernels per step, counted on the eager pass; the graph replays the same ones
    # (a routed GEMM call is three: routing, operand gather, tile GEMM)
    per_step = sum(c1[k] - c0[k] for k in ("quantize", "xprep", "q4k_tc", "q6k_tc", "q4k_small", "q6k_small",
                                            "ptq1_tc", "q4k_side"))
    per_step += 2 * (c1["routed"] - c0["routed"])
    launches = per_step  # == K_steps x kernels per step, the count in each of the two timed loops

    # ---- end to end through the public API with host buffers.  The inputs (X, and
    # the expert ids of a routed step) start in pinned host memory and Y ends
    # there, both crossing the host link inside the timed region.  Two ways:
    #   zero-copy: the quantizer reads X and the GEMM's epilogue writes Y in
    #              host memory directly (the library's kernels move the bytes);
    #   copies:    cudaMemcpyAsync of X to the device, the step, and a copy of Y back.
    x_pin = torch.from_numpy(x_host).pin_memory()
    y_pin = torch.empty((rows_out, N), dtype=torch.float32).pin_memory()
    ids_pin = torch.from_numpy(wl.ids()).pin_memory() if is_routed else None
    h2d_bytes = int(x_host.nbytes) + (int(ids_pin.nbytes) if is_routed else 0)
    d2h_bytes = int(rows_out * N * 4)

    def e2e_zero_copy():
        step_on(x_pin, y_pin, ids_pin)

    def e2e_copies():
        x.copy_(x_pin, non_blocking=True)
        if is_routed:
            ids.copy_(ids_pin, non_blocking=True)
        step()
        y_pin.copy_(y, non_blocking=True)

    def time_e2e(fn):
        e_s = [torch.cuda.Event(enable_timing=True) for _ in range(K_steps)]
        e_e = [torch.cuda.Event(enable_timing=True) for _ in range(K_steps)]
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        barrier()
        for i in range(K_steps):
            flush_l2()
            e_s[i].record(stream)
            fn()
            e_e[i].record(stream)
        torch.cuda.synchronize()
        barrier()
        ms = sum(e_s[i].elapsed_time(e_e[i]) for i in range(K_steps)) / K_steps
        return max_over_ranks([ms], world, dev)[0]

    e2e_ms = time_e2e(e2e_zero_copy)
    e2e_copies_ms = time_e2e(e2e_copies)
    e2e_value = job_tops(world, ops, e2e_ms)
    e2e_copies_value = job_tops(world, ops, e2e_copies_ms)

    # ---- the quantizer alone, reported against HBM: the launch the step's call
    # makes for this workload (with the tile GEMM's operand planes when the
    # tile GEMM follows; none when the small-M kernel quantizes X itself)
    fused_small = c1["small_fused"] > c0["small_fused"]
    tile_next = not is_routed and any(c1[k] > c0[k] for k in ("q4k_tc", "q6k_tc", "ptq1_tc"))
    quant_us = None
    if not fused_small:
        def quant_only():
            if tile_next:
                qg.qgemm_quantize_q8k_prep(x, ws, out=q)
            else:
                qg.qgemm_quantize_q8k(x, out=q)
        for _ in range(3):
            quant_only()
        q_s = [torch.cuda.Event(enable_timing=True) for _ in range(K_steps)]
        q_e = [torch.cuda.Event(enable_timing=True) for _ in range(K_steps)]
        torch.cuda.synchronize()
        for i in range(K_steps):
            flush_l2()
            q_s[i].record(stream)
            quant_only()
            q_e[i].record(stream)
        torch.cuda.synchronize()
        quant_us = max_over_ranks([sum(q_s[i].elapsed_time(q_e[i]) for i in range(K_steps)) / K_steps],
                                  world, dev)[0] * 1e3

    bits, site = qg.qgemm_get_device_status()

    if rank == 0:
        peaks, peak_src = measured_peaks()
        wbytes = w_host.shape[0] * (K // 256) * wl.block_bytes   # every expert's rows (routed)
        small = (c1["q4k_small"] + c1["q6k_small"]) > (c0["q4k_small"] + c0["q6k_small"])
        if small:
            # the streaming kernel is bound by the weight bytes it reads once
            achieved = wbytes / (gemm_mean_ms * 1e-3) / 1e9
            roof = {"kernel": "smallm_kernel (small-M streaming)", "bound": "hbm", "achieved": achieved,
                    "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                    "frac": achieved / float(peaks["hbm_gbs"]),
                    "peak_source": f"{peak_src} hbm_gbs", "traffic": NCU_TRAFFIC_BYTES.get(wl.name)}
        else:
            peak = float(peaks["bf16_tflops"])
            achieved = ops / (gemm_mean_ms * 1e-3) / 1e12
            roof = {"kernel": "gemm_tc_kernel (tile GEMM)", "bound": "tensor", "achieved": achieved,
                    "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                    "peak_source": f"{peak_src} bf16_tflops (burst; fp16 has the bf16 rate)",
                    "int8_peak": None,
                    "int8_note": "no int8 tensor-core MMA on sm_103a (ptxas rejects tcgen05 kind::i8 there): "
                                 "the integer products run exactly as fp16 MMAs, so the fp16/bf16 dense peak "
                                 "is this kernel's ceiling",
                    "traffic": NCU_TRAFFIC_BYTES.get(wl.name)}
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K_steps,
            "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic", "config": config_of(wl),
            "weight_gbs": wbytes / (gemm_mean_ms * 1e-3) / 1e9,
            "kernels_us": {"step": mean_ms * 1e3, "step_eager_calls": eager_mean_ms * 1e3,
                           "gemm": gemm_mean_ms * 1e3, "quantize_prep_and_gaps": (mean_ms - gemm_mean_ms) * 1e3},
            "launch": "one CUDA graph per step (captured from the API calls)" if graph is not None
                      else "eager API calls",
            "roofline": roof,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d_bytes,
                    "d2h_bytes_per_step": d2h_bytes, "ms_per_step": e2e_ms,
                    "path": "zero-copy: X read and Y written in pinned host memory by the library's kernels",
                    "copies": {"value": e2e_copies_value, "ms_per_step": e2e_copies_ms,
                               "path": "cudaMemcpyAsync of X and Y around the device step"}},
            "quantize": quantize_report(M, K, quant_us, tile_next, measured_peaks()[0]["hbm_gbs"]),
            "gpu_launches": int(launches),
            "clocks": sampler.summary(t0, t1),
            "device_status": bits,
        }
        if not args.no_cpu_baseline and world == 1:
            # the oracle over all host cores, `cpu_rows` token rows per core, repeated
            # until about `cpu_seconds` of wall time; then on one core the same way
            cores = host_cores()
            pool = OraclePool(wl, x_host, cores)
            rows = min(args.cpu_rows * cores, M)
            runs, total, cops = 0, 0.0, 0.0
            while total < args.cpu_seconds and runs < 1000:
                dt, cops = pool.run(rows)
                total += dt
                runs += 1
            pool.close()
            line["cpu_baseline"] = {"value": runs * cops / total / 1e12, "unit": UNIT, "cores": cores,
                                    "kind": "oracle",
                                    "sample": f"{rows} of {M} token rows split over {cores} oracle processes "
                                              f"(quantize + GEMM over all N{', both slots' if is_routed else ''}) "
                                              f"x {runs} runs, {total:.1f} s wall"}
            rows = min(args.cpu_rows, M)
            runs, total, cops = 0, 0.0, 0.0
            while total < args.cpu_seconds and runs < 1000:
                dt, cops = oracle_sample(wl, rows, x_host, w_host)
                total += dt
                runs += 1
            line["cpu_baseline_single_core"] = {
                "value": runs * cops / total / 1e12, "unit": UNIT, "cores": 1, "kind": "oracle",
                "sample": f"{rows} of {M} token rows (quantize + GEMM over all N"
                          f"{', both slots' if is_routed else ''}) x {runs} runs, {total:.1f} s"}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
