#!/usr/bin/env python
"""Benchmark of the routed Q4_0 x Q8_1 MoE expert matmul (quantize + route +
matmul per step) on GB300; prints one JSON line.

Default workload: the prefill batch shaped like the kernel benchmark of
FreeToken PR #185 ("Performance": nrows 1408, hidden 2816, top_k 8, 8191
tokens), with 128 experts, uniform routing, seed 1; synthetic inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME:TOKENS]

ours       value = routed tokens/s over all ranks with inputs resident in HBM
           (L2 flushed between steps); e2e = the same through the Python API
           with pinned host buffers and every step's host<->device copies in
           the timed region (copies in, compute and copies out pipelined on
           three streams; the serial figure beside it); roofline of the
           dominant kernel from CUDA events the library
           records on its launch stream; cpu_baseline = the CPU oracle on a
           bounded sample (rank 0 only).
reference  the CPU oracle (the only reference this project has) on a bounded
           sample of the same workload per step, rank 0 only.
Multi-GPU: one process per GPU, each an independent replica on its own batch
(weak scaling, no collective on the data path).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "routed tokens/s"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Tesla T4, moe_vec q4_0 x q8_1 after the grid.x fix, 8191 tokens: 705.8 ms
# (FreeToken PR #185, "Performance"); context only, other hardware.
PAGES_T4_TOKENS_PER_S = {("prefill", 8191): 8191 / 0.7058, ("prefill", 4096): 4096 / 0.3461,
                         ("prefill", 2048): 2048 / 0.1740}
# DRAM bytes (read + write) per launch of the dominant kernel from one ncu
# capture (profiles/moe_gemm_tc_prefill.md), keyed by a hash of the sources that
# kernel is built from (its own files and the tile constants it takes from the
# internal header), so a changed kernel reports null instead.
GEMM_SOURCES = ("bit_quantized_moe_quantize_gb300/csrc/moe_gemm_tc.cu", "bit_quantized_moe_quantize_gb300/csrc/gemm_common.cuh",
                "bit_quantized_moe_quantize_gb300/csrc/ft_common.cuh")
GEMM_CONSTANTS = ("bit_quantized_moe_quantize_gb300/csrc/ft_internal.h", "kGemm")
NCU_TRAFFIC = {("moe_gemm_tc_kernel", "9356abed6442eb8b", "prefill:8191"): 667560704 + 341054720}
# the same for the mma.sync GEMV kernel (profiles/moe_gemv_mma_decode.md)
MMA_SOURCES = ("bit_quantized_moe_quantize_gb300/csrc/moe_gemv_mma.cu", "bit_quantized_moe_quantize_gb300/csrc/gemv_rows.cuh",
               "bit_quantized_moe_quantize_gb300/csrc/gemv_blocks.cuh", "bit_quantized_moe_quantize_gb300/csrc/ft_common.cuh")
NCU_TRAFFIC_GEMV = {("moe_gemv_mma_kernel", "84c18d9629a18982", "mixtral_8x7b:32", "q4_0"): 264453120 + 4717568}


def mma_tiles(S, E, K, wtype="q4_0") -> bool:
    """The library's rule for the mma.sync GEMV tiles of a Q4_0, Q4_1, Q8_0 or
    Q4_K batch (rows of whole 256-weight runs): more than 4 slots per expert
    on average, and the staged activations of an 8-slot tile (352 B per block,
    384 for the types with an offset term) plus a ring of two 16-row boxes
    within 227 KB of shared memory."""
    pitch = {"q4_0": 144, "q4_k": 144, "q4_1": 176, "q8_0": 272}.get(wtype)
    if pitch is None:
        return False
    nb = K // 32
    head = 8 * 2 * 16 + 16
    ring0 = (head + nb * (384 if wtype in ("q4_k", "q4_1") else 352) + 127) // 128 * 128
    return S / E > 4.0 and ring0 + 2 * pitch * 16 <= 227 * 1024


def kernel_source_hash(files, constants=GEMM_CONSTANTS) -> str:
    """Hash of the code of a kernel's source files (comments and blank space
    left out, so that a comment edit keeps a capture valid) and, optionally,
    of the lines of a header that hold its constants."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f)) as fh:
            code = re.sub(r"/\*.*?\*/", " ", fh.read(), flags=re.S)
            code = re.sub(r"//[^\n]*", " ", code)
            h.update(os.path.basename(f).encode())
            h.update(" ".join(code.split()).encode())
    if constants:
        path, key = constants
        with open(os.path.join(ROOT, path)) as fh:
            h.update("".join(line for line in fh if key in line).encode())
    return h.hexdigest()[:16]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="prefill:8191")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--per-slot", action="store_true",
                    help="one activation row per routed slot (ft_moe_q4_0_q8_1_slots, the second expert layer)")
    ap.add_argument("--two-calls", action="store_true",
                    help="time ft_quantize_q8_1 + ft_moe_q4_0_q8_1 instead of the single entry point ft_moe_q4_0_fp16")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager launches instead of a CUDA-graph replay of the step")
    ap.add_argument("--wtype", default="q4_0",
                    choices=["q4_0", "q4_1", "q5_0", "q5_1", "q8_0", "q4_k", "q5_k", "q6_k", "q2_k", "q3_k"],
                    help="GGUF type of the expert weights (other than q4_0: ft_moe_gguf_q8_1; GEMV path, tensor cores too for q4_k)")
    ap.add_argument("--path", choices=["auto", "gemv", "gemm", "gemv_dp4a"], default="auto",
                    help="force the library's path (ft_moe_set_path); gemv_dp4a: the GEMV path without the "
                         "mma.sync 8-slot tiles")
    ap.add_argument("--ffn", choices=["silu", "gelu_tanh"], default=None,
                    help="time both expert layers (ft_moe_ffn_q4_0_q8_1) with the workload's ncols as the hidden "
                         "size and its nrows as the intermediate size")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload(spec):
    from bit_quantized_moe_quantize_gb300 import synth
    name, _, t = spec.partition(":")
    wl = synth.WORKLOADS[name]
    T = int(t) if t else max(wl.tokens)
    return name, wl, T


def replica_workload(wl, rank):
    """Rank r's replica: the same expert weights, its own batch of tokens."""
    from bit_quantized_moe_quantize_gb300 import synth
    return synth.Workload(**{**wl.__dict__, "seed": wl.seed + 7919 * rank}) if rank else wl


def make_inputs(wl, T, rank, with_weights=True):
    from bit_quantized_moe_quantize_gb300 import synth
    w = synth.make_weights(wl) if with_weights else None
    wl_r = replica_workload(wl, rank)
    x = synth.make_activations(wl_r, T)
    ids = synth.make_topk_ids(wl_r, T)
    return w, x, ids


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank scalar over the process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job routed tokens/s: every rank's tokens over the slowest rank's step time."""
    return tokens_per_rank * world / (ms_max / 1000.0)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "begin":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.samples:
            if self.t0 is not None and not (self.t0 - 0.1 <= ts <= (self.t1 or ts) + 0.1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({self.NAMES[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------- CPU oracle
def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_tokens_per_s(wl, w, x, ids, budget_s, max_tokens=None, threads=1):
    """Time the CPU oracle (quantize + route + matmul) on the first n tokens, n
    sized so the run takes about budget_s; returns (tokens/s, n, seconds).
    With threads > 1 the n tokens are cut into that many contiguous slices and
    each thread runs the oracle's quantizer and matmul on its own slice (the
    oracle's C calls release the interpreter lock); the routing of all n
    tokens runs once.  The oracle itself is unchanged."""
    import oracle as oracle_pkg
    from concurrent.futures import ThreadPoolExecutor
    o = oracle_pkg.get()

    def part(lo, hi):
        act = o.quantize_q8_1(x[lo:hi])
        o.moe(w, act, ids[lo:hi])

    def run(n, pool):
        t0 = time.perf_counter()
        o.route(ids[:n], wl.n_experts)
        if pool is None:
            part(0, n)
        else:
            cuts = np.linspace(0, n, threads + 1).astype(int)
            list(pool.map(lambda i: part(cuts[i], cuts[i + 1]), [i for i in range(threads) if cuts[i] < cuts[i + 1]]))
        return time.perf_counter() - t0

    with ThreadPoolExecutor(max_workers=threads) if threads > 1 else _null_ctx() as pool:
        t1 = run(1, None)
        n = int(max(1, min(max_tokens or x.shape[0], threads * budget_s / max(t1, 1e-6))))
        dt = run(n, pool)
    return n / dt, n, dt


class _null_ctx:
    def __enter__(self):
        return None

    def __exit__(self, *a):
        return False


def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    name, wl, T = workload(args.workload)
    w, x, ids = make_inputs(wl, T, 0)
    import oracle as oracle_pkg
    o = oracle_pkg.get()
    total_budget = 150.0
    per_step = total_budget / max(1, args.steps + args.warmup)
    t0 = time.perf_counter()
    act = o.quantize_q8_1(x[:1])
    o.moe(w, act, ids[:1])
    t_tok = time.perf_counter() - t0
    n = int(max(1, min(T, per_step / max(t_tok, 1e-6))))
    times = []
    for i in range(args.warmup + args.steps):
        s0 = (i * n) % max(1, T - n + 1)
        t0 = time.perf_counter()
        act = o.quantize_q8_1(x[s0:s0 + n])
        o.route(ids[s0:s0 + n], wl.n_experts)
        o.moe(w, act, ids[s0:s0 + n])
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1000 * statistics.mean(times)
    value = n / (ms / 1000)
    sample = f"{n} of {T} tokens per step (quantize + route + matmul in the oracle, single thread)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(name, wl, T, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_of(name, wl, T, world):
    return {"workload": f"{name} E={wl.n_experts} k={wl.top_k} K={wl.ncols} N={wl.nrows} T={T}",
            "n_experts": wl.n_experts, "top_k": wl.top_k, "ncols": wl.ncols, "nrows": wl.nrows, "tokens": T,
            "routing": wl.routing, "seed": wl.seed, "replicas": world,
            "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write)"}


# ------------------------------------------------------------------ ours
def ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    import bit_quantized_moe_quantize_gb300 as ft
    from bit_quantized_moe_quantize_gb300 import build
    build.build()
    ft.load()

    name, wl, T = workload(args.workload)
    w, x, ids = make_inputs(wl, T, rank)
    E, k, K, N = wl.n_experts, wl.top_k, wl.ncols, wl.nrows
    wtype = args.wtype
    if wtype != "q4_0":
        if args.per_slot or args.impl == "reference":
            raise SystemExit("--wtype takes the per-token matmul of our arm only")
        from bit_quantized_moe_quantize_gb300 import synth
        w = synth.make_weights_gguf(wl, wtype)
    S = T * k
    if args.per_slot:                       # one fp16 activation row per slot
        from bit_quantized_moe_quantize_gb300 import synth
        x = synth.make_activations(replica_workload(wl, rank), S)
    rows = S if args.per_slot else T
    # the path the library takes for this shape and weight type
    path_setting = args.path
    ft.set_path(path_setting)
    path = {1: "gemv", 2: "gemm"}[ft.selected_path(T, k, E, N, K, wtype)]

    dw = torch.from_numpy(w).to(dev)
    dx = torch.from_numpy(x).to(dev)
    di = torch.from_numpy(ids).to(dev)
    act = torch.empty((rows, K // 32, 36), dtype=torch.uint8, device=dev)
    out = torch.empty((T, k, N), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    ft.reserve(T, k, E, N, K)
    stream = torch.cuda.current_stream()

    matmul = ft.moe_q4_0_q8_1_slots if args.per_slot else ft.moe_q4_0_q8_1
    if wtype != "q4_0":
        def matmul(dw_, act_, di_, out=None):
            return ft.moe_gguf_q8_1(wtype, dw_, act_, di_, out=out)

    # the hot path from fp16 activations: one call (one launch for a decode
    # batch), or the quantizer and the matmul called one after the other
    one_call = not args.two_calls and not args.per_slot and wtype == "q4_0"

    def step():
        if one_call:
            ft.moe_q4_0_fp16(dw, dx, di, out=out)
            return
        ft.quantize_q8_1(dx, out=act)
        matmul(dw, act, di, out=out)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if ft.read_device_error():
        raise RuntimeError("device error flag raised during warm-up")

    # the timed step: one CUDA-graph replay of quantize + route + matmul (the
    # library's launches are fixed per shape and allocate nothing once the
    # workspace is reserved), so small batches are not timed as host launch gaps
    run, launch_mode = step, "eager"
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                step()
        stream.wait_stream(side)
        run, launch_mode = graph.replay, "cuda graph"
        for _ in range(3):
            flush.zero_()
            run()
        torch.cuda.synchronize()

    gpu_index = torch.cuda.current_device()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            gpu_index = int(vis.split(",")[gpu_index])
        except ValueError:
            pass
    clocks = ClockSampler(gpu_index)
    clocks.start()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.mark("begin")
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        run()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    clocks.mark("end")
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = max_over_ranks(statistics.mean(step_ms), dev)
    value = job_throughput(T, world, ms)

    # kernel times for the roofline: the same step, eager, with the library's
    # own CUDA events around each kernel on its launch stream
    n_prof = max(3, min(args.steps, 50))
    ft.profile_enable(n_prof)
    for _ in range(n_prof):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    prof = ft.profile_read()
    ft.profile_enable(0)
    launches_per_step = prof["launches"] / max(1, prof["calls"])

    # e2e through the public API: pinned host input -> device -> result -> pinned host
    e2e = None
    if not args.no_e2e:
        hx = torch.from_numpy(x).pin_memory()
        hi = torch.from_numpy(ids).pin_memory()
        ho = torch.empty((T, k, N), dtype=torch.float32).pin_memory()
        n_e2e = max(3, min(args.steps, 50))
        e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_e2e)]
        for i in range(args.warmup + n_e2e):
            flush.zero_()
            j = i - args.warmup
            if j >= 0:
                e_ev[j][0].record(stream)
            dx.copy_(hx, non_blocking=True)
            di.copy_(hi, non_blocking=True)
            step()
            ho.copy_(out, non_blocking=True)
            if j >= 0:
                e_ev[j][1].record(stream)
        torch.cuda.synchronize()
        serial_ms = statistics.mean(a.elapsed_time(b) for a, b in e_ev)
        assert np.array_equal(ho.numpy(), out.cpu().numpy())
        # the same steps pipelined the way a serving loop runs them: inputs of step
        # i+1 copied in on one stream while step i computes on another and the
        # result of step i-1 is copied out on a third; device inputs and outputs
        # double-buffered; every step's copies inside the timed region (first
        # copy in to last copy out), each step's L2 flush on the compute stream
        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        dxs, dis = [dx, torch.empty_like(dx)], [di, torch.empty_like(di)]
        outs, hos = [out, torch.empty_like(out)], [ho, torch.empty_like(ho).pin_memory()]
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        ev_cmp = [torch.cuda.Event(), torch.cuda.Event()]
        ev_out = [torch.cuda.Event(), torch.cuda.Event()]
        for e_ in ev_cmp + ev_out:
            e_.record(stream)
        t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        n_run = args.warmup + n_e2e
        for i in range(n_run):
            b = i % 2
            if i == args.warmup:
                t_begin.record(s_in)
            s_in.wait_event(ev_cmp[b])                  # step i-2 done reading this input buffer
            with torch.cuda.stream(s_in):
                dxs[b].copy_(hx, non_blocking=True)
                dis[b].copy_(hi, non_blocking=True)
                ev_in[b].record(s_in)
            s_cmp.wait_event(ev_in[b])
            s_cmp.wait_event(ev_out[b])                 # step i-2's result copied out of this buffer
            with torch.cuda.stream(s_cmp):
                flush.zero_()
                if one_call:
                    ft.moe_q4_0_fp16(dw, dxs[b], dis[b], out=outs[b])
                else:
                    ft.quantize_q8_1(dxs[b], out=act)
                    matmul(dw, act, dis[b], out=outs[b])
                ev_cmp[b].record(s_cmp)
            s_out.wait_event(ev_cmp[b])
            with torch.cuda.stream(s_out):
                hos[b].copy_(outs[b], non_blocking=True)
                ev_out[b].record(s_out)
        t_end.record(s_out)
        torch.cuda.synchronize()
        pipe_ms = max_over_ranks(t_begin.elapsed_time(t_end) / n_e2e, dev)
        serial_ms = max_over_ranks(serial_ms, dev)
        assert np.array_equal(hos[(n_run - 1) % 2].numpy(), outs[(n_run - 1) % 2].cpu().numpy())
        # the better of the two ways to run it: pipelining pays when the copies
        # are long (prefill); for a few-µs decode step the host's issue of the
        # three streams' work costs more than it hides
        e_ms = min(pipe_ms, serial_ms)
        e2e = {"value": job_throughput(T, world, e_ms), "unit": UNIT, "ms_per_step": e_ms,
               "h2d_bytes_per_step": int(x.nbytes + ids.nbytes), "d2h_bytes_per_step": int(S * N * 4),
               "mode": "pipelined" if pipe_ms <= serial_ms else "serial",
               "pipelined_ms_per_step": pipe_ms, "serial_ms_per_step": serial_ms,
               "note": "serial: copy in, step, copy out on one stream per step; pipelined: copies in, compute and "
                       "copies out on three streams, double-buffered; both with every step's copies timed"}
    if ft.read_device_error():
        raise RuntimeError("device error flag raised during the timed region")
    clk = clocks.stop()

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    calls = max(1, prof["calls"])
    mm_ms = prof["matmul_ms"] / calls
    flops = 2.0 * S * N * K
    counts = np.bincount(ids.reshape(-1), minlength=E)
    nb = K // 32
    _, wbytes, wper = ft.WEIGHT_TYPES[wtype]
    alg_bytes = int((counts > 0).sum()) * N * (K // wper) * wbytes + rows * nb * 36 + S * N * 4
    fused = one_call and path == "gemv" and launches_per_step == 1
    if fused:   # one launch reads the fp16 rows instead of Q8_1 blocks
        alg_bytes += rows * K * 2 - rows * nb * 36
    if path == "gemm":
        kern = "moe_gemm_tc_kernel" if wtype == "q4_0" else f"moe_gemm_tc_kernel<{wtype}>"
        achieved = flops / (mm_ms / 1000.0) / 1e12
        roof = {"kernel": kern, "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "peak_note": f"fp16 kind::f16 MMA at the bf16 rate (nominal ratio 1.0), burst, of {peak_src}",
                "algorithmic": f"2*S*N*K = {flops:.4g} FLOP per launch", "kernel_ms": mm_ms}
    else:
        # the library's GEMV plan: one weight row per lane when rows are whole
        # 256-weight runs (all types but Q6_K, Q2_K, Q3_K), else one block per lane
        rows_ok = K % 256 == 0 and wtype not in ("q6_k", "q2_k", "q3_k")
        kern = ("moe_gemv_rows_kernel<fused>" if fused else "moe_gemv_rows_kernel") if rows_ok else "moe_gemv_kernel"
        if rows_ok and not fused and path_setting != "gemv_dp4a" and mma_tiles(S, E, K, wtype):
            kern = "moe_gemv_mma_kernel"
        achieved = alg_bytes / (mm_ms / 1000.0) / 1e9
        roof = {"kernel": kern, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_note": f"copy bandwidth, of {peak_src}",
                "algorithmic": f"unique expert weights + {'fp16 x' if fused else 'Q8_1 act'} + fp32 out = "
                               f"{alg_bytes} B per launch",
                "kernel_ms": mm_ms}
    if path == "gemm":
        tr = NCU_TRAFFIC.get((kern, kernel_source_hash(GEMM_SOURCES), args.workload))
    elif kern == "moe_gemv_mma_kernel":
        tr = NCU_TRAFFIC_GEMV.get((kern, kernel_source_hash(MMA_SOURCES, None), args.workload, wtype))
    else:
        tr = None
    roof["traffic"] = tr
    if path == "gemv":
        # the same number of bytes streamed by a plain read kernel (L2 flushed
        # before each): what the memory system delivers at this size at all
        nread = min(alg_bytes, dw.numel()) // 16 * 16
        rl = []
        for _ in range(n_prof):
            flush.zero_()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            ft.debug_stream_read(dw, nread)
            a1.record(stream)
            rl.append((a0, a1))
        torch.cuda.synchronize()
        read_ms = statistics.mean(x.elapsed_time(y) for x, y in rl)
        read_gbs = nread / (read_ms / 1000.0) / 1e9
        roof["same_size_read"] = {"bytes": nread, "ms": read_ms, "gbs": read_gbs,
                                  "frac": roof["achieved"] / read_gbs,
                                  "note": "ft_debug_stream_read of the same bytes: plain 16-byte loads, L2 flushed"}

    cpu = None
    if not args.no_cpu_baseline and world == 1 and wtype == "q4_0":
        cores = host_cores()
        tps, n, dt = oracle_tokens_per_s(wl, w, x, ids, budget_s=10.0, threads=cores)
        tps1, n1, dt1 = oracle_tokens_per_s(wl, w, x, ids, budget_s=6.0)
        cpu = {"value": tps, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"first {n} of {T} tokens: quantize + route + matmul, {dt:.1f} s on {cores} threads "
                         f"(contiguous token slices, one per thread; host has {os.cpu_count()} cores)",
               "single_thread": {"value": tps1, "unit": UNIT, "cores": 1,
                                 "sample": f"first {n1} of {T} tokens, {dt1:.1f} s"}}

    base = PAGES_T4_TOKENS_PER_S.get((name, T))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (value / base) if base else None,
        "vs_baseline_note": "pages' Tesla T4 moe_vec time for this token count (context, other hardware)"
        if base else None,
        "dtype": f"{wtype} x q8_1: exact int block dots (f16 MMA / dp4a), f32 scaling",
        "data": "synthetic", "config": {**config_of(name, wl, T, world), "path": path, "path_setting": path_setting,
                                        "launch": launch_mode,
                                        "activations": "per slot" if args.per_slot else "per token",
                                        "entry": "ft_moe_q4_0_fp16" if one_call else "ft_quantize_q8_1 + matmul",
                                        "weights": wtype},
        "effective_tops": 2.0 * S * N * K * world / (ms / 1000.0) / 1e12,
        "kernels_ms_per_step": {"quantize": prof["quantize_ms"] / calls, "prepare": prof["route_ms"] / calls,
                                "matmul": mm_ms,
                                "note": "eager pass; prepare = routing (+ activation gather on the tensor-core path)"},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": int(round(launches_per_step * args.steps)), "launches_per_step": launches_per_step,
        "clocks": clk, "wall_s_timed": wall,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


# ------------------------------------------------------------ both layers
def ffn(args):
    """quantize + layer 1 (gate and up rows) with the activation/requantize
    fused into it + layer 2 per step, CUDA-graph replayed; per-stage times
    from an eager pass of the same calls, with the unfused layer 1 and
    activation step beside them; roofline of the fused layer 1 (tensor pipe
    on the tensor-core path, HBM on the GEMV path)."""
    import torch
    rank, world, _ = dist_env()
    if world > 1:
        raise SystemExit("--ffn runs on one GPU")
    dev = torch.device("cuda", torch.cuda.current_device())
    import bit_quantized_moe_quantize_gb300 as ft
    from bit_quantized_moe_quantize_gb300 import build, synth
    build.build()
    ft.load()
    name, wl, T = workload(args.workload)
    E, k, H, I = wl.n_experts, wl.top_k, wl.ncols, wl.nrows
    S = T * k
    kind = {"silu": ft.ACT_SILU, "gelu_tanh": ft.ACT_GELU_TANH}[args.ffn]
    w13 = synth.make_weights(synth.custom_workload(E, k, H, 2 * I, wl.seed))
    w2 = synth.make_weights(synth.custom_workload(E, k, I, H, wl.seed + 1000))
    x = synth.make_activations(wl, T)
    ids = synth.make_topk_ids(wl, T)
    d13, d2 = torch.from_numpy(w13).to(dev), torch.from_numpy(w2).to(dev)
    dx, di = torch.from_numpy(x).to(dev), torch.from_numpy(ids).to(dev)
    act = torch.empty((T, H // 32, 36), dtype=torch.uint8, device=dev)
    h = torch.empty((T, k, 2 * I), dtype=torch.float32, device=dev)
    mid = torch.empty((S, I // 32, 36), dtype=torch.uint8, device=dev)
    out = torch.empty((T, k, H), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    ft.ffn_reserve(T, k, E, H, I)
    stream = torch.cuda.current_stream()

    def step():
        ft.quantize_q8_1(dx, out=act)
        ft.moe_ffn_q4_0_q8_1(d13, d2, act, di, kind, out=out, act_mid=mid, keep_h=False)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    run, launch_mode = step, "eager"
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                step()
        stream.wait_stream(side)
        run, launch_mode = graph.replay, "cuda graph"
        for _ in range(3):
            flush.zero_()
            run()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    clocks.mark("begin")
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        run()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clocks.mark("end")
    clk = clocks.stop()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)

    # per stage, eager, events on the launching stream (torch's current stream)
    stages = {"quantize": lambda: ft.quantize_q8_1(dx, out=act),
              "layer1_act_fused": lambda: ft.moe_q4_0_q8_1_act(d13, act, di, kind, out=mid),
              "layer2": lambda: ft.moe_q4_0_q8_1_slots(d2, mid, di, out=out),
              "unfused_layer1": lambda: ft.moe_q4_0_q8_1(d13, act, di, out=h),
              "unfused_act_requant": lambda: ft.act_mul_quantize_q8_1(h, kind, out=mid)}
    n_prof = max(3, min(args.steps, 30))
    st_ms = {}
    for key, fn in stages.items():
        tl = []
        for _ in range(n_prof):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            tl.append((a, b))
        torch.cuda.synchronize()
        st_ms[key] = statistics.mean(a.elapsed_time(b) for a, b in tl)
    if ft.read_device_error():
        raise RuntimeError("device error flag raised")
    peaks, peak_src = load_peaks()
    flops = 2.0 * S * (2 * I) * H + 2.0 * S * H * I
    l1_flops = 2.0 * S * (2 * I) * H
    tc = ft.selected_path(T, k, E, 2 * I, H) == ft.FT_PATH_GEMM
    if tc:
        achieved = l1_flops / (st_ms["layer1_act_fused"] / 1000.0) / 1e12
        roof = {"kernel": "moe_gemm_tc_kernel<act>", "bound": "tensor", "achieved": achieved,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "algorithmic": f"2*S*2I*H = {l1_flops:.4g} FLOP per call (route and gather included in the time)",
                "peak_note": f"dense bf16 tensor peak, of {peak_src}", "traffic": None}
    else:
        l1_bytes = E * 2 * I * (H // 32) * 18 + T * (H // 32) * 36 + S * (I // 32) * 36
        achieved = l1_bytes / (st_ms["layer1_act_fused"] / 1000.0) / 1e9
        gemv_k = "moe_gemv_mma_kernel" if H % 256 == 0 and mma_tiles(S, E, H) else "moe_gemv_rows_kernel"
        roof = {"kernel": f"{gemv_k} + act_mul_quantize_q8_1_kernel", "bound": "hbm",
                "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"],
                "algorithmic": f"all expert weights + act + act_mid = {l1_bytes} B per call",
                "peak_note": f"copy bandwidth, of {peak_src}", "traffic": None}
    line = {"metric": "routed tokens/s through both expert layers", "value": T / (ms / 1000.0), "unit": UNIT,
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "dtype": "q4_0 x q8_1 exact int block dots, f32 scaling and activation", "data": "synthetic",
            "config": {"workload": f"{name} E={E} k={k} hidden={H} inter={I} T={T} act={args.ffn}",
                       "launch": launch_mode, "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write)"},
            "effective_tops": flops / (ms / 1000.0) / 1e12,
            "stages_ms": st_ms,
            "roofline": roof,
            "clocks": clk}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return reference_arm(args)
    if args.ffn:
        return ffn(args)
    return ours(args)


if __name__ == "__main__":
    sys.exit(main())
