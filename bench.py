#!/usr/bin/env python
"""Benchmark of the integer-quantised matmul hot path on GB300.

Headline workload: the A8W8 GEMM at M = K = N = 4096 (int8 x int8, exact int32
accumulation, act_scale[M] / weight_scale[N] epilogue, bf16 output), reported
as TOPS (2*M*N*K integer operations per second). One step = one call of
qmm_a8w8 on inputs resident in HBM; a 256 MiB write flushes L2 before every
timed iteration (the inputs, 32 MiB, would otherwise sit in the 126 MiB L2).

The same JSON line also carries the other benchmark workloads of the path,
each timed with CUDA events on the launching stream: the decode GEMV (int8
weight 8192x28672, M in {1,4,16}) in GB/s of algorithmic bytes and as a
fraction of measured HBM bandwidth; DynamicQuantizeLinear on 8192x4096 fp32;
MatMulInteger 8192x4096x11008 (u8 x s8, zero points); batched MatMulInteger
65536x1024x1024 with a shared B; and the small fp32 x int8 matmul.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl qmm|reference]
With N > 1 (torchrun) every rank runs an independent replica (the path has no
exchange step); value = all ranks' operations / the slowest rank's time.
--impl reference times the CPU oracle (test infrastructure) on rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import qmm_workloads as W  # noqa: E402

METRIC = "A8W8 int8 GEMM TOPS at 4096^3 (% int8 peak); int8-weight GEMV GB/s (% HBM)"
WORKLOAD = "a8w8_4096x4096x4096_bf16"
M = K = N = 4096
OPS = 2.0 * M * N * K
FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_traffic(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    source is unchanged since the counters were taken; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)[kernel_key]
        src = os.path.join(ROOT, d["source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()
        if h != d["source_sha256"]:
            return None
        return float(d["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError, TypeError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed regions run."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = None
        self.windows = []

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="qmm_clocks_", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.uuid:
            cmd[1:1] = ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "", 1).isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        power = [float(r[3]) for r in rows if r[3].replace(".", "", 1).isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


SPIN_CYCLES = 400000   # ~200 us of GPU spin: the host enqueues the timed call while it runs


def time_gpu(fn, steps, warmup, flush=None):
    """Per-iteration device time (ms) of fn, CUDA events on the current stream.

    Before each timed call the stream runs the optional L2 flush and a short
    spin kernel, so the host has enqueued the call (and its end event) before
    the start event fires: host-side marshalling never shows up as device time."""
    import torch
    for _ in range(warmup):
        if flush is not None:
            flush()
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush()
        torch.cuda._sleep(SPIN_CYCLES)
        ev[i][0].record()
        fn()
        ev[i][1].record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def time_gpu_split(first, second, steps, warmup, flush=None):
    """Like time_gpu for a step made of two calls on the current stream: returns
    per-step device times (ms) of the whole step and of the second call alone
    (CUDA events before, between and after the two calls)."""
    import torch
    for _ in range(warmup):
        if flush is not None:
            flush()
        first()
        second()
    torch.cuda.synchronize()
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush()
        torch.cuda._sleep(SPIN_CYCLES)
        ev[i][0].record()
        first()
        ev[i][1].record()
        second()
        ev[i][2].record()
    torch.cuda.synchronize()
    return [a.elapsed_time(c) for a, b, c in ev], [b.elapsed_time(c) for a, b, c in ev]


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


_ORACLE_W = None


def _oracle_worker_init():
    """Process-pool worker: one copy of the 4096^3 A8W8 workload per process."""
    global _ORACLE_W
    _ORACLE_W = W.a8w8_4096()


def _oracle_rows(task):
    """The oracle as it stands on rows [r0, r1) x all columns; returns the seconds taken."""
    from oracle import qmm_oracle as O
    r0, r1 = task
    w = _ORACLE_W
    t0 = time.perf_counter()
    O.a8w8(w.A[r0:r1], w.B, w.act_scale[r0:r1], w.weight_scale, "bf16")
    return time.perf_counter() - t0


def oracle_pool(cores):
    """A spawn pool (never forked from a process that holds a CUDA context), one
    single-threaded oracle process per host core, each with the workload loaded."""
    import multiprocessing as mp
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    pool = mp.get_context("spawn").Pool(cores, initializer=_oracle_worker_init)
    pool.map(_oracle_rows, [(0, 1)] * cores)   # every worker loaded and warm
    return pool


def cpu_baseline_a8w8(budget_s=12.0, rows_per_task=4):
    """The oracle as it stands, on all host cores, over a bounded sample of the
    rows of the 4096^3 workload (row blocks handed out until the budget is spent)."""
    cores = host_cores()
    pool = oracle_pool(cores)
    try:
        tasks = [(r, r + rows_per_task) for r in range(0, M, rows_per_task)]
        rows, t_end = 0, 0.0
        t0 = time.perf_counter()
        for _ in pool.imap_unordered(_oracle_rows, tasks):
            rows += rows_per_task
            t_end = time.perf_counter() - t0
            if t_end > budget_s:
                break
    finally:
        pool.terminate()
        pool.join()
    ops = 2.0 * rows * K * N
    return {"value": ops / t_end / 1e12, "unit": "TOPS", "cores": cores, "kind": "oracle",
            "sample": f"{rows} of 4096 rows of the 4096^3 A8W8 workload in blocks of {rows_per_task} rows, one "
                      f"single-threaded oracle process per host core (numpy int64 matmul + float32 epilogue), "
                      f"{t_end:.1f} s wall"}


def run_reference(args, rank):
    """The oracle on the host cores, each step one output row (all 4096 columns)
    per core of the 4096^3 A8W8 workload."""
    if rank != 0:
        return
    cores = host_cores()
    pool = oracle_pool(cores)
    times = []
    try:
        for i in range(args.warmup + args.steps):
            r0 = (i * cores) % M
            tasks = [((r0 + c) % M, (r0 + c) % M + 1) for c in range(cores)]
            t0 = time.perf_counter()
            pool.map(_oracle_rows, tasks)
            dt = time.perf_counter() - t0
            if i >= args.warmup:
                times.append(dt)
    finally:
        pool.terminate()
        pool.join()
    per_step_ops = 2.0 * K * N * cores
    mean = statistics.mean(times)
    value = per_step_ops / mean / 1e12
    sample = f"{cores} output rows x 4096 columns of the 4096^3 A8W8 workload per step, one row per host core"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int64 (oracle)", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N, "step": sample},
            "cpu_baseline": {"value": value, "unit": "TOPS", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def int8_mma_peak(q, torch, launches=6, iters=4096):
    """Rate of the legacy int8 tensor path (mma.sync m16n8k32 s8) measured with
    CUDA events: the median of `launches` timed launches after one warm-up."""
    q.int8_mma_peak_launch(64)
    torch.cuda.synchronize()
    rates = []
    for _ in range(launches):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        ops = q.int8_mma_peak_launch(iters)
        b.record()
        b.synchronize()
        rates.append(ops / (a.elapsed_time(b) * 1e-3) / 1e12)
    return statistics.median(rates)


def cublas_int8_tops(torch, A, B, steps=20):
    """cuBLAS int8 GEMM (torch._int_mm, int32 out) on the same operands, for context."""
    try:
        torch._int_mm(A, B)
        torch.cuda.synchronize()
        ts = time_gpu(lambda: torch._int_mm(A, B), steps, 3)
        return OPS / (statistics.median(ts) * 1e-3) / 1e12
    except (RuntimeError, AttributeError):
        return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="qmm", choices=["qmm", "reference"])
    ap.add_argument("--no-secondary", action="store_true", help="time only the headline workload")
    ap.add_argument("--case", default=None, help="time one named workload alone and exit")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.case:
        run_case(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    def barrier():
        if dist is not None:
            dist.barrier()

    def max_over_ranks(v):
        if dist is None:
            return v
        t = torch.tensor([v], dtype=torch.float64, device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    import quantized_int8_matmul_gb300 as q
    lib = q.lib()
    peaks, peaks_src = load_peaks()
    props = torch.cuda.get_device_properties(local_rank)
    uuid = None
    try:
        u = str(props.uuid)
        uuid = u if u.startswith("GPU-") else "GPU-" + u
    except AttributeError:
        pass
    clocks = ClockSampler(uuid)

    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def flush():
        flush_buf.fill_(1)

    # ---------------- headline: A8W8 4096^3 ----------------
    w = W.a8w8_4096()
    A = torch.from_numpy(w.A).cuda()
    B = torch.from_numpy(w.B).cuda()
    a_s = torch.from_numpy(w.act_scale).cuda()
    w_s = torch.from_numpy(w.weight_scale).cuda()
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    # One step of the path: qmm_a8w8 with a workspace, i.e. the fp16 operand
    # pre-pass, then the SM-pair GEMM with the fused scaling (two kernels).
    ws = torch.empty(q.qmm_a8w8_workspace_bytes(M, K, N), dtype=torch.uint8, device="cuda")

    def pack():
        q.qmm_a8w8_pack(A, B, ws)

    def gemm():
        q.qmm_a8w8_packed(M, K, N, a_s, w_s, ws, out=C)

    def step():
        q.qmm_a8w8(A, B, a_s, w_s, out=C, workspace=ws)

    clocks.start()
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    # the whole step (the GEMM is launched as a programmatic dependent of the
    # pre-pass and overlaps its tail)
    times = time_gpu(step, args.steps, args.warmup, flush=flush)
    t1 = time.time()
    barrier()
    clocks.mark(t0, t1)
    kernel_name = q.last_kernel()
    # the GEMM kernel alone (operands packed once), for the roofline
    pack()
    gemm()
    gemm_kernel = q.last_kernel()
    t0g = time.time()
    gemm_times = time_gpu(gemm, max(20, min(args.steps, 200)), args.warmup, flush=flush)
    clocks.mark(t0g, time.time())
    q.check_device_error()
    mean_ms = statistics.mean(times)
    slow_ms = max_over_ranks(mean_ms)
    value = world * OPS / (slow_ms * 1e-3) / 1e12
    gemm_ms = statistics.mean(gemm_times)
    achieved = OPS / (gemm_ms * 1e-3) / 1e12

    # end to end: pinned host inputs -> device, call, result -> pinned host
    hA = torch.from_numpy(w.A).pin_memory()
    hB = torch.from_numpy(w.B).pin_memory()
    ha = torch.from_numpy(w.act_scale).pin_memory()
    hw = torch.from_numpy(w.weight_scale).pin_memory()
    hC = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()

    # the library's host-buffer call: row panels of A copied in, multiplied and
    # copied back with the copies of other panels in flight
    ws_host = torch.empty(q.qmm_a8w8_host_workspace_bytes(M, K, N, M, N), dtype=torch.uint8, device="cuda")

    def e2e_call():
        q.qmm_a8w8_host(hA, hB, ha, hw, out=hC, workspace=ws_host)

    e2e_steps = min(args.steps, 50)
    e2e_times = time_gpu(e2e_call, e2e_steps, 3)
    e2e_ms = max_over_ranks(statistics.mean(e2e_times))
    h2d = hA.numel() + hB.numel() + 4 * (ha.numel() + hw.numel())
    d2h = 2 * hC.numel()

    # the int8 denominators the metric names: the legacy int8 tensor path's
    # rate (mma.sync s8, measured here), and cuBLAS's int8 GEMM on the operands
    t0p = time.time()
    imma_tops = int8_mma_peak(q, torch)
    cublas_tops = cublas_int8_tops(torch, A, B)
    clocks.mark(t0p, time.time())

    rows = {}
    if not args.no_secondary:
        rows = secondary(q, torch, flush, clocks, peaks)
    clk = clocks.stop()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    cpu = cpu_baseline_a8w8() if world == 1 else None
    line = {
        "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": slow_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "s8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N, "out": "bf16",
                   "l2": "flushed before every timed iteration (256 MiB write)",
                   "parallelism": f"replicas x{world}", "kernel": kernel_name,
                   "contraction": "int8 operands copied once to exact fp16 (pre-pass), then exact products on "
                                  "tcgen05 kind::f16 in 2-SM pairs, K-chunked fp32 TMEM accumulators "
                                  "(double-buffered) drained to int32",
                   "prepass_exposed_ms": mean_ms - gemm_ms},
        "roofline": {"bound": "tensor", "kernel": gemm_kernel, "achieved": achieved, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                     "traffic": kernel_traffic(gemm_kernel), "kernel_ms": gemm_ms,
                     "peak_source": f"{peaks_src} dense bf16 (burst); fp16 kind::f16 runs at the same rate",
                     "int8_imma_peak": imma_tops, "frac_int8_imma": achieved / imma_tops,
                     "int8_peak_source": "measured in this run: mma.sync m16n8k32 s8 (sm_103a has no tcgen05 "
                                         "kind::i8); the exact fp16 tcgen05 path runs above it",
                     "cublas_int8_gemm_tops": cublas_tops},
        "cpu_baseline": cpu,
        "e2e": {"value": world * OPS / (e2e_ms * 1e-3) / 1e12, "unit": "TOPS", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * args.steps,   # per step: the pre-pass + the GEMM
        "clocks": clk,
        "rows": rows,
        "configs": config_summary(rows, value, mean_ms, achieved, peaks, imma_tops),
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def case_setups(q, torch, peaks):
    """Setup functions for each benchmark workload. Each returns (call, use_flush, report),
    report(ms) -> dict. Inputs are created on the device before timing."""
    hbm = peaks["hbm_gbs"]
    tc = peaks["bf16_tflops"]

    def a8w8():
        w = W.a8w8_4096()
        A, B = torch.from_numpy(w.A).cuda(), torch.from_numpy(w.B).cuda()
        a_s, w_s = torch.from_numpy(w.act_scale).cuda(), torch.from_numpy(w.weight_scale).cuda()
        C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        return (lambda: q.qmm_a8w8(A, B, a_s, w_s, out=C)), True, \
            (lambda ms: {"us": ms * 1e3, "value": OPS / (ms * 1e-3) / 1e12, "unit": "TOPS"})

    def a8w8_single_pass():
        w = W.a8w8_4096()
        A, B = torch.from_numpy(w.A).cuda(), torch.from_numpy(w.B).cuda()
        a_s, w_s = torch.from_numpy(w.act_scale).cuda(), torch.from_numpy(w.weight_scale).cuda()
        C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        return (lambda: q.qmm_a8w8(A, B, a_s, w_s, out=C, workspace=None)), True, \
            (lambda ms: {"us": ms * 1e3, "value": OPS / (ms * 1e-3) / 1e12, "unit": "TOPS",
                         "frac": OPS / (ms * 1e-3) / 1e12 / tc, "note": "single-pass fused kernel, no workspace"})

    def gemv(Mg):
        def setup():
            g = W.decode_gemv(Mg)
            Ad = torch.from_numpy(g.A_bits.view(np.int16)).view(torch.bfloat16).cuda()
            Wd = torch.from_numpy(g.W).cuda()
            sd = torch.from_numpy(g.scale).cuda()
            Cd = torch.empty((Mg, 28672), dtype=torch.bfloat16, device="cuda")
            nbytes = 8192 * 28672 + Mg * 8192 * 2 + 28672 * 4 + Mg * 28672 * 2
            wsg = torch.empty(q.qmm_w8_dequant_workspace_bytes(torch.bfloat16, Mg, 8192, 28672), dtype=torch.uint8,
                              device="cuda")

            def report(ms):
                gbs = nbytes / (ms * 1e-3) / 1e9
                return {"us": ms * 1e3, "value": gbs, "unit": "GB/s", "bound": "hbm", "frac": gbs / hbm,
                        "algorithmic_bytes": nbytes}
            # the weight stream (235 MB) exceeds L2: no flush needed
            return (lambda: q.qmm_w8_dequant(Ad, Wd, sd, None, out=Cd, workspace=wsg)), False, report
        return setup

    def gemv_packed(Mg):
        def setup():
            g = W.decode_gemv(Mg)
            Ad = torch.from_numpy(g.A_bits.view(np.int16)).view(torch.bfloat16).cuda()
            Wd = torch.from_numpy(g.W).cuda()
            sd = torch.from_numpy(g.scale).cuda()
            Cd = torch.empty((Mg, 28672), dtype=torch.bfloat16, device="cuda")
            packed = q.qmm_w8_pack_decode_weight(Wd)   # once, outside the timed calls (a frozen weight)
            del Wd
            nbytes = 8192 * 28672 + Mg * 8192 * 2 + 28672 * 4 + Mg * 28672 * 2
            wsg = torch.empty(q.qmm_w8_dequant_packed_workspace_bytes(Mg, 8192), dtype=torch.uint8, device="cuda")

            def report(ms):
                gbs = nbytes / (ms * 1e-3) / 1e9
                return {"us": ms * 1e3, "value": gbs, "unit": "GB/s", "bound": "hbm", "frac": gbs / hbm,
                        "algorithmic_bytes": nbytes, "note": "weight re-laid out once for the decode kernel"}
            return (lambda: q.qmm_w8_dequant_packed(Ad, packed, 28672, sd, out=Cd, workspace=wsg)), False, report
        return setup

    def dql():
        d = W.dql_matmul_integer_8192x4096x11008()
        x = torch.from_numpy(d.x).cuda()
        ws = torch.empty(q.dynamic_quantize_linear_workspace_bytes(x.numel()), dtype=torch.uint8, device="cuda")
        n = x.numel()

        def report(ms):
            gbs = 9 * n / (ms * 1e-3) / 1e9
            return {"us": ms * 1e3, "value": gbs, "unit": "GB/s", "bound": "hbm", "frac": gbs / hbm,
                    "algorithmic_bytes": 9 * n,
                    "note": f"9 B/element (x read twice, y written); {5 * n / (ms * 1e-3) / 1e9:.0f} GB/s "
                            "against the 5 B/element floor"}
        # x (134 MB) exceeds L2: no flush needed
        return (lambda: q.dynamic_quantize_linear(x, row_len=4096, workspace=ws)), False, report

    def mmi():
        d = W.dql_matmul_integer_8192x4096x11008()
        x = torch.from_numpy(d.x).cuda()
        y, _, zp, _ = q.dynamic_quantize_linear(x, row_len=4096)
        del x
        Bd, bz = torch.from_numpy(d.B).cuda(), torch.from_numpy(d.b_zp).cuda()
        Ci = torch.empty((8192, 11008), dtype=torch.int32, device="cuda")
        ops = 2.0 * 8192 * 4096 * 11008

        def report(ms):
            tops = ops / (ms * 1e-3) / 1e12
            return {"us": ms * 1e3, "value": tops, "unit": "TOPS", "bound": "tensor", "frac": tops / tc,
                    "note": "inputs + int32 output (440 MB) exceed L2"}
        wsm = torch.empty(q.matmul_integer_workspace_bytes(1, 8192, 4096, 11008, 0, 0), dtype=torch.uint8,
                          device="cuda")
        return (lambda: q.matmul_integer(y, Bd, a_zero_point=zp, b_zero_point=bz, out=Ci, workspace=wsm)), False, \
            report

    def batched():
        bm = W.batched_matmul_integer()
        Ab, Bb = torch.from_numpy(bm.A).cuda(), torch.from_numpy(bm.B).cuda()
        za = torch.tensor([bm.a_zp], dtype=torch.int8, device="cuda")
        zb = torch.tensor([bm.b_zp], dtype=torch.int8, device="cuda")
        Cb = torch.empty((8, 16, 512, 1024), dtype=torch.int32, device="cuda")
        ops = 2.0 * 65536 * 1024 * 1024
        nbytes = 65536 * 1024 + 1024 * 1024 + 65536 * 1024 * 4

        def report(ms):
            tops = ops / (ms * 1e-3) / 1e12
            gbs = nbytes / (ms * 1e-3) / 1e9
            return {"us": ms * 1e3, "value": tops, "unit": "TOPS", "frac_tensor": tops / tc, "gbs": gbs,
                    "frac_hbm": gbs / hbm}
        wsb = torch.empty(q.matmul_integer_workspace_bytes(128, 512, 1024, 1024, 512 * 1024, 0), dtype=torch.uint8,
                          device="cuda")
        return (lambda: q.matmul_integer(Ab, Bb, a_zero_point=za, b_zero_point=zb, out=Cb, workspace=wsb)), False, \
            report

    def w8_prefill():
        g = W.decode_gemv(4096)   # A bf16 [4096, 8192], W int8 [8192, 28672], per-column scale
        Ad = torch.from_numpy(g.A_bits.view(np.int16)).view(torch.bfloat16).cuda()
        Wd = torch.from_numpy(g.W).cuda()
        sd = torch.from_numpy(g.scale).cuda()
        Cd = torch.empty((4096, 28672), dtype=torch.bfloat16, device="cuda")
        wsp = torch.empty(q.qmm_w8_dequant_workspace_bytes(torch.bfloat16, 4096, 8192, 28672), dtype=torch.uint8,
                          device="cuda")
        ops = 2.0 * 4096 * 8192 * 28672

        def report(ms):
            tops = ops / (ms * 1e-3) / 1e12
            return {"us": ms * 1e3, "value": tops, "unit": "TOPS", "bound": "tensor", "frac": tops / tc,
                    "note": "bf16 x int8 weight (weight pre-pass to bf16 + SM-pair GEMM), fp32 accumulation"}
        return (lambda: q.qmm_w8_dequant(Ad, Wd, sd, None, out=Cd, workspace=wsp)), False, report

    def a8w8_acc(Ma, Ka, Na, b_trans):
        def setup():
            w = W.a8w8_acc(Ma, Ka, Na, seed=0, b_trans=b_trans)
            A, B = torch.from_numpy(w.A).cuda(), torch.from_numpy(w.B).cuda()
            acc = torch.from_numpy(w.acc_in).cuda()
            a_s, w_s = torch.from_numpy(w.act_scale).cuda(), torch.from_numpy(w.weight_scale).cuda()
            C = torch.empty((Ma, Na), dtype=torch.bfloat16, device="cuda")
            wsa = torch.empty(q.qmm_a8w8_acc_workspace_bytes(Ma, Ka, Na), dtype=torch.uint8, device="cuda")
            ops = 2.0 * Ma * Ka * Na
            nbytes = Ma * Ka + Ka * Na + Ma * Na * 4 + Ma * 4 + Na * 4 + Ma * Na * 2

            def report(ms):
                tops = ops / (ms * 1e-3) / 1e12
                gbs = nbytes / (ms * 1e-3) / 1e9
                return {"us": ms * 1e3, "value": tops, "unit": "TOPS", "frac_tensor": tops / tc, "gbs": gbs,
                        "frac_hbm": gbs / hbm, "algorithmic_bytes": nbytes,
                        "note": f"int32 acc_in + A @ B, {'B stored [N,K] (b_trans)' if b_trans else 'B [K,N]'}, "
                                "bf16 out"}
            call = lambda: q.qmm_a8w8_acc(A, B, a_s, w_s, acc_in=acc, b_trans=b_trans, out=C,  # noqa: E731
                                          workspace=wsa)
            return call, Ma * Ka + Ka * Na < 2 * FLUSH_BYTES // 3, report
        return setup

    def dq_chain():
        d = W.dql_matmul_integer_8192x4096x11008()
        rng = np.random.default_rng(9)
        x, Bd, bz = torch.from_numpy(d.x).cuda(), torch.from_numpy(d.B).cuda(), torch.from_numpy(d.b_zp).cuda()
        w_s = torch.from_numpy(rng.uniform(0.001, 0.01, 11008).astype(np.float32)).cuda()
        bias = torch.from_numpy(rng.standard_normal(11008).astype(np.float32)).cuda()
        Cf = torch.empty((8192, 11008), dtype=torch.float32, device="cuda")
        wsd = torch.empty(q.dynamic_quantize_matmul_workspace_bytes(8192, 4096, 11008), dtype=torch.uint8,
                          device="cuda")
        ops = 2.0 * 8192 * 4096 * 11008

        def report(ms):
            tops = ops / (ms * 1e-3) / 1e12
            return {"us": ms * 1e3, "value": tops, "unit": "TOPS", "frac_tensor": tops / tc,
                    "note": "x fp32 -> DynamicQuantizeLinear -> MatMulInteger(per-column w_zp) -> fp32 "
                            "* y_scale*w_scale[n] + bias[n], one call; weight converted every call"}
        return (lambda: q.dynamic_quantize_matmul(x, Bd, w_s, bz, bias, out=Cf, workspace=wsd)), False, report

    def dq_chain_packed():
        d = W.dql_matmul_integer_8192x4096x11008()
        rng = np.random.default_rng(9)
        x, Bd, bz = torch.from_numpy(d.x).cuda(), torch.from_numpy(d.B).cuda(), torch.from_numpy(d.b_zp).cuda()
        w_s = torch.from_numpy(rng.uniform(0.001, 0.01, 11008).astype(np.float32)).cuda()
        bias = torch.from_numpy(rng.standard_normal(11008).astype(np.float32)).cuda()
        Cf = torch.empty((8192, 11008), dtype=torch.float32, device="cuda")
        pw = q.dynamic_quantize_matmul_pack_weight(Bd)   # once, outside the timed calls
        wsd = torch.empty(q.dynamic_quantize_matmul_packed_workspace_bytes(8192, 4096), dtype=torch.uint8,
                          device="cuda")
        ops = 2.0 * 8192 * 4096 * 11008

        def report(ms):
            tops = ops / (ms * 1e-3) / 1e12
            return {"us": ms * 1e3, "value": tops, "unit": "TOPS", "frac_tensor": tops / tc,
                    "note": "the fused chain on a weight packed once (fp16 copy + column sums); per call: "
                            "DynamicQuantizeLinear into the fp16 operand, then the GEMM with its epilogue"}
        return (lambda: q.dynamic_quantize_matmul_packed(x, pw, w_s, bz, bias, out=Cf, workspace=wsd)), False, \
            report

    def conv(make):
        def setup():
            c = make()
            x, w = torch.from_numpy(c.x).cuda(), torch.from_numpy(c.w).cuda()
            xz, wz = torch.from_numpy(c.x_zp).cuda(), torch.from_numpy(c.w_zp).cuda()
            y = q.conv_integer(x, w, xz, wz, pads=c.pads, strides=c.strides, dilations=c.dilations, group=c.group)
            wsc = torch.empty(q.conv_integer_workspace_bytes(tuple(c.x.shape), tuple(c.w.shape), c.pads, c.strides,
                                                             c.dilations, c.group), dtype=torch.uint8, device="cuda")
            taps = int(np.prod(c.w.shape[1:]))
            ops = 2.0 * y.numel() * taps

            def report(ms):
                tops = ops / (ms * 1e-3) / 1e12
                return {"us": ms * 1e3, "value": tops, "unit": "TOPS", "frac_tensor": tops / tc,
                        "note": f"x {list(c.x.shape)} u8, w {list(c.w.shape)} s8, scalar x_zp, per-channel w_zp; "
                                "implicit GEMM: fp16 NHWC input, im2col tensor copies into the SM-pair GEMM"}
            call = lambda: q.conv_integer(x, w, xz, wz, pads=c.pads, strides=c.strides,  # noqa: E731
                                          dilations=c.dilations, group=c.group, out=y, workspace=wsc)
            return call, True, report
        return setup

    def w8():
        sw = W.w8_dequant_f32_64x256x192()
        As, Bs = torch.from_numpy(sw.A).cuda(), torch.from_numpy(sw.B).cuda()
        ss, zs = torch.from_numpy(sw.scale).cuda(), torch.from_numpy(sw.zero_point).cuda()
        Cs = torch.empty((64, 192), dtype=torch.float32, device="cuda")
        return (lambda: q.qmm_w8_dequant(As, Bs, ss, zs, out=Cs)), True, \
            (lambda ms: {"us": ms * 1e3, "unit": "us", "bound": "latency"})

    return {"a8w8_4096x4096x4096_bf16": a8w8,
            "a8w8_4096x4096x4096_bf16_single_pass": a8w8_single_pass,
            "w8_prefill_bf16_4096x8192x28672": w8_prefill,
            "decode_gemv_M1": gemv(1), "decode_gemv_M4": gemv(4), "decode_gemv_M16": gemv(16),
            "decode_gemv_packed_M1": gemv_packed(1), "decode_gemv_packed_M4": gemv_packed(4),
            "decode_gemv_packed_M16": gemv_packed(16),
            "dql_8192x4096": dql, "matmul_integer_8192x4096x11008": mmi,
            "batched_matmul_integer_65536x1024x1024": batched, "w8_dequant_f32_64x256x192": w8,
            "a8w8_acc_4096x4096x4096_bf16": a8w8_acc(4096, 4096, 4096, False),
            "a8w8_acc_4096x4096x4096_bf16_b_trans": a8w8_acc(4096, 4096, 4096, True),
            "a8w8_acc_decode_M1_8192x28672_b_trans": a8w8_acc(1, 8192, 28672, True),
            "a8w8_acc_decode_M1_8192x28672": a8w8_acc(1, 8192, 28672, False),
            "a8w8_acc_decode_M8_8192x28672_b_trans": a8w8_acc(8, 8192, 28672, True),
            "a8w8_acc_decode_M16_8192x28672_b_trans": a8w8_acc(16, 8192, 28672, True),
            "dql_matmul_dequant_fused_8192x4096x11008": dq_chain,
            "dql_matmul_dequant_fused_packed_8192x4096x11008": dq_chain_packed,
            "conv_integer_3x3_8x256x56x56": conv(W.conv2d_3x3_8x256x56x56),
            "conv_integer_1d_k3_4x512x3000": conv(W.conv1d_k3_4x512x3000)}


# The rows beyond the five configurations first, then the five (their compact
# summary closes the JSON line).
SECONDARY = ["a8w8_4096x4096x4096_bf16_single_pass", "w8_prefill_bf16_4096x8192x28672",
             "a8w8_acc_4096x4096x4096_bf16", "a8w8_acc_4096x4096x4096_bf16_b_trans",
             "a8w8_acc_decode_M1_8192x28672_b_trans", "a8w8_acc_decode_M1_8192x28672",
             "a8w8_acc_decode_M8_8192x28672_b_trans", "a8w8_acc_decode_M16_8192x28672_b_trans",
             "conv_integer_3x3_8x256x56x56",
             "conv_integer_1d_k3_4x512x3000", "dql_matmul_dequant_fused_8192x4096x11008",
             "dql_matmul_dequant_fused_packed_8192x4096x11008",
             "w8_dequant_f32_64x256x192", "dql_8192x4096", "matmul_integer_8192x4096x11008",
             "batched_matmul_integer_65536x1024x1024", "decode_gemv_M1", "decode_gemv_M4", "decode_gemv_M16",
             "decode_gemv_packed_M1", "decode_gemv_packed_M4", "decode_gemv_packed_M16"]


def config_summary(rows, value, step_ms, gemm_achieved, peaks, imma_tops):
    """Compact figures of the five benchmark configurations (the line's last key)."""
    def r3(v):
        return None if v is None else float(f"{v:.3g}")

    def pick(name, *keys):
        r = rows.get(name)
        if r is None:
            return None
        out = {k: r3(r[k]) if isinstance(r.get(k), float) else r.get(k) for k in keys if k in r}
        out["kernel"] = r.get("kernel")
        return out

    hbm = peaks["hbm_gbs"]
    s = {"peaks": {"hbm_gbs": hbm, "bf16_tflops": peaks["bf16_tflops"], "int8_imma_tops": r3(imma_tops)},
         "cfg1_w8_f32_64x256x192": pick("w8_dequant_f32_64x256x192", "us"),
         "cfg2_a8w8_4096": {"us": r3(step_ms * 1e3), "TOPS": r3(value),
                            "gemm_frac_bf16": r3(gemm_achieved / peaks["bf16_tflops"]),
                            "gemm_frac_int8_imma": r3(gemm_achieved / imma_tops)},
         "cfg3_dql_8192x4096": pick("dql_8192x4096", "us", "value", "frac"),
         "cfg3_mmi_8192x4096x11008": pick("matmul_integer_8192x4096x11008", "us", "value", "frac"),
         "cfg5_batched_mmi_65536x1024x1024": pick("batched_matmul_integer_65536x1024x1024", "us", "value",
                                                  "frac_tensor", "frac_hbm")}
    for m in (1, 4, 16):
        s[f"cfg4_gemv_M{m}_8192x28672"] = pick(f"decode_gemv_M{m}", "us", "value", "frac")
    for m in (1, 4, 16):
        s[f"cfg4_gemv_packed_M{m}"] = pick(f"decode_gemv_packed_M{m}", "us", "frac")
    return s


def secondary(q, torch, flush, clocks, peaks):
    out = {}
    setups = case_setups(q, torch, peaks)
    for name in SECONDARY:
        fn, use_flush, report = setups[name]()
        t0 = time.time()
        ts = time_gpu(fn, 20, 3, flush=flush if use_flush else None)
        clocks.mark(t0, time.time())
        r = report(statistics.mean(ts))
        r["kernel"] = q.last_kernel()
        out[name] = r
        del fn
        torch.cuda.empty_cache()
    return out


def run_case(args):
    """Time one workload alone (used for profiler captures of a single kernel)."""
    import torch
    import quantized_int8_matmul_gb300 as q
    peaks, _ = load_peaks()
    setups = case_setups(q, torch, peaks)
    fn, use_flush, report = setups[args.case]()
    flush = None
    if use_flush:
        buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        flush = lambda: buf.fill_(1)  # noqa: E731
    ts = time_gpu(fn, args.steps, args.warmup, flush=flush)
    q.check_device_error()
    r = report(statistics.mean(ts))
    r.update({"case": args.case, "kernel": q.last_kernel(), "steps": args.steps})
    print(json.dumps(r), flush=True)


if __name__ == "__main__":
    main()
