"""Benchmark of the fused MX-FP8 dim0 + dim1 cast with blocked scales.

One step = one call of mx_cast_dim0_dim1 (one kernel launch) on the
16384 x 16384 bf16 weight-like workload: read X once, write the row-major and
column-major e4m3 copies and both e8m0 scale sets in 128x4 blocked layout.
The metric is achieved HBM throughput: algorithmic bytes (2 B read + 1 + 1 B
written per element, plus the padded blocked scales) per second of device
time, and its fraction of the measured GB300 copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mx|reference]
                  [--row ROW] [--workload NAME] [--shape ...] [--graph]

--row times another row of the hot path instead (one JSON line each): the
dim0-only or dim1-only cast (dim0, dim1), the grouped-M MoE cast (grouped;
16640 x 5120, 4 groups), the 3D expert casts (experts: dim1, experts0: dim0,
experts01: both; 16 x 8192 x 5120), the standalone scale blocking (blocked;
262144 x 512), MX dequantisation to bf16 (dequant) and the tensorwise and
rowwise fp8 casts (tensorwise, rowwise; 16384 x 16384).  --graph replays the
timed steps from CUDA graphs (for launch-bound small workloads).

--impl reference times the CPU oracle (the plain C implementation used by the
tests) on the host cores on a bounded sample of the same workload.  Under
torchrun (N > 1) every rank casts its own copy of the workload on its own GPU
(weak scaling, no collective on the data path); rank 0 prints the line.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused MXFP8 dim0+dim1 cast HBM GB/s and fraction of GB300 HBM peak (1 GPU)"
NOMINAL_HBM_GBS = 8000.0   # nominal HBM bandwidth, the peak figure pytorch/ao PR #2990's perf analysis uses
WORKLOAD = "square16384_weight"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["mxfp8_block_scaled_dim0_gb300/csrc/mx_cast.cu",
                  "mxfp8_block_scaled_dim0_gb300/csrc/mx_common.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "mx_cast_fused_16384x16384.txt")
E2E_RUNS = 5                # timed end-to-end runs; the median is reported
E2E_SETS = 3                # end-to-end buffer sets and streams, used in rotation
HOLD_CYCLES = 2_000_000     # spin ahead of a timed region (about 1 ms at 2 GHz)


def algorithmic_bytes(M, K):
    """Bytes the fused cast must move: read X, write q0, q1 and both padded
    blocked scale buffers."""
    def blk(R, C):
        return -(-R // 128) * 128 * (-(-C // 4) * 4)
    return 2 * M * K + M * K + M * K + blk(M, K // 32) + blk(K, M // 32)


def _code_tokens(text):
    """Source text without comments and with whitespace collapsed, so that
    edits to comments or layout do not count as a kernel change."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash():
    """Hash of the fused kernel's code (comments and whitespace ignored)."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(units_scale=1.0):
    """dram__bytes_read.sum + dram__bytes_write.sum per full launch from the
    committed ncu summary, or None if absent or taken on other kernel code."""
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith(("#", " ", "|")):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256_16") != kernel_source_hash():
            return None
        return float(kv["dram_bytes_per_full_launch"]) * units_scale
    except (OSError, KeyError, ValueError):
        return None


def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---- clocks during the timed region ------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1].split()[0]))
                    smax.append(float(parts[2].split()[0]))
                except ValueError:
                    continue
                n += 1
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": n}


# ---- distributed plumbing (host logic; testable with gloo) ---------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value, ws, device=None):
    """Largest value over all ranks (identity when not distributed)."""
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_value(bytes_per_step, steps, n_ranks, max_elapsed_s):
    """Whole-job GB/s: bytes every rank moved, over the slowest rank's time."""
    return bytes_per_step * steps * n_ranks / max_elapsed_s / 1e9


def roofline(bytes_per_step, launches, steps, elapsed_s, peak, peak_kind, kernel, traffic,
             timing):
    """Roofline record of one rank's timed region.  The steps run back to
    back with no event between them, so a launch's duration is the region's
    time over the launches in it; `achieved` is a step's algorithmic bytes
    over a step's time (one launch per step for every row but the two-kernel
    ones, where it covers both kernels of the step)."""
    step_s = elapsed_s / steps
    achieved = bytes_per_step / step_s / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_kind": peak_kind, "traffic": traffic,
            "kernel": kernel, "launches_per_step": launches,
            "avg_launch_us": 1e6 * step_s / launches,
            "timing": timing + ", %d steps back to back, no events between them" % steps}


# ---- CPU oracle timing (the CPU baseline and the reference arm) ---------------

def host_cores():
    """Host threads this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or "unknown"."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def time_oracle(seconds_budget=12.0, rows_per_slab=512, threads=1):
    """Time the oracle's fused cast (dim0 + dim1 + blocked scales) on row slabs
    of the workload, on `threads` host threads, until the budget is spent.
    Returns (GB/s, rows, seconds, threads used)."""
    import oracle
    from mxfp8_block_scaled_dim0_gb300 import workloads as W
    M, K = W.WORKLOADS[WORKLOAD].shape
    x = W.bf16_bits(W.normal((rows_per_slab, K), W.WORKLOADS[WORKLOAD].seed, std=0.02))
    used = oracle.set_threads(threads)
    try:
        done_rows, t_used = 0, 0.0
        while done_rows == 0 or (t_used < seconds_budget and done_rows < M):
            t0 = time.perf_counter()
            oracle.cast_dim0_dim1_blocked(x)
            t_used += time.perf_counter() - t0
            done_rows += rows_per_slab
    finally:
        oracle.set_threads(1)
    gbs = algorithmic_bytes(done_rows, K) / t_used / 1e9
    return gbs, done_rows, t_used, used


def cpu_baseline(seconds_budget):
    """The oracle on all host cores and on one, on row slabs of the workload
    (same value mix); the all-core figure is the baseline's value."""
    n = host_cores()
    gbs_n, rows_n, secs_n, used = time_oracle(seconds_budget * 2 / 3, rows_per_slab=2048, threads=n)
    gbs_1, rows_1, secs_1, _ = time_oracle(seconds_budget / 3, rows_per_slab=512, threads=1)
    return {"value": gbs_n, "unit": "GB/s", "cores": used, "kind": "oracle",
            "sample": "first %d rows x 16384 cols of the 16384x16384 workload (same value mix), "
                      "%.1f s, fused dim0+dim1+blocked scales, %d threads (OpenMP over rows / "
                      "columns)" % (rows_n, secs_n, used),
            "cores_1": {"value": gbs_1, "unit": "GB/s",
                        "sample": "first %d rows, %.1f s, single thread" % (rows_1, secs_1)},
            "nproc": n, "cpu_model": cpu_model()}


def run_reference(args, budget_s=90.0):
    """Reference arm: the oracle as it stands on the host cores.  Each step is
    one fused cast of a bounded row slab of the workload, sized so that the
    whole run (warm-up included) takes about budget_s seconds."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from mxfp8_block_scaled_dim0_gb300 import workloads as W
    M, K = W.WORKLOADS[WORKLOAD].shape
    seed = W.WORKLOADS[WORKLOAD].seed
    n = host_cores()
    # Single-thread figure on a small slab, for the record.
    gbs_1, rows_1, secs_1, _ = time_oracle(min(3.0, budget_s / 10), rows_per_slab=256, threads=1)
    used = oracle.set_threads(n)
    try:
        calib = W.bf16_bits(W.normal((32 * n, K), seed, std=0.02))
        t0 = time.perf_counter()
        oracle.cast_dim0_dim1_blocked(calib)
        t_row = (time.perf_counter() - t0) / (32 * n)
        rows = int(budget_s * 0.9 / (args.steps + args.warmup) / t_row) // 32 * 32
        rows = max(32, min(M, rows))
        x = W.bf16_bits(W.normal((rows, K), seed, std=0.02))
        times = []
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            oracle.cast_dim0_dim1_blocked(x)
            dt = time.perf_counter() - t0
            if i >= args.warmup:
                times.append(dt)
    finally:
        oracle.set_threads(1)
    t = sum(times)
    rows_total = rows * len(times)
    value = algorithmic_bytes(rows, K) * len(times) / t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "shape": [16384, 16384],
                   "sample": "%d-row slab of the workload per step (bounded CPU sample)" % rows},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": used, "kind": "oracle",
                         "sample": "%d rows x %d cols over %d steps, %d threads"
                                   % (rows_total, K, len(times), used),
                         "cores_1": {"value": gbs_1, "unit": "GB/s",
                                     "sample": "%d rows, %.1f s, single thread" % (rows_1, secs_1)},
                         "nproc": n, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---- GPU arm ----------------------------------------------------------------------

def blk(R, C):
    return -(-R // 128) * 128 * (-(-C // 4) * 4)


class Row:
    """One scope row of the hot path as a timed step: how to build its buffers,
    how to call it through the binding, and the bytes it must move."""

    def __init__(self, name, workload, kernel, bytes_per_step, launches, build, call,
                 inputs, outputs):
        self.name, self.workload, self.kernel = name, workload, kernel
        self.bytes_per_step, self.launches = bytes_per_step, launches
        self.build, self.call, self.inputs, self.outputs = build, call, inputs, outputs


def hold_gpu(torch, stream):
    """Enqueue a short spin kernel (about a millisecond) on `stream`, ahead of
    a timed region's start event: the GPU is then still busy while the host
    issues the region's first launches, so the host's launch latency does not
    sit between the two events.  The spin itself is outside the region."""
    if hasattr(torch.cuda, "_sleep"):
        with torch.cuda.stream(stream):
            torch.cuda._sleep(HOLD_CYCLES)


def make_row(row, args, dev, rank):
    import torch
    import mxfp8_block_scaled_dim0_gb300 as mx
    from mxfp8_block_scaled_dim0_gb300 import workloads as W
    u8 = lambda n: torch.empty(n, dtype=torch.uint8, device=dev)

    if row in ("fused", "dim1", "dim0", "dequant", "tensorwise", "rowwise"):
        wl = args.workload or WORKLOAD
        if args.shape:
            M, K = args.shape
            wl = "custom_%dx%d_weight" % (M, K)
            gen = lambda i: W.normal((M, K), 1003 + 100 * i + rank, device=dev, std=0.02)
        else:
            M, K = W.WORKLOADS[wl].shape
            gen = lambda i: W.make(wl, device=dev)["x"] if i == 0 else \
                W.normal((M, K), W.WORKLOADS[wl].seed + 100 * i + rank, device=dev, std=0.02)
        if row == "fused":
            def build(i):
                return (gen(i), torch.empty((M, K), dtype=torch.uint8, device=dev),
                        u8(mx.mx_blocked_bytes(M, K // 32)),
                        torch.empty((K, M), dtype=torch.uint8, device=dev),
                        u8(mx.mx_blocked_bytes(K, M // 32)))
            return Row("fused", wl, "mx_cast_kernel<fused2d>", algorithmic_bytes(M, K), 1, build,
                       lambda a, st: mx.mx_cast_dim0_dim1(*a, stream=st), (0,), (1, 2, 3, 4))

        if row == "dim0":
            def build(i):
                return (gen(i), torch.empty((M, K), dtype=torch.uint8, device=dev),
                        u8(mx.mx_blocked_bytes(M, K // 32)))
            return Row("dim0", wl, "mx_cast_kernel<dim0>", 2 * M * K + M * K + blk(M, K // 32), 1,
                       build, lambda a, st: mx.mx_cast_dim0(*a, stream=st), (0,), (1, 2))
        if row == "tensorwise":
            # Two passes over x (global amax, then the cast) and the q write.
            def build(i):
                return (gen(i), torch.empty((M, K), dtype=torch.uint8, device=dev),
                        torch.empty(1, dtype=torch.float32, device=dev),
                        torch.empty(1, dtype=torch.float32, device=dev))
            return Row("tensorwise", wl, "tensor_amax_kernel + tensorwise_kernel",
                       2 * M * K + 2 * M * K + M * K + 8, 2, build,
                       lambda a, st: mx.mx_cast_tensorwise(*a, stream=st), (0,), (1, 2, 3))
        if row == "rowwise":
            def build(i):
                return (gen(i), torch.empty((M, K), dtype=torch.uint8, device=dev),
                        torch.empty(M, dtype=torch.bfloat16, device=dev))
            kernel = "rowwise_bulk_kernel" if K <= 24576 else "rowwise_kernel"
            return Row("rowwise", wl, kernel, 2 * M * K + M * K + 2 * M, 1, build,
                       lambda a, st: mx.mx_cast_rowwise(*a, stream=st), (0,), (1, 2))
        if row == "dequant":
            # The dim0 copy of the workload (cast once, untimed) back to bf16.
            def build(i):
                q, s_blk = mx.cast_dim0(gen(i))
                return (q, s_blk, torch.empty((M, K), dtype=torch.bfloat16, device=dev))
            kernel = "dequant_tma_kernel" if K >= 1024 else "dequant_blocked_kernel"
            return Row("dequant", wl, kernel, M * K + blk(M, K // 32) + 2 * M * K,
                       1, build, lambda a, st: mx.mx_dequant_blocked(*a, stream=st), (0, 1), (2,))

        def build(i):
            return (gen(i), torch.empty((K, M), dtype=torch.uint8, device=dev),
                    u8(mx.mx_blocked_bytes(K, M // 32)))
        return Row("dim1", wl, "mx_cast_kernel<dim1>", 2 * M * K + M * K + blk(K, M // 32), 1,
                   build, lambda a, st: mx.mx_cast_dim1(*a, stream=st), (0,), (1, 2))

    if row == "grouped":
        wl = args.workload or "moe16640x5120_g4"
        M, K = W.WORKLOADS[wl].shape
        G = W.WORKLOADS[wl].groups
        n0 = mx.mx_grouped_m_scale_bytes(M, K, G, 0)
        n1 = mx.mx_grouped_m_scale_bytes(M, K, G, 1)

        def build(i):
            w = W.make(wl, device=dev)
            x = w["x"] if i == 0 else W.normal((M, K), W.WORKLOADS[wl].seed + 100 * i, device=dev)
            return (x, w["offs"].to(dev), torch.empty((M, K), dtype=torch.uint8, device=dev), u8(n0),
                    torch.empty(G + 1, dtype=torch.int64, device=dev),
                    torch.empty((K, M), dtype=torch.uint8, device=dev), u8(n1),
                    torch.empty(G + 1, dtype=torch.int64, device=dev),
                    torch.empty(1, dtype=torch.int32, device=dev))
        nbytes = 2 * M * K + 4 * G + M * K + n0 + M * K + n1 + 16 * (G + 1) + 4
        # Up to 1024 groups the cast kernel builds its group table itself (one
        # launch); more groups take the offsets kernel first.
        one = G <= 1024
        return Row("grouped", wl, "mx_cast_kernel<grouped>" if one else
                   "group_offsets_kernel + mx_cast_kernel<grouped>", nbytes, 1 if one else 2,
                   build, lambda a, st: mx.mx_cast_grouped_m(*a, stream=st), (0, 1),
                   (2, 3, 4, 5, 6, 7, 8))

    if row in ("experts", "experts0", "experts01"):
        wl = args.workload or "experts16x8192x5120"
        E, N, K = W.WORKLOADS[wl].shape
        if args.shape:
            E, N, K = args.shape
            wl = "custom_experts_%dx%dx%d" % (E, N, K)
        ns = mx.mx_3d_scale_bytes(E, N, K)
        n0 = mx.mx_3d_dim0_scale_bytes(E, N, K)
        if row == "experts0":
            def build(i):
                w = W.experts(E, N, K, 1005 + 100 * i, device=dev)
                return (w, torch.empty((E, N, K), dtype=torch.uint8, device=dev), u8(n0))
            return Row("experts0", wl, "mx_cast_kernel<experts0>", 3 * E * N * K + n0, 1, build,
                       lambda a, st: mx.mx_cast_3d_dim0(*a, stream=st), (0,), (1, 2))
        if row == "experts01":
            def build(i):
                w = W.experts(E, N, K, 1005 + 100 * i, device=dev)
                return (w, torch.empty((E, N, K), dtype=torch.uint8, device=dev), u8(n0),
                        torch.empty((K, E * N), dtype=torch.uint8, device=dev), u8(ns))
            return Row("experts01", wl, "mx_cast_kernel<experts01>", 4 * E * N * K + n0 + ns, 1,
                       build, lambda a, st: mx.mx_cast_3d_dim0_dim1(*a, stream=st), (0,),
                       (1, 2, 3, 4))

        def build(i):
            w = W.experts(E, N, K, 1005 + 100 * i, device=dev)
            return (w, torch.empty((K, E * N), dtype=torch.uint8, device=dev), u8(ns))
        return Row("experts", wl, "mx_cast_kernel<experts>", 3 * E * N * K + ns, 1, build,
                   lambda a, st: mx.mx_cast_3d_dim1(*a, stream=st), (0,), (1, 2))

    if row == "blocked":
        R, C = args.shape or (262144, 512)
        wl = "scales_%dx%d" % (R, C)

        def build(i):
            g = torch.Generator(device=dev)
            g.manual_seed(77 + i)
            s = torch.randint(0, 256, (R, C), dtype=torch.uint8, device=dev, generator=g)
            return (s, u8(mx.mx_blocked_bytes(R, C)))
        return Row("blocked", wl, "to_blocked_kernel", R * C + blk(R, C), 1, build,
                   lambda a, st: mx.mx_scales_to_blocked(*a, stream=st), (0,), (1,))
    raise ValueError(row)


def run_gpu(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)

    import mxfp8_block_scaled_dim0_gb300 as mx
    mx.library()

    # Clock samples cover the timed region; nvidia-smi starts now, while the
    # buffers are built, so that no idle pause is needed before timing (a
    # GPU left idle before the timed region ran its first steps slower).
    gpu_index = dev.index if ws > 1 else int(
        (os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0] or "0").strip() or 0)
    clocks = ClockSampler(gpu_index)
    clocks.start()

    R = make_row(args.row, args, dev, rank)
    nbytes = R.bytes_per_step
    stream = torch.cuda.current_stream(dev)
    # Two buffer sets, each larger than the 129 MB L2, alternated step by step.
    sets = [R.build(0), R.build(1)]

    def step(i, st=stream):
        R.call(sets[i & 1], st)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)

    graph = None
    if args.graph:
        # Launch-bound small workloads: capture the steps in a CUDA graph so
        # that host-side launch overhead stays out of the timed region.
        per_graph = min(args.steps, 100)
        args.steps = max(1, args.steps // per_graph) * per_graph
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cs = torch.cuda.current_stream()
            for i in range(per_graph):
                step(i, cs)
        graph.replay()
        torch.cuda.synchronize(dev)

    # Timed region: K steps back to back between two events on the launching
    # stream.  No event is recorded between steps: an event between two
    # programmatic-dependent launches would end their overlap and add launch
    # latency to what it measures.
    t_beg = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize(dev)
    hold_gpu(torch, stream)
    t_beg.record(stream)
    if graph is not None:
        for _ in range(args.steps // per_graph):
            graph.replay()
    else:
        for i in range(args.steps):
            step(i)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clock_info = clocks.stop()
    barrier(ws)
    elapsed = t_beg.elapsed_time(t_end) / 1e3
    max_elapsed = max_over_ranks(elapsed, ws, dev)
    value = whole_job_value(nbytes, args.steps, ws, max_elapsed)
    peak, peak_kind = hbm_peak()

    # End to end through the public API with host buffers: every step copies
    # its inputs from pinned host memory, calls the cast, and copies every
    # output back to pinned host memory.  Consecutive steps rotate over
    # E2E_SETS buffer sets on as many streams, so that the device-to-host
    # copies of step i run while the host-to-device copies of the next steps
    # do (separate copy engines), and the cast of step i is off the copy
    # engines' path: with two sets, step i+2's inputs wait for step i's cast
    # and outputs on the same stream.
    e2e = None
    if args.e2e_steps > 0:
        esets = sets + [R.build(k) for k in range(len(sets), E2E_SETS)]
        streams = [torch.cuda.Stream(dev) for _ in range(E2E_SETS)]
        host_in = [{j: esets[k][j].cpu().pin_memory() for j in R.inputs} for k in range(E2E_SETS)]
        host_out = [{j: torch.empty(esets[k][j].shape, dtype=esets[k][j].dtype).pin_memory()
                     for j in R.outputs} for k in range(E2E_SETS)]

        def e2e_step(i):
            k = i % E2E_SETS
            st = streams[k]
            with torch.cuda.stream(st):
                for j in R.inputs:
                    esets[k][j].copy_(host_in[k][j], non_blocking=True)
                R.call(esets[k], st)
                for j in R.outputs:
                    host_out[k][j].copy_(esets[k][j], non_blocking=True)

        for i in range(E2E_SETS):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        # E2E_RUNS timed runs of e2e_steps steps each; the line reports the
        # median run.  One run lasts about 40 ms at 16384^2, short enough for
        # a stall of the host link (about 70 ms, seen in one run of three now
        # and then) to cut a single run's figure to a third.
        runs = []
        for _ in range(E2E_RUNS):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier(ws)
            hold_gpu(torch, streams[0])
            a.record(streams[0])
            for s in streams[1:]:
                s.wait_event(a)
            for i in range(args.e2e_steps):
                e2e_step(i)
            for s in streams[1:]:
                streams[0].wait_stream(s)
            b.record(streams[0])
            torch.cuda.synchronize(dev)
            runs.append(max_over_ranks(a.elapsed_time(b) / 1e3, ws, dev))
        e_el = statistics.median(runs)
        h2d = sum(t.numel() * t.element_size() for t in host_in[0].values())
        d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
        e2e = {"value": whole_job_value(nbytes, args.e2e_steps, ws, e_el), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": args.e2e_steps, "ms_per_step": 1e3 * e_el / args.e2e_steps,
               "runs": [whole_job_value(nbytes, args.e2e_steps, ws, r) for r in runs],
               "timing": "median of %d timed runs of %d steps each" % (E2E_RUNS, args.e2e_steps),
               "pipelining": "%d streams, %d buffer sets: the D2H of step i overlaps the H2D of "
                             "the next steps" % (E2E_SETS, E2E_SETS)}
        del host_in, host_out, esets

    cpu = None
    if (rank == 0 and ws == 1 and args.cpu_seconds > 0 and R.name == "fused" and not args.shape
            and not args.workload):
        cpu = cpu_baseline(args.cpu_seconds)

    if rank == 0:
        shape = list(sets[0][0].shape)
        line = {
            "metric": METRIC if R.name == "fused" else METRIC.replace("fused MXFP8 dim0+dim1 cast",
                                                                      "MXFP8 %s" % R.name),
            "value": value, "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * max_elapsed / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": R.workload, "row": R.name, "shape": shape,
                       "bytes_per_step": nbytes,
                       "l2": "inputs %d MiB each, two buffer sets alternated (L2 is 129 MB)"
                             % (sets[0][0].numel() * sets[0][0].element_size() >> 20),
                       "parallelism": "replicas" if ws > 1 else "single"},
            "roofline": roofline(nbytes, R.launches, args.steps, elapsed, peak, peak_kind,
                                 R.kernel, measured_traffic() if R.name == "fused"
                                 and not args.shape and not args.workload else None,
                                 "cuda graph replay" if graph is not None else "stream launches"),
            "frac_of_peak": value / ws / peak,
            # the pages' nominal HBM figure (8 TB/s), beside the measured copy peak
            "frac_of_nominal": {"value": value / ws / NOMINAL_HBM_GBS, "nominal_gbs": NOMINAL_HBM_GBS},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": R.launches * args.steps,
            "clocks": clock_info,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["mx", "reference"], default="mx")
    p.add_argument("--e2e-steps", type=int, default=12)
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--shape", type=int, nargs="+", default=None,
                   help="fused / dim1: M K of a matrix of the same value mix instead; "
                        "experts: E N K; blocked: R C of the scale matrix (profiling)")
    p.add_argument("--row", choices=["fused", "dim1", "dim0", "grouped", "experts", "experts0",
                                     "experts01", "blocked", "dequant", "tensorwise", "rowwise"],
                   default="fused", help="which row of the hot path one step runs")
    p.add_argument("--workload", default=None, help="named workload for the row")
    p.add_argument("--graph", action="store_true",
                   help="replay the timed steps from a CUDA graph (small, launch-bound workloads)")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
