"""Benchmark of the RMSNorm forward hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c5a]
                    [--impl ours|reference] [--no-cpu-baseline] [--no-e2e]

A step is one full RMSNorm forward over the workload (all rows) through the
C ABI.  Prints ONE JSON line (rank 0).  Default workload: c5a, x (262144, 8192)
bf16 in/out with fp32 arithmetic, 8.59 GB moved per step (larger than L2, so
no L2 flush is needed between steps).  Under torchrun (N > 1) every rank runs
the same workload on its own GPU (rows are independent: weak scaling, no
data-path collective); the time is the max over ranks.

``--impl reference`` times the CPU oracle on the host cores on a bounded
sample of the same workload (the only other leg that executes ``oracle/``).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
# GB300 datasheet HBM3e bandwidth, reported beside the measured copy peak.
NOMINAL_HBM_GBS = 7900.0
L2_BYTES = 129e6
# Timed after the main region of the default run, same method and clocks: the
# other graded RMSNorm config, the few-row split-row config, the few very wide
# rows, and the prefill-logit row softmax.
SECONDARY_DEFAULT = ("c4", "c5b", "w16m", "w4m", "sm_prefill_f32", "sm_prefill_bf16",
                     "sm_wide_f32")
METRIC = "RMSNorm GB/s and rows/s on 1 GB300; % of HBM roofline"
METRIC_SOFTMAX = "row softmax GB/s and rows/s on 1 GB300; % of HBM roofline"


# ------------------------------------------------------------------ helpers --

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(files=None) -> str:
    """Hash of CUDA sources (all of csrc/, or the named files); a profile's
    traffic figure is valid only for the sources it was captured from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "row_wise_rmsnorm_fwd_gb300", "csrc")
    names = sorted(files) if files else sorted(
        n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh", ".h")))
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary profiles/<kernel>_<workload>.txt (lines 'traffic_bytes_per_launch:',
    'kernel_source_files:' and 'kernel_source_hash:'); None if there is none or
    if those sources have changed since the capture."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith(" "):
                k, v = line.split(":", 1)
                fields.setdefault(k.strip(), v.strip())
    files = fields.get("kernel_source_files", "").split()
    try:
        ok = fields.get("kernel_source_hash") == kernel_source_hash(files or None)
    except OSError:
        ok = False
    if ok and "traffic_bytes_per_launch" in fields:
        return int(float(fields["traffic_bytes_per_launch"].split()[0]))
    return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._thread = threading.Thread(target=self._read, daemon=True)
            self._thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def roofline_block(achieved, peak, peak_src, traffic=None):
    """The roofline object: `frac` is of the measured copy peak (a torch
    copy's read+write rate, so a kernel that streams reads and writes
    separately can sit a little above 1); `frac_of_nominal` is of the
    datasheet HBM3e bandwidth."""
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak,
            "peak_source": (f"{peak_src} copy peak (MEASURED_PEAKS.json hbm_gbs: torch "
                            "b.copy_(a), read+write bytes)" if peak_src == "measured"
                            else f"{peak_src} copy peak"),
            "nominal_gbs": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
            "traffic": traffic}


def max_over_ranks(values, device="cpu"):
    """All-reduce a list of timings with MAX over the ranks of the default
    process group (NCCL on GPUs, gloo on CPU); returns the reduced list."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def weak_scaling_rates(world, bytes_per_step, rows_per_step, steps, slowest_ms):
    """Whole-job GB/s and rows/s: every rank processed the full workload in
    at most `slowest_ms` (the max over ranks)."""
    seconds = slowest_ms / 1e3
    return (world * bytes_per_step * steps / seconds / 1e9,
            world * rows_per_step * steps / seconds)


def device_info(dev):
    """GPU name, SM count and L2 size of `dev`, and the repository's git commit."""
    import torch
    props = torch.cuda.get_device_properties(dev)
    sha = None
    try:
        sha = subprocess.run(["git", "rev-parse", "--short", "HEAD"], cwd=ROOT,
                             capture_output=True, text=True, timeout=10).stdout.strip() or None
    except (OSError, subprocess.SubprocessError):
        pass
    return {"name": props.name, "sms": props.multi_processor_count,
            "l2_bytes": getattr(props, "L2_cache_size", None),
            "memory_bytes": props.total_memory, "git": sha}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------ CPU baseline --

_oracle_out = threading.local()


def _oracle_chunk_call(oracle, wl, x, w):
    """One oracle call on a host chunk of rows (the arithmetic is all in C).
    Each thread writes into its own output buffers, reused from call to
    call: fresh buffers would make the threads fault pages in side by side,
    which the host kernel serialises."""
    import numpy as np

    bufs = getattr(_oracle_out, "bufs", None)
    if bufs is None or bufs[0].shape != x.shape:
        bufs = (np.zeros(x.shape, np.float64), np.zeros(x.shape, np.uint16))
        _oracle_out.bufs = bufs
    y64, y16 = bufs
    softmax = wl.op == "softmax"
    if wl.dtype == "bf16":
        if softmax:
            oracle.rowsoftmax_bf16(x, out64=y64, out16=y16)
        else:
            oracle.rmsnorm_bf16(x, w, wl.eps, out64=y64, out16=y16)
    elif softmax:
        oracle.rowsoftmax_f32(x, out=y64)
    else:
        oracle.rmsnorm_f32(x, w, wl.eps, out=y64)


def host_cores() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def cpu_oracle_sample(wl, budget_s: float = 10.0, threads: int = 1, max_rounds: int = 64):
    """Time the oracle (as it stands) on bounded samples of the workload's rows.

    Each round draws ``threads`` fresh chunks of rows (outside the clock), then
    ``threads`` host threads run the oracle on one chunk each at the same time
    (the oracle is a C library called through ctypes, which releases the
    interpreter lock); the wall clock of the rounds is summed until about
    ``budget_s`` seconds.  ``threads=1`` is the plain single-thread oracle."""
    import concurrent.futures as cf

    import oracle
    from row_wise_rmsnorm_fwd_gb300 import workloads

    oracle.build()
    softmax = wl.op == "softmax"
    chunk_rows = max(1, min(wl.rows, (1 << 22) // wl.hidden))
    w = None
    if not softmax:
        w = workloads.make_w(wl)
        w = workloads.bf16_bits(w) if wl.dtype == "bf16" else w.numpy()

    def draw(k):
        x = workloads.make_x(wl, rows=chunk_rows, seed_offset=k)
        return workloads.bf16_bits(x) if wl.dtype == "bf16" else x.numpy()

    done_rows, elapsed, rounds = 0, 0.0, 0
    with cf.ThreadPoolExecutor(threads) as ex:
        while elapsed < budget_s and rounds < max_rounds:
            chunks = list(ex.map(draw, range(rounds * threads, (rounds + 1) * threads)))
            t0 = time.perf_counter()
            list(ex.map(lambda c: _oracle_chunk_call(oracle, wl, c, w), chunks))
            elapsed += time.perf_counter() - t0
            done_rows += threads * chunk_rows
            rounds += 1
    bytes_done = (2 * done_rows * wl.hidden) * wl.elem_bytes + \
        (0 if softmax else rounds * threads * wl.hidden * wl.elem_bytes)
    how = ("single-thread" if threads == 1 else
           f"{threads} host threads, one chunk each at a time,")
    return {
        "value": bytes_done / elapsed / 1e9,
        "unit": "GB/s",
        "rows_per_s": done_rows / elapsed,
        "cores": threads,
        "kind": "oracle",
        "sample": f"{done_rows} rows x {wl.hidden} of workload {wl.name}: {rounds} rounds of "
                  f"{threads} chunk(s) of {chunk_rows} rows ({elapsed:.1f} s wall clock of "
                  f"{how} fp64 oracle)",
        "seconds": elapsed,
    }


def cpu_baseline_line(wl):
    """The bench line's cpu_baseline: the oracle row-parallel over all host
    cores, with the single-thread figure beside it."""
    par = cpu_oracle_sample(wl, budget_s=10.0, threads=host_cores())
    one = cpu_oracle_sample(wl, budget_s=5.0, threads=1)
    for c in (par, one):
        c.pop("seconds", None)
    par["single_thread"] = one
    return par


def run_reference(args, wl):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    budget = 10.0 / max(1, args.steps)      # every step runs at least one round
    threads = host_cores()
    for _ in range(args.warmup):
        cpu_oracle_sample(wl, budget_s=0.1, threads=threads, max_rounds=1)
    per = []
    for _ in range(args.steps):
        per.append(cpu_oracle_sample(wl, budget_s=budget, threads=threads))
    total_bytes = sum(c["value"] * c["seconds"] for c in per)
    total_s = sum(c["seconds"] for c in per)
    value = total_bytes / total_s
    line = {
        "impl": "reference",
        "metric": METRIC_SOFTMAX if wl.op == "softmax" else METRIC, "value": value,
        "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(wl, world),
        "rows_per_s": sum(c["rows_per_s"] * c["seconds"] for c in per) / total_s,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} steps, each: {per[-1]['sample']}"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def forced(args) -> bool:
    return bool(args.path != "auto" or args.cluster or args.grid or args.threads or args.chunk
                or args.stages or args.epilogue != "none")


def l2_note(wl, args=None) -> str:
    if wl.bytes_per_call > 4 * 129e6:
        return "inputs larger than L2 (no flush needed)"
    if args is not None and args.l2 == "hot":
        return "L2 hot: no flush between steps (inputs may be served from L2)"
    return "L2 flushed between steps (read of a 258 MB buffer)"


def config_block(wl, world, args=None):
    extra = {}
    if args is not None and forced(args):
        extra["forced"] = {"path": args.path, "cluster": args.cluster, "grid": args.grid,
                           "threads": args.threads, "chunk_bytes": args.chunk,
                           "stages": args.stages, "epilogue": args.epilogue}
    return {**extra,
        "workload": f"{wl.name}: {wl.description}",
        "shape": list(wl.shape), "io_dtype": wl.dtype, "eps": wl.eps,
        "bytes_per_step_per_gpu": wl.bytes_per_call,
        "rows_per_step_per_gpu": wl.rows,
        "l2": l2_note(wl, args),
        "parallelism": f"rows replicated per GPU x{world} (independent rows, no collective)",
    }


# -------------------------------------------------------------- GPU timing --

def run_ours(args, wl):
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    import __graft_entry__
    __graft_entry__.build()
    from row_wise_rmsnorm_fwd_gb300 import binding, workloads

    x = workloads.make_x(wl, device="cuda")
    softmax = wl.op == "softmax"
    w = torch.empty(0, device="cuda") if softmax else workloads.make_w(wl, device="cuda")
    y = torch.empty_like(x)
    rows, hidden = wl.rows, wl.hidden
    stream = torch.cuda.current_stream()
    handle = stream.cuda_stream
    options = None
    if softmax:
        staged = args.path in ("staged", "stream")
        options = binding.make_options(
            path=args.path if args.path in ("rowreg", "twopass", "cluster", "staged", "stream",
                                            "grid") else "auto",
            cluster=args.cluster if args.path in ("cluster", "staged", "twopass", "stream") else 0,
            grid=args.grid, threads=args.threads,
            chunk_bytes=args.chunk if staged else 0, stages=args.stages if staged else 0)
        dt_code = binding.RMSNORM_DTYPE_BF16 if wl.dtype == "bf16" else binding.RMSNORM_DTYPE_F32

        def fwd(xp, wp, yp, r, h, eps, s):
            return binding.raw.rowsoftmax_fwd_ex(dt_code, xp, yp, r, h, options, s)
    elif forced(args):
        options = binding.make_options(path=args.path, cluster=args.cluster, grid=args.grid,
                                       threads=args.threads, chunk_bytes=args.chunk,
                                       stages=args.stages, epilogue=args.epilogue, alpha=0.5)
        dt_code = binding.RMSNORM_DTYPE_BF16 if wl.dtype == "bf16" else binding.RMSNORM_DTYPE_F32

        def fwd(xp, wp, yp, r, h, eps, s):
            return binding.raw.rmsnorm_fwd_ex(dt_code, xp, wp, yp, r, h, eps, options, s)
    else:
        fwd = binding.raw.rmsnorm_fwd_bf16 if wl.dtype == "bf16" else binding.raw.rmsnorm_fwd_f32
    plan = (binding.rowsoftmax_plan(x, y, options=options) if softmax
            else binding.rmsnorm_plan(x, w, y, options=options))
    flush = None
    if wl.bytes_per_call <= 4 * 129e6 and args.l2 == "cold":
        # read-only flush: summing a 258 MB buffer evicts x and y from L2 and
        # leaves only clean lines (a write-based flush would leave ~129 MB of
        # dirty lines whose write-back then competes with the next launch)
        flush = torch.ones(int(2 * 129e6) // 4 + 1024, dtype=torch.float32, device=dev)

    def step():
        st = fwd(x.data_ptr(), w.data_ptr(), y.data_ptr(), rows, hidden, wl.eps, handle)
        if st != 0:
            raise RuntimeError(f"rmsnorm failed: {binding.rmsnorm_status_string(st)}")

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        if flush is not None:
            flush.sum()
        step()
    barrier()

    # Inputs larger than L2: the K launches run back to back and the timed
    # region (one event pair around all of them) is the job's time; the
    # per-launch distribution comes from a separate event-bracketed pass.
    # Inputs that fit L2: a flush before every launch, outside a per-launch
    # event pair, and the job's time is the sum of the launch times.
    back_to_back = flush is None
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        time.sleep(0.3)          # let the sampler start before the timed region
        barrier()
        torch.cuda.nvtx.range_push("timed region")
        t_begin = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_begin.record(stream)
        for i in range(args.steps):
            if back_to_back:
                step()
                continue
            flush.sum()            # outside the per-launch event pair
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        t_end.record(stream)
        torch.cuda.nvtx.range_pop()
        barrier()
    region_ms = t_begin.elapsed_time(t_end)  # whole timed region
    if back_to_back:
        kernel_ms = region_ms                  # device time of the K launches, gaps included
        n_dist = min(args.steps, 50)           # launch-time distribution, outside the region
        for i in range(n_dist):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        per_launch_ms = [s.elapsed_time(e) for s, e in zip(starts[:n_dist], ends[:n_dist])]
    else:
        per_launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        kernel_ms = sum(per_launch_ms)          # device time of the K launches
    if world > 1:
        kernel_ms, region_ms = max_over_ranks([kernel_ms, region_ms], dev)
    ms_per_step = kernel_ms / args.steps
    bytes_step = wl.bytes_per_call
    value, rows_per_s = weak_scaling_rates(world, bytes_step, rows, args.steps, kernel_ms)

    peak, peak_src = peaks()
    avg_launch_s = ms_per_step / 1e3            # average launch duration over the timed region
    achieved = bytes_step / avg_launch_s / 1e9
    per_launch_sorted = sorted(per_launch_ms)
    traffic = profiled_traffic(wl.name, plan["kernel"])

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, wl, x, w, y, fwd, binding, world)

    del x, y
    torch.cuda.empty_cache()
    secondary = None
    names = secondary_names(args) if world == 1 else []
    if names:
        secondary = {}
        with ClockSampler(local) as clocks2:
            time.sleep(0.3)
            for name in names:
                secondary[name] = time_secondary(workloads.WORKLOADS[name], 50, binding,
                                                 workloads, peak, peak_src)
        secondary["clocks"] = clocks2.summary()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_line(wl)

    if rank == 0:
        line = {
            "metric": METRIC_SOFTMAX if softmax else METRIC, "value": value, "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic", "config": config_block(wl, world, args),
            "rows_per_s": rows_per_s,
            "kernel": {"name": plan["kernel"], "path": plan["path_name"],
                       "grid": plan["grid"], "block": plan["block_threads"],
                       "cluster": plan["cluster"], "vec_bytes": plan["vec_bytes"],
                       "vecs_per_thread": plan["vecs_per_thread"],
                       "threads_per_row": plan["threads_per_row"],
                       "timing": ("timed region of back-to-back launches; launch_ms_* from a "
                                  "separate pass of event-bracketed launches" if back_to_back else
                                  "sum of event-bracketed launches, L2 flushed before each"),
                       "launch_ms_median": per_launch_sorted[len(per_launch_sorted) // 2],
                       "launch_ms_p10": per_launch_sorted[len(per_launch_sorted) // 10],
                       "launch_ms_p90": per_launch_sorted[(9 * len(per_launch_sorted)) // 10],
                       "launch_ms_min": per_launch_sorted[0],
                       "launch_ms_max": per_launch_sorted[-1]},
            "roofline": roofline_block(achieved, peak, peak_src, traffic),
            "cpu_baseline": cpu,
            "e2e": e2e,
            "secondary": secondary,
            "gpu_launches": args.steps,
            "timed_region_ms": region_ms,
            "device": device_info(dev),
            "clocks": clocks.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def secondary_names(args):
    """Workloads timed after the main region: by default only on the default
    run (the headline workload, nothing forced, all rows); --secondary
    overrides the list, --secondary none switches it off."""
    if args.secondary is not None:
        return [n for n in args.secondary.split(",") if n and n != "none"]
    if args.workload != "c5a" or args.rows or forced(args):
        return []
    return list(SECONDARY_DEFAULT)


def time_secondary(wl, steps, binding, workloads, peak, peak_src):
    """One secondary workload through its automatic entry point, timed with
    CUDA events on the launching stream.  Inputs larger than 4x L2 run back to
    back (one event pair around all launches); smaller inputs rotate through
    enough copies of x and y (more than 3x L2 in rotation) that every launch
    finds its input and output out of L2, and one event pair times the
    launches back to back (single launches of a few microseconds are below
    the event timer's resolution)."""
    import torch

    softmax = wl.op == "softmax"
    x = workloads.make_x(wl, device="cuda")
    w = torch.empty(0, device="cuda") if softmax else workloads.make_w(wl, device="cuda")
    io_bytes = 2 * x.numel() * x.element_size()
    rotate = wl.bytes_per_call <= 4 * L2_BYTES
    nbuf = int(3.2 * L2_BYTES // io_bytes) + 1 if rotate else 1
    xs = [x] + [x.clone() for _ in range(nbuf - 1)]
    ys = [torch.empty_like(x) for _ in range(nbuf)]
    stream = torch.cuda.current_stream()
    handle = stream.cuda_stream
    bf16 = wl.dtype == "bf16"
    rows, hidden = wl.rows, wl.hidden
    if softmax:
        fn = binding.raw.rowsoftmax_fwd_bf16 if bf16 else binding.raw.rowsoftmax_fwd_f32

        def launch(i):
            return fn(xs[i % nbuf].data_ptr(), ys[i % nbuf].data_ptr(), rows, hidden, handle)
        plan = binding.rowsoftmax_plan(x, ys[0])
    else:
        fn = binding.raw.rmsnorm_fwd_bf16 if bf16 else binding.raw.rmsnorm_fwd_f32

        def launch(i):
            return fn(xs[i % nbuf].data_ptr(), w.data_ptr(), ys[i % nbuf].data_ptr(), rows,
                      hidden, wl.eps, handle)
        plan = binding.rmsnorm_plan(x, w, ys[0])
    n = max(steps, 2 * nbuf) if rotate else steps
    for i in range(max(3, nbuf)):
        st = launch(i)
        if st != 0:
            raise RuntimeError(f"{wl.name}: {binding.rmsnorm_status_string(st)}")
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(n):
        launch(i)
    t1.record(stream)
    torch.cuda.synchronize()
    if binding.rmsnorm_last_device_status() != binding.RMSNORM_OK:
        raise RuntimeError(f"{wl.name}: device status word set")
    ms = t0.elapsed_time(t1) / n
    achieved = wl.bytes_per_call / (ms / 1e3) / 1e9
    del xs, ys, x, w
    torch.cuda.empty_cache()
    return {
        "workload": f"{wl.name}: {wl.description}", "shape": list(wl.shape),
        "io_dtype": wl.dtype, "op": wl.op, "bytes_per_launch": wl.bytes_per_call,
        "ms_per_launch": ms, "value": achieved, "unit": "GB/s",
        "rows_per_s": rows / (ms / 1e3), "launches": n,
        "kernel": {"name": plan["kernel"], "grid": plan["grid"], "block": plan["block_threads"],
                   "cluster": plan["cluster"]},
        "timing": (f"{n} launches back to back rotating over {nbuf} copies of x and y "
                   f"({nbuf * io_bytes / 1e6:.0f} MB, more than 3x L2), one event pair"
                   if rotate else f"{n} launches back to back (inputs larger than L2), "
                                  "one event pair"),
        "roofline": roofline_block(achieved, peak, peak_src,
                                   profiled_traffic(wl.name, plan["kernel"])),
    }


def measure_e2e(args, wl, x_dev, w_dev, y_dev, fwd, binding, world):
    """Same metric end to end: pinned host x,w -> device, the C-ABI call, device
    y -> pinned host, every step.  The row range is split into 32 chunks run
    on three streams so that copies in both directions overlap each other and
    the kernel (measured on GB300: host<->device copies run at about 200 GB/s
    each way and 343 GB/s both ways at once, so this number is bound by the
    host link, not by the kernel; 32 chunks on 3 streams came within 4% of
    the two-way link, 16 on 2 within 8%)."""
    import torch

    dt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    x_h = torch.empty(wl.shape, dtype=dt, pin_memory=True)
    x_h.copy_(x_dev.cpu())
    w_h = w_dev.cpu().pin_memory()
    w_bytes = w_dev.numel() * wl.elem_bytes
    y_h = torch.empty(wl.shape, dtype=dt, pin_memory=True)
    rows, hidden = wl.rows, wl.hidden
    xh2, yh2 = x_h.view(rows, hidden), y_h.view(rows, hidden)
    xd2, yd2 = x_dev.view(rows, hidden), y_dev.view(rows, hidden)
    nchunks = 32 if rows >= 32 else 1
    bounds = [rows * i // nchunks for i in range(nchunks + 1)]
    streams = [torch.cuda.Stream() for _ in range(3)]
    launches = [0]

    def step():
        ev_w = torch.cuda.Event()
        s0 = streams[0]
        with torch.cuda.stream(s0):
            if w_dev.numel():
                w_dev.copy_(w_h, non_blocking=True)
            ev_w.record(s0)
        for i in range(nchunks):
            s = streams[i % len(streams)]
            a, b = bounds[i], bounds[i + 1]
            with torch.cuda.stream(s):
                s.wait_event(ev_w)
                xd2[a:b].copy_(xh2[a:b], non_blocking=True)
                st = fwd(xd2[a:b].data_ptr(), w_dev.data_ptr(), yd2[a:b].data_ptr(),
                         b - a, hidden, wl.eps, s.cuda_stream)
                if st != 0:
                    raise RuntimeError(binding.rmsnorm_status_string(st))
                launches[0] += 1
                yh2[a:b].copy_(yd2[a:b], non_blocking=True)
        for s in streams:
            s.synchronize()

    for _ in range(max(3, min(args.warmup, 5))):
        step()
    torch.cuda.synchronize()
    n = max(3, min(args.steps, 10))
    launches[0] = 0
    t0 = time.perf_counter()
    for _ in range(n):
        step()
    dt_s = time.perf_counter() - t0
    if world > 1:
        dt_s = max_over_ranks([dt_s], x_dev.device)[0]
    # check the round trip landed (cheap spot check of one row against the device)
    if not torch.equal(yh2[-1].to(y_dev.device), yd2[-1]):
        raise RuntimeError("end-to-end copy-back mismatch")
    return {"value": world * wl.bytes_per_call * n / dt_s / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": rows * hidden * wl.elem_bytes + w_bytes,
            "d2h_bytes_per_step": rows * hidden * wl.elem_bytes,
            "steps": n, "ms_per_step": 1e3 * dt_s / n, "chunks_per_step": nchunks,
            "streams": len(streams), "gpu_launches": launches[0], "timing": "host wall clock"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="c5a")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--rows", type=int, default=0,
                    help="use only this many rows of the workload (small profiling cases)")
    ap.add_argument("--path", default="auto",
                    choices=["auto", "rowreg", "staged", "cluster", "twopass", "page", "ringreg",
                             "stream", "grid"],
                    help="force a kernel family through rmsnorm_fwd_ex (evidence runs)")
    ap.add_argument("--cluster", type=int, default=0)
    ap.add_argument("--grid", type=int, default=0, help="force the CTA count")
    ap.add_argument("--threads", type=int, default=0, help="force threads per row group")
    ap.add_argument("--chunk", type=int, default=0, help="staged path: bytes per bulk copy")
    ap.add_argument("--stages", type=int, default=0, help="staged path: ring slots")
    ap.add_argument("--epilogue", default="none", choices=["none", "scale", "relu"],
                    help="fused epilogue (measures its cost; default none)")
    ap.add_argument("--l2", default="cold", choices=["cold", "hot"],
                    help="cold (default): read a 258 MB buffer between steps of workloads "
                         "that fit L2; hot: no flush, for the L2-resident figure")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--secondary", default=None,
                    help="comma-separated workloads timed after the main region (default: "
                         + ",".join(SECONDARY_DEFAULT) + " on the default run; 'none' = off)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    import dataclasses
    from row_wise_rmsnorm_fwd_gb300 import workloads
    wl = workloads.WORKLOADS[args.workload]
    if args.rows:
        wl = dataclasses.replace(wl, name=f"{wl.name}_rows{args.rows}",
                                 shape=(args.rows, wl.hidden),
                                 description=f"first {args.rows} rows of {wl.description}")
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
