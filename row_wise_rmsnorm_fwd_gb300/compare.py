"""Side-by-side timing of librmsnorm against the write-up's comparison axes.

    python -m row_wise_rmsnorm_fwd_gb300.compare [--workloads c1,c2,c3,c4,c5a]
                                                 [--iters 50] [--out FILE]

The compiler write-up measures its generated kernels against PyTorch eager and
torch.compile.  This runs, on the same GPU and inputs, for each workload
(row-softmax workloads compare ours with torch.softmax eager and compiled):
  - ``ours``: librmsnorm's automatic choice (rmsnorm_fwd_f32 / _bf16),
  - ``page``: librmsnorm's rebuild of the write-up's own kernel schedule
    (RMSNORM_PATH_PAGE: one CTA per row, smem staging, scalar accesses),
  - ``eager``: torch.nn.functional.rms_norm,
  - ``compile``: torch.compile of the same call (if it compiles here).
Timing: CUDA events around each call on the current stream after warm-up;
workloads smaller than 4x L2 are preceded by a read of a 258 MB buffer
(outside the events) so every call reads its inputs from HBM with no dirty
lines left in L2.  GB/s counts algorithmic bytes (x read,
y written, w read once).  One JSON line per (workload, implementation).
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from row_wise_rmsnorm_fwd_gb300 import binding, build, workloads  # noqa: E402

L2_BYTES = 129e6


def _timed(fn, iters: int, flush):
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    times = []
    s = torch.cuda.current_stream()
    for _ in range(iters):
        if flush is not None:
            flush.sum()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s)
        fn()
        b.record(s)
        times.append((a, b))
    torch.cuda.synchronize()
    ms = sorted(a.elapsed_time(b) for a, b in times)
    return ms[len(ms) // 2]


def run(names, iters: int):
    build.build()
    binding.load()
    rows_out = []
    for name in names:
        wl = workloads.WORKLOADS[name]
        dev = "cuda"
        x = workloads.make_x(wl, device=dev).reshape(-1, wl.hidden)
        softmax = wl.op == "softmax"
        w = None if softmax else workloads.make_w(wl, device=dev)
        y = torch.empty_like(x)
        flush = None
        if wl.bytes_per_call <= 4 * L2_BYTES:
            flush = torch.ones(int(2 * L2_BYTES) // 4, dtype=torch.float32, device=dev)
        eps = wl.eps
        H = wl.hidden

        def ours():
            if softmax:
                binding.rowsoftmax_fwd_ex(x, y)
            else:
                binding.rmsnorm_fwd_ex(x, w, y, eps)

        def page():
            binding.rmsnorm_fwd_ex(x, w, y, eps, options={"path": "page"})

        def eager():
            if softmax:
                return torch.softmax(x, -1)
            return torch.nn.functional.rms_norm(x, (H,), w, eps)

        impls = [("ours", ours), ("eager", eager)] if softmax else \
            [("ours", ours), ("page", page), ("eager", eager)]
        try:
            compiled = torch.compile(
                (lambda t: torch.softmax(t, -1)) if softmax
                else (lambda t: torch.nn.functional.rms_norm(t, (H,), w, eps)))
            compiled(x)
            impls.append(("compile", lambda: compiled(x)))
        except Exception as e:  # noqa: BLE001 -- report, do not fail the comparison
            rows_out.append({"workload": name, "impl": "compile",
                             "unavailable": f"{type(e).__name__}: {str(e)[:200]}"})
        for impl, fn in impls:
            try:
                ms = _timed(fn, iters, flush)
            except binding.RmsnormError as e:
                rows_out.append({"workload": name, "impl": impl, "unavailable": str(e)})
                continue
            rec = {"workload": name, "impl": impl, "shape": list(wl.shape), "dtype": wl.dtype,
                   "us": ms * 1e3, "gbs": wl.bytes_per_call / (ms * 1e-3) / 1e9,
                   "rows_per_s": wl.rows / (ms * 1e-3),
                   "l2": "flushed" if flush is not None else "inputs larger than L2"}
            rows_out.append(rec)
            print(json.dumps(rec), flush=True)
        del x, y
        torch.cuda.empty_cache()
    return rows_out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workloads", default="c1,c2,c2t,c3,c4,c5a")
    ap.add_argument("--iters", type=int, default=50)
    ap.add_argument("--out", default="")
    args = ap.parse_args()
    rows = run(args.workloads.split(","), args.iters)
    if args.out:
        with open(args.out, "w") as f:
            for r in rows:
                f.write(json.dumps(r) + "\n")


if __name__ == "__main__":
    main()
