"""Measure the register-resident kernel's compile-time policies on this GPU.

    python -m row_wise_rmsnorm_fwd_gb300.tune [--variants base,nopf,...]
                                              [--workloads c4,c5a] [--out FILE]

The row kernel has four compile-time policies (``rowreg_instances.cuh``):
register prefetch of the next row (PF), weights held in registers (WREG), the
cache policy of the x loads (LD) and of the y stores (ST).  This builds one
library per variant from the same sources (``_build/tune/``), then times every
variant on each workload for a few grid sizes (the automatic one among them),
interleaving variants and
repeating three times (median), and prints one JSON line per (variant,
workload, grid).  The product library keeps the defaults this measured best.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import ctypes
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from row_wise_rmsnorm_fwd_gb300 import build as B  # noqa: E402

VARIANTS = {
    "base": {},                      # the product defaults (PF 1, WREG 1, LD 0, ST 0)
    "nopf": {"PF": 0},               # no register prefetch of the next row
    "nowreg": {"WREG": 0},           # weights re-read from L1 every row
    "ld_nc_l2_256": {"LD": 1},       # ld.global.nc.L1::no_allocate.L2::256B
    "ld_nc": {"LD": 2},              # ld.global.nc.L1::no_allocate
    "ld_evict_first": {"LD": 3},     # ld.global.L1::no_allocate + L2 evict-first policy
    "st_plain": {"ST": 1},           # st.global
    "st_no_allocate": {"ST": 2},     # st.global.L1::no_allocate
}
OUT_DIR = os.path.join(B.BUILD_DIR, "tune")


def build_variants(names):
    nvcc = B._nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    srcs = B.sources()
    common = [s for s in srcs if not os.path.basename(s).startswith("rowreg_")]
    rowreg = [s for s in srcs if os.path.basename(s).startswith("rowreg_")]
    jobs = [(s, os.path.join(OUT_DIR, "common_" + os.path.basename(s) + ".o"), [])
            for s in common]
    for n in names:
        defines = [f"-DRMSNORM_ROWREG_{k}={v}" for k, v in VARIANTS[n].items()]
        jobs += [(s, os.path.join(OUT_DIR, f"{n}_" + os.path.basename(s) + ".o"), defines)
                 for s in rowreg]

    def compile_one(job):
        src, obj, defines = job
        r = subprocess.run([nvcc, *B.ARCH_FLAGS, *B.NVCC_FLAGS, *defines, "-c", src, "-o", obj],
                           capture_output=True, text=True)
        if r.returncode:
            raise RuntimeError(r.stderr)

    with cf.ThreadPoolExecutor(os.cpu_count() or 1) as ex:
        list(ex.map(compile_one, jobs))
    libs = {}
    for n in names:
        objs = [os.path.join(OUT_DIR, "common_" + os.path.basename(s) + ".o") for s in common]
        objs += [os.path.join(OUT_DIR, f"{n}_" + os.path.basename(s) + ".o") for s in rowreg]
        lib = os.path.join(OUT_DIR, f"librmsnorm_{n}.so")
        subprocess.run([nvcc, *B.ARCH_FLAGS, "-shared", "-cudart", "static", "-o", lib, *objs],
                       check=True)
        libs[n] = lib
    return libs


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--variants", default=",".join(VARIANTS))
    ap.add_argument("--workloads", default="c4,c5a")
    ap.add_argument("--grids", default="0,9728,29184,86944",
                    help="CTA counts to time (0 = the library's automatic grid)")
    ap.add_argument("--iters", type=int, default=30)
    ap.add_argument("--out", default="")
    args = ap.parse_args()
    names = args.variants.split(",")
    libs = build_variants(names)

    import torch
    from row_wise_rmsnorm_fwd_gb300 import binding, workloads

    lines = []
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    for wname in args.workloads.split(","):
        wl = workloads.WORKLOADS[wname]
        x = workloads.make_x(wl, device="cuda").reshape(-1, wl.hidden)
        w = workloads.make_w(wl, device="cuda")
        y = torch.empty_like(x)
        dt = binding.RMSNORM_DTYPE_F32 if wl.dtype == "f32" else binding.RMSNORM_DTYPE_BF16
        handle = torch.cuda.current_stream().cuda_stream
        auto_grid = binding.rmsnorm_plan(x, w, y, options={"path": "rowreg"})["grid"]
        grids = [int(g) or auto_grid for g in args.grids.split(",")]
        times = {}
        for _ in range(3):
            for n in names:
                lib = binding.open_library(libs[n])
                for g in grids:
                    o = binding.make_options(path="rowreg", grid=g)
                    call = lambda: lib.rmsnorm_fwd_ex(dt, x.data_ptr(), w.data_ptr(),  # noqa
                                                      y.data_ptr(), wl.rows, wl.hidden, wl.eps,
                                                      ctypes.byref(o), handle)
                    for _ in range(3):
                        assert call() == 0
                    a, b = ev(), ev()
                    a.record()
                    for _ in range(args.iters):
                        call()
                    b.record()
                    torch.cuda.synchronize()
                    times.setdefault((n, g), []).append(a.elapsed_time(b) / args.iters)
        for (n, g), v in sorted(times.items(), key=lambda kv: sorted(kv[1])[1]):
            ms = sorted(v)[1]
            rec = {"workload": wname, "variant": n, "defines": VARIANTS[n], "grid": g,
                   "ms": ms, "gbs": wl.bytes_per_call / ms / 1e6}
            lines.append(rec)
            print(json.dumps(rec), flush=True)
        del x, y
        torch.cuda.empty_cache()
    if args.out:
        with open(args.out, "w") as f:
            for r in lines:
                f.write(json.dumps(r) + "\n")


if __name__ == "__main__":
    main()
