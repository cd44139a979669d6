"""Build librmsnorm.so in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel into
``row_wise_rmsnorm_fwd_gb300/_build/``, then linked into one shared library
with the CUDA runtime linked statically.  A second library,
``librmsnorm_faultinject.so``, is the same sources compiled with
``-DRMSNORM_FAULT_INJECT=1``: only the failure-detection tests load it (it
honours ``rmsnorm_options_t.fault_inject``; the product library refuses it).
``python -m row_wise_rmsnorm_fwd_gb300.build [--force] [--ptxas-verbose]``
runs the build by hand.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "librmsnorm.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
FAULT_LIB_PATH = os.path.join(BUILD_DIR, "librmsnorm_faultinject.so")
VARIANTS = {LIB_PATH: [], FAULT_LIB_PATH: ["-DRMSNORM_FAULT_INJECT=1"]}

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-Wall", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"),
                 "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librmsnorm")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list[str]:
    return sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        sorted(glob.glob(os.path.join(CSRC, "*.h"))) + \
        sorted(glob.glob(os.path.join(INCLUDE, "*.h"))) + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    for lib in VARIANTS:
        if not os.path.exists(lib):
            return False
        t = os.path.getmtime(lib)
        if any(os.path.getmtime(d) > t for d in _deps()):
            return False
    return True


def _compile(nvcc: str, src: str, obj: str, defines: list, verbose_ptxas: bool):
    cmd = [nvcc, *ARCH_FLAGS, *NVCC_FLAGS, *defines, "-c", src, "-o", obj]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(force: bool = False, verbose_ptxas: bool = False, quiet: bool = True) -> str:
    """Compile and link librmsnorm.so (and its fault-injection test twin);
    returns the product library's path."""
    if not force and not verbose_ptxas and up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    for lib, defines in VARIANTS.items():
        sub = os.path.join(BUILD_DIR, "obj_" + os.path.basename(lib)[:-3])
        os.makedirs(sub, exist_ok=True)
        for src in sources():
            obj = os.path.join(sub, os.path.basename(src)[:-3] + ".o")
            jobs.append((lib, src, obj, defines))
    workers = max(1, min(len(jobs), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        logs = list(ex.map(lambda j: _compile(nvcc, j[1], j[2], j[3],
                                              verbose_ptxas and j[0] == LIB_PATH), jobs))
    for lib in VARIANTS:
        objs = [j[2] for j in jobs if j[0] == lib]
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH_FLAGS, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    if verbose_ptxas:
        with open(os.path.join(BUILD_DIR, "ptxas.log"), "w") as f:
            f.write("\n".join(logs))
    if not quiet:
        print(f"built {LIB_PATH} and {FAULT_LIB_PATH}")
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="--ptxas-verbose" in sys.argv,
          quiet=False)
