"""CPU oracle for the row-wise RMSNorm forward pass (and row-wise softmax).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py`` may import this package.  The CUDA library
never imports, links or calls it, and it imports nothing from the CUDA side.

The arithmetic lives in ``rmsnorm_oracle.c`` (plain C, binary64 throughout,
compiled with ``gcc -O2`` and no fast-math); this module only compiles it and
marshals numpy arrays through ctypes.

Definition followed (page "A hackable Python ML compiler, part 2", the
RMSNorm Loop-IR listing and the generated kernel's epilogue):
``y[r,j] = (x[r,j] * (1/sqrt(mean_j x[r,j]^2 + eps))) * w[j]``.

Every function here is pinned by ``tests/test_oracle_pins.py`` against hand
evaluations, closed forms, invariants, an independent library routine and an
exhaustive bfloat16 search; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rmsnorm_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "rowsoftmax_oracle.c")]
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_rmsnorm.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/liboracle_rmsnorm.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(s) for s in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-Wall", "-Wextra", "-o", tmp, *_SRCS, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, dbl = ctypes.c_int64, ctypes.c_double
        vp = ctypes.c_void_p
        lib.oracle_rmsnorm_f64.argtypes = [vp, vp, vp, i64, i64, dbl]
        lib.oracle_rmsnorm_f32.argtypes = [vp, vp, vp, i64, i64, dbl]
        lib.oracle_rmsnorm_bf16.argtypes = [vp, vp, vp, vp, i64, i64, dbl]
        lib.oracle_rmsnorm_stats_f64.argtypes = [vp, vp, vp, i64, i64, dbl]
        lib.oracle_apply_epilogue_f64.argtypes = [vp, i64, ctypes.c_int, dbl]
        lib.oracle_rowsoftmax_f64.argtypes = [vp, vp, i64, i64]
        lib.oracle_rowsoftmax_f32.argtypes = [vp, vp, i64, i64]
        lib.oracle_rowsoftmax_bf16.argtypes = [vp, vp, vp, i64, i64]
        for f in ("oracle_rowsoftmax_f64", "oracle_rowsoftmax_f32", "oracle_rowsoftmax_bf16"):
            getattr(lib, f).restype = ctypes.c_int
        lib.oracle_f64_to_bf16_array.argtypes = [vp, vp, i64]
        for f in ("oracle_rmsnorm_f64", "oracle_rmsnorm_f32",
                  "oracle_rmsnorm_bf16", "oracle_rmsnorm_stats_f64",
                  "oracle_apply_epilogue_f64", "oracle_f64_to_bf16_array"):
            getattr(lib, f).restype = ctypes.c_int
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_bf16_rne.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16_rne.restype = ctypes.c_uint16
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _as2d(x: np.ndarray, w: np.ndarray):
    if x.ndim < 1:
        raise ValueError("x needs at least one dimension")
    hidden = x.shape[-1]
    if w.shape != (hidden,):
        raise ValueError(f"w has shape {w.shape}, expected ({hidden},)")
    rows = int(np.prod(x.shape[:-1], dtype=np.int64)) if x.ndim > 1 else 1
    return rows, hidden


def _out(out, shape, dtype):
    """A caller-supplied output buffer (reused across calls, so that host
    threads running the oracle side by side do not all fault in fresh pages),
    else a new one."""
    if out is None:
        return np.empty(shape, dtype=dtype)
    if out.shape != tuple(shape) or out.dtype != dtype or not out.flags.c_contiguous:
        raise ValueError(f"output buffer must be a contiguous {dtype} array of shape {shape}")
    return out


def _check(status: int):
    if status != 0:
        raise ValueError(f"oracle rejected the arguments (status {status})")


def rmsnorm_f64(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """binary64 in, binary64 out.  Leading dims of ``x`` are rows."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    rows, hidden = _as2d(x, w)
    y = np.empty_like(x)
    _check(_load().oracle_rmsnorm_f64(_ptr(x), _ptr(w), _ptr(y), rows,
                                      hidden, float(eps)))
    return y


def rmsnorm_f32(x: np.ndarray, w: np.ndarray, eps: float, out=None) -> np.ndarray:
    """binary32 inputs (widened exactly), binary64 result of the same shape
    (written into ``out`` when given)."""
    x = np.ascontiguousarray(x)
    w = np.ascontiguousarray(w)
    if x.dtype != np.float32 or w.dtype != np.float32:
        raise TypeError("rmsnorm_f32 takes float32 arrays")
    rows, hidden = _as2d(x, w)
    y = _out(out, x.shape, np.float64)
    _check(_load().oracle_rmsnorm_f32(_ptr(x), _ptr(w), _ptr(y), rows,
                                      hidden, float(eps)))
    return y


def rmsnorm_bf16(x_bits: np.ndarray, w_bits: np.ndarray, eps: float,
                 out64=None, out16=None):
    """bfloat16 bit patterns (uint16) in.

    Returns ``(y64, y16)``: the binary64 result and its single
    round-to-nearest-even rounding to bfloat16 bits (written into ``out64``
    and ``out16`` when given).
    """
    x_bits = np.ascontiguousarray(x_bits)
    w_bits = np.ascontiguousarray(w_bits)
    if x_bits.dtype != np.uint16 or w_bits.dtype != np.uint16:
        raise TypeError("rmsnorm_bf16 takes uint16 bit patterns")
    rows, hidden = _as2d(x_bits, w_bits)
    y64 = _out(out64, x_bits.shape, np.float64)
    y16 = _out(out16, x_bits.shape, np.uint16)
    _check(_load().oracle_rmsnorm_bf16(_ptr(x_bits), _ptr(w_bits), _ptr(y64),
                                       _ptr(y16), rows, hidden, float(eps)))
    return y64, y16


def rmsnorm_stats_f64(x: np.ndarray, eps: float):
    """Per-row (mean of squares, 1/sqrt(mean + eps)) in binary64."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    hidden = x.shape[-1]
    rows = int(np.prod(x.shape[:-1], dtype=np.int64)) if x.ndim > 1 else 1
    ms = np.empty(rows, dtype=np.float64)
    rstd = np.empty(rows, dtype=np.float64)
    _check(_load().oracle_rmsnorm_stats_f64(_ptr(x), _ptr(ms), _ptr(rstd),
                                            rows, hidden, float(eps)))
    return ms, rstd


EPILOGUES = {"none": 0, "scale": 1, "relu": 2}


def apply_epilogue(y: np.ndarray, kind, alpha: float = 1.0) -> np.ndarray:
    """The fused epilogue on binary64 outputs (copy): none, scale by alpha, or
    ReLU (NaN kept, non-positive values become +0)."""
    k = EPILOGUES[kind] if isinstance(kind, str) else int(kind)
    out = np.array(y, dtype=np.float64, copy=True, order="C")
    _check(_load().oracle_apply_epilogue_f64(_ptr(out), out.size, k, float(alpha)))
    return out


def f64_to_bf16_fast(values) -> np.ndarray:
    """Vectorised binary64 -> bfloat16 bits (one RNE rounding per element)."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _check(_load().oracle_f64_to_bf16_array(_ptr(v), _ptr(out), v.size))
    return out


def rmsnorm_epilogue_f32(x: np.ndarray, w: np.ndarray, eps: float, kind, alpha=1.0):
    """fp32 inputs; RMSNorm then the epilogue, all in binary64."""
    return apply_epilogue(rmsnorm_f32(x, w, eps), kind, alpha)


def rmsnorm_epilogue_bf16(x_bits, w_bits, eps: float, kind, alpha=1.0):
    """bf16 inputs; RMSNorm and the epilogue in binary64, then ONE rounding.
    Returns (y64, y16)."""
    y64, _ = rmsnorm_bf16(x_bits, w_bits, eps)
    e64 = apply_epilogue(y64, kind, alpha)
    return e64, f64_to_bf16_fast(e64)


# ------------------------------------------------------------ row softmax --
# Plain definition (the write-up names softmax-style small reductions but
# prints no formula): y = exp(x - max) / sum exp(x - max) per row, binary64.

def _rows_cols(x: np.ndarray):
    if x.ndim < 1 or x.shape[-1] == 0:
        raise ValueError("x needs a non-empty last dimension")
    cols = x.shape[-1]
    rows = int(np.prod(x.shape[:-1], dtype=np.int64)) if x.ndim > 1 else 1
    return rows, cols


def rowsoftmax_f64(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    rows, cols = _rows_cols(x)
    y = np.empty_like(x)
    _check(_load().oracle_rowsoftmax_f64(_ptr(x), _ptr(y), rows, cols))
    return y


def rowsoftmax_f32(x: np.ndarray, out=None) -> np.ndarray:
    """binary32 input (widened exactly), binary64 result (into ``out`` when given)."""
    x = np.ascontiguousarray(x)
    if x.dtype != np.float32:
        raise TypeError("rowsoftmax_f32 takes float32")
    rows, cols = _rows_cols(x)
    y = _out(out, x.shape, np.float64)
    _check(_load().oracle_rowsoftmax_f32(_ptr(x), _ptr(y), rows, cols))
    return y


def rowsoftmax_bf16(x_bits: np.ndarray, out64=None, out16=None):
    """bfloat16 bits in; returns (y64, y16) with y16 the single RNE rounding
    (written into ``out64`` and ``out16`` when given)."""
    x_bits = np.ascontiguousarray(x_bits)
    if x_bits.dtype != np.uint16:
        raise TypeError("rowsoftmax_bf16 takes uint16 bit patterns")
    rows, cols = _rows_cols(x_bits)
    y64 = _out(out64, x_bits.shape, np.float64)
    y16 = _out(out16, x_bits.shape, np.uint16)
    _check(_load().oracle_rowsoftmax_bf16(_ptr(x_bits), _ptr(y64), _ptr(y16), rows, cols))
    return y64, y16


def bf16_to_f64(bits) -> np.ndarray:
    """Exact decode of bfloat16 bit patterns."""
    lib = _load()
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return np.array([lib.oracle_bf16_to_f64(int(v)) for v in b.ravel()],
                    dtype=np.float64).reshape(b.shape)


def f64_to_bf16(values) -> np.ndarray:
    """binary64 -> bfloat16 bits, one round-to-nearest-even rounding."""
    lib = _load()
    v = np.ascontiguousarray(values, dtype=np.float64)
    return np.array([lib.oracle_f64_to_bf16_rne(float(t)) for t in v.ravel()],
                    dtype=np.uint16).reshape(v.shape)
