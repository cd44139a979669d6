"""ctypes binding of librmsnorm's C ABI (``include/rmsnorm.h``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``librmsnorm.so``.  Functions carry the C names.  Tensor-level
functions take torch CUDA tensors (torch supplies device memory and the
current stream); the ``raw`` namespace takes plain integers (device pointers
and a ``cudaStream_t`` handle) and returns the C status code.

If the library has not been built this module raises on first use: there is
no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from types import SimpleNamespace

from . import build as _build

RMSNORM_OK = 0
RMSNORM_ERR_INVALID_ARG = 1
RMSNORM_ERR_UNSUPPORTED = 2
RMSNORM_ERR_CUDA = 3
RMSNORM_ERR_TIMEOUT = 4

RMSNORM_DTYPE_F32 = 0
RMSNORM_DTYPE_BF16 = 1

PATHS = {"auto": 0, "rowreg": 1, "staged": 2, "cluster": 3, "twopass": 4, "page": 5,
         "ringreg": 6, "stream": 7, "grid": 8}
PATH_NAMES = {v: k for k, v in PATHS.items()}


class rmsnorm_options_t(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("cluster", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("vec_bytes", ctypes.c_int32), ("chunk_bytes", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("weights", ctypes.c_int32),
                ("fault_inject", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("epilogue", ctypes.c_int32), ("epilogue_alpha", ctypes.c_float),
                ("wait_timeout_ns", ctypes.c_uint64)]


class rmsnorm_plan_t(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("cluster", ctypes.c_int32),
                ("threads_per_row", ctypes.c_int32), ("block_threads", ctypes.c_int32),
                ("rows_per_cta", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("vec_bytes", ctypes.c_int32), ("vecs_per_thread", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("chunk_bytes", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("weights_staged", ctypes.c_int32),
                ("kernel", ctypes.c_char * 48)]


class RmsnormError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        detail = ""
        if status == RMSNORM_ERR_CUDA:
            code, text = rmsnorm_last_cuda_error()
            detail = f" [{text}]" if code else ""
        super().__init__(f"{what}: {rmsnorm_status_string(status)} (status {status}){detail}")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def open_library(path: str):
    """dlopen a build of librmsnorm at `path` and declare its C signatures."""
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with row_wise_rmsnorm_fwd_gb300.build.build() "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    for name in ("rmsnorm_fwd_f32", "rmsnorm_fwd_bf16"):
        fn = getattr(lib, name)
        fn.argtypes = [vp, vp, vp, i64, i64, f32, vp]
        fn.restype = ctypes.c_int
    lib.rmsnorm_fwd_ex.argtypes = [i32, vp, vp, vp, i64, i64, f32,
                                   ctypes.POINTER(rmsnorm_options_t), vp]
    lib.rmsnorm_fwd_ex.restype = ctypes.c_int
    lib.rmsnorm_fwd_grid_noalloc.argtypes = [i32, vp, vp, vp, i64, i64, f32, vp]
    lib.rmsnorm_fwd_grid_noalloc.restype = ctypes.c_int
    lib.rmsnorm_plan.argtypes = [i32, vp, vp, vp, i64, i64,
                                 ctypes.POINTER(rmsnorm_options_t),
                                 ctypes.POINTER(rmsnorm_plan_t)]
    lib.rmsnorm_plan.restype = ctypes.c_int
    lib.rmsnorm_last_device_status.argtypes = [vp]
    lib.rmsnorm_last_device_status.restype = ctypes.c_int
    lib.rmsnorm_status_string.argtypes = [ctypes.c_int]
    lib.rmsnorm_status_string.restype = ctypes.c_char_p
    lib.rmsnorm_last_cuda_error.argtypes = [ctypes.c_char_p, ctypes.c_size_t]
    lib.rmsnorm_last_cuda_error.restype = ctypes.c_int32
    lib.rmsnorm_fault_injection_enabled.argtypes = []
    lib.rmsnorm_fault_injection_enabled.restype = ctypes.c_int32
    lib.rmsnorm_abi_version.argtypes = []
    lib.rmsnorm_abi_version.restype = ctypes.c_int32
    for name in ("rowsoftmax_fwd_f32", "rowsoftmax_fwd_bf16"):
        fn = getattr(lib, name)
        fn.argtypes = [vp, vp, i64, i64, vp]
        fn.restype = ctypes.c_int
    lib.rowsoftmax_fwd_ex.argtypes = [i32, vp, vp, i64, i64, ctypes.POINTER(rmsnorm_options_t),
                                      vp]
    lib.rowsoftmax_fwd_ex.restype = ctypes.c_int
    lib.rowsoftmax_plan.argtypes = [i32, vp, vp, i64, i64, ctypes.POINTER(rmsnorm_options_t),
                                    ctypes.POINTER(rmsnorm_plan_t)]
    lib.rowsoftmax_plan.restype = ctypes.c_int
    return lib


def load():
    """Load librmsnorm.so (built in-tree by ``build.build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = open_library(library_path())
        return _lib


def declared_functions() -> list[str]:
    """Names of the functions declared in include/*.h (for export checks)."""
    names = []
    inc = os.path.join(_build.ROOT, "include")
    for fname in sorted(os.listdir(inc)):
        if not fname.endswith(".h"):
            continue
        text = open(os.path.join(inc, fname)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b((?:rmsnorm|rowsoftmax)_[a-z0-9_]+)\s*\(", text):
            if m.group(1) not in names:
                names.append(m.group(1))
    return names


WEIGHTS = {"auto": 0, "smem": 1, "l2": 2}
EPILOGUES = {"none": 0, "scale": 1, "relu": 2}


def make_options(path="auto", cluster=0, threads=0, grid=0, vec_bytes=0,
                 chunk_bytes=0, stages=0, weights=0, wait_timeout_ns=0,
                 fault_inject=0, epilogue=0, alpha=1.0) -> rmsnorm_options_t:
    o = rmsnorm_options_t()
    o.path = PATHS[path] if isinstance(path, str) else int(path)
    o.cluster, o.threads, o.grid = int(cluster), int(threads), int(grid)
    o.vec_bytes, o.chunk_bytes = int(vec_bytes), int(chunk_bytes)
    o.stages = int(stages)
    o.weights = WEIGHTS[weights] if isinstance(weights, str) else int(weights)
    o.fault_inject = int(fault_inject)
    o.epilogue = EPILOGUES[epilogue] if isinstance(epilogue, str) else int(epilogue)
    o.epilogue_alpha = float(alpha)
    o.wait_timeout_ns = int(wait_timeout_ns)
    return o


# ------------------------------------------------------------ raw pointers --

def _raw_fwd_f32(x, w, y, rows, hidden, eps, stream=0) -> int:
    return load().rmsnorm_fwd_f32(x, w, y, rows, hidden, eps, stream or None)


def _raw_fwd_bf16(x, w, y, rows, hidden, eps, stream=0) -> int:
    return load().rmsnorm_fwd_bf16(x, w, y, rows, hidden, eps, stream or None)


def _raw_fwd_ex(dtype, x, w, y, rows, hidden, eps, options=None, stream=0) -> int:
    opt = ctypes.byref(options) if options is not None else None
    return load().rmsnorm_fwd_ex(dtype, x, w, y, rows, hidden, eps, opt, stream or None)


def _raw_plan(dtype, x, w, y, rows, hidden, options=None):
    plan = rmsnorm_plan_t()
    opt = ctypes.byref(options) if options is not None else None
    st = load().rmsnorm_plan(dtype, x, w, y, rows, hidden, opt, ctypes.byref(plan))
    return st, plan


def _raw_sm_f32(x, y, rows, cols, stream=0) -> int:
    return load().rowsoftmax_fwd_f32(x, y, rows, cols, stream or None)


def _raw_sm_bf16(x, y, rows, cols, stream=0) -> int:
    return load().rowsoftmax_fwd_bf16(x, y, rows, cols, stream or None)


def _raw_sm_ex(dtype, x, y, rows, cols, options=None, stream=0) -> int:
    opt = ctypes.byref(options) if options is not None else None
    return load().rowsoftmax_fwd_ex(dtype, x, y, rows, cols, opt, stream or None)


raw = SimpleNamespace(rmsnorm_fwd_f32=_raw_fwd_f32, rmsnorm_fwd_bf16=_raw_fwd_bf16,
                      rmsnorm_fwd_ex=_raw_fwd_ex, rmsnorm_plan=_raw_plan,
                      rowsoftmax_fwd_f32=_raw_sm_f32, rowsoftmax_fwd_bf16=_raw_sm_bf16,
                      rowsoftmax_fwd_ex=_raw_sm_ex)


# ------------------------------------------------------------------ tensors --

def _torch():
    import torch
    return torch


def _stream_handle(stream) -> int:
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check_tensors(x, w, y, dtype):
    torch = _torch()
    want = torch.float32 if dtype == RMSNORM_DTYPE_F32 else torch.bfloat16
    for name, t in (("x", x), ("w", w), ("y", y)):
        if t.dtype != want:
            raise TypeError(f"{name} must be {want}, got {t.dtype}")
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    hidden = x.shape[-1] if x.dim() > 0 else 0
    if w.dim() != 1 or w.shape[0] != hidden:
        raise ValueError(f"w must have shape ({hidden},), got {tuple(w.shape)}")
    if y.shape != x.shape:
        raise ValueError(f"y must have the shape of x {tuple(x.shape)}, got {tuple(y.shape)}")
    rows = x.numel() // hidden if hidden else 0
    return rows, hidden


def _fwd(dtype, x, w, y, eps, options, stream):
    if y is None:
        y = _torch().empty_like(x)
    rows, hidden = _check_tensors(x, w, y, dtype)
    st = _raw_fwd_ex(dtype, x.data_ptr(), w.data_ptr(), y.data_ptr(), rows, hidden,
                     float(eps), options, _stream_handle(stream))
    if st != RMSNORM_OK:
        raise RmsnormError(st, "rmsnorm forward")
    return y


def rmsnorm_fwd_f32(x, w, y=None, eps: float = 1e-6, stream=None):
    """y = RMSNorm(x) * w for float32 CUDA tensors (last dim = hidden)."""
    if y is None:
        y = _torch().empty_like(x)
    rows, hidden = _check_tensors(x, w, y, RMSNORM_DTYPE_F32)
    st = _raw_fwd_f32(x.data_ptr(), w.data_ptr(), y.data_ptr(), rows, hidden, float(eps),
                      _stream_handle(stream))
    if st != RMSNORM_OK:
        raise RmsnormError(st, "rmsnorm_fwd_f32")
    return y


def rmsnorm_fwd_bf16(x, w, y=None, eps: float = 1e-6, stream=None):
    """y = RMSNorm(x) * w for bfloat16 CUDA tensors (fp32 arithmetic)."""
    if y is None:
        y = _torch().empty_like(x)
    rows, hidden = _check_tensors(x, w, y, RMSNORM_DTYPE_BF16)
    st = _raw_fwd_bf16(x.data_ptr(), w.data_ptr(), y.data_ptr(), rows, hidden, float(eps),
                       _stream_handle(stream))
    if st != RMSNORM_OK:
        raise RmsnormError(st, "rmsnorm_fwd_bf16")
    return y


def rmsnorm_fwd_ex(x, w, y=None, eps: float = 1e-6, options=None, stream=None):
    """Either dtype, with explicit options (see ``make_options``)."""
    torch = _torch()
    dtype = RMSNORM_DTYPE_F32 if x.dtype == torch.float32 else RMSNORM_DTYPE_BF16
    if isinstance(options, dict):
        options = make_options(**options)
    return _fwd(dtype, x, w, y, eps, options, stream)


def rmsnorm_fwd_grid_noalloc(x, w, y=None, eps: float = 1e-6, stream=None):
    """The whole-grid kernel with the library's fixed exchange array: the C
    call allocates no device memory (for callers that must not allocate).
    Calls that can overlap on the GPU share that array and race."""
    torch = _torch()
    dtype = RMSNORM_DTYPE_F32 if x.dtype == torch.float32 else RMSNORM_DTYPE_BF16
    if y is None:
        y = torch.empty_like(x)
    rows, hidden = _check_tensors(x, w, y, dtype)
    st = load().rmsnorm_fwd_grid_noalloc(dtype, x.data_ptr(), w.data_ptr(), y.data_ptr(), rows,
                                         hidden, float(eps), _stream_handle(stream) or None)
    if st != RMSNORM_OK:
        raise RmsnormError(st, "rmsnorm_fwd_grid_noalloc")
    return y


def rmsnorm_plan(x, w, y=None, options=None) -> dict:
    """What rmsnorm_fwd_ex would launch for these tensors (no launch)."""
    torch = _torch()
    dtype = RMSNORM_DTYPE_F32 if x.dtype == torch.float32 else RMSNORM_DTYPE_BF16
    if isinstance(options, dict):
        options = make_options(**options)
    y_ptr = (y if y is not None else x).data_ptr()
    hidden = x.shape[-1]
    rows = x.numel() // hidden
    st, plan = _raw_plan(dtype, x.data_ptr(), w.data_ptr(), y_ptr, rows, hidden, options)
    if st != RMSNORM_OK:
        raise RmsnormError(st, "rmsnorm_plan")
    d = {f: getattr(plan, f) for f, _ in rmsnorm_plan_t._fields_ if f != "kernel"}
    d["kernel"] = plan.kernel.decode()
    d["path_name"] = PATH_NAMES.get(plan.path, "?")
    return d


# -------------------------------------------------------------- row softmax --

def _check_sm(x, y):
    torch = _torch()
    if x.dtype not in (torch.float32, torch.bfloat16) or y.dtype != x.dtype:
        raise TypeError("x and y must both be float32 or both bfloat16")
    for name, t in (("x", x), ("y", y)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if y.shape != x.shape or x.dim() == 0 or x.shape[-1] == 0:
        raise ValueError("x and y must share a shape with a non-empty last dim")
    cols = x.shape[-1]
    return x.numel() // cols, cols


def rowsoftmax_fwd_f32(x, y=None, stream=None):
    """y = softmax(x) along the last dim, float32 CUDA tensors."""
    if y is None:
        y = _torch().empty_like(x)
    rows, cols = _check_sm(x, y)
    st = _raw_sm_f32(x.data_ptr(), y.data_ptr(), rows, cols, _stream_handle(stream))
    if st != RMSNORM_OK:
        raise RmsnormError(st, "rowsoftmax_fwd_f32")
    return y


def rowsoftmax_fwd_bf16(x, y=None, stream=None):
    """y = softmax(x) along the last dim, bfloat16 CUDA tensors (fp32 math)."""
    if y is None:
        y = _torch().empty_like(x)
    rows, cols = _check_sm(x, y)
    st = _raw_sm_bf16(x.data_ptr(), y.data_ptr(), rows, cols, _stream_handle(stream))
    if st != RMSNORM_OK:
        raise RmsnormError(st, "rowsoftmax_fwd_bf16")
    return y


def rowsoftmax_fwd_ex(x, y=None, options=None, stream=None):
    """Either dtype with options (path auto / rowreg / cluster / staged /
    twopass, threads, grid; chunk_bytes and stages for the staged path)."""
    torch = _torch()
    if y is None:
        y = torch.empty_like(x)
    rows, cols = _check_sm(x, y)
    if isinstance(options, dict):
        options = make_options(**options)
    dt = RMSNORM_DTYPE_F32 if x.dtype == torch.float32 else RMSNORM_DTYPE_BF16
    st = _raw_sm_ex(dt, x.data_ptr(), y.data_ptr(), rows, cols, options, _stream_handle(stream))
    if st != RMSNORM_OK:
        raise RmsnormError(st, "rowsoftmax_fwd_ex")
    return y


def rowsoftmax_plan(x, y=None, options=None) -> dict:
    torch = _torch()
    if isinstance(options, dict):
        options = make_options(**options)
    cols = x.shape[-1]
    rows = x.numel() // cols
    dt = RMSNORM_DTYPE_F32 if x.dtype == torch.float32 else RMSNORM_DTYPE_BF16
    plan = rmsnorm_plan_t()
    opt = ctypes.byref(options) if options is not None else None
    st = load().rowsoftmax_plan(dt, x.data_ptr(), (y if y is not None else x).data_ptr(),
                                rows, cols, opt, ctypes.byref(plan))
    if st != RMSNORM_OK:
        raise RmsnormError(st, "rowsoftmax_plan")
    d = {f: getattr(plan, f) for f, _ in rmsnorm_plan_t._fields_ if f != "kernel"}
    d["kernel"] = plan.kernel.decode()
    d["path_name"] = PATH_NAMES.get(plan.path, "?")
    return d


def rmsnorm_last_device_status(stream=None) -> int:
    return load().rmsnorm_last_device_status(_stream_handle(stream) or None)


def rmsnorm_status_string(status: int) -> str:
    try:
        return load().rmsnorm_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def rmsnorm_last_cuda_error():
    """(cudaError_t code, "name: description") of the library's last failed
    CUDA call on this thread; clears it."""
    buf = ctypes.create_string_buffer(256)
    code = load().rmsnorm_last_cuda_error(buf, len(buf))
    return code, buf.value.decode(errors="replace")


def rmsnorm_abi_version() -> int:
    return load().rmsnorm_abi_version()
