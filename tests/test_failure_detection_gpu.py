"""Failure detection on the GPU without a GPU fault.

Every device-side wait of the library is bounded.  The test build of the
library (compiled with RMSNORM_FAULT_INJECT, loaded here from
librmsnorm_faultinject.so) can be told to withhold one bulk copy of a staged
kernel (its mbarrier is armed for bytes that never arrive) or one CTA's
partial sum -- or (maximum, sum) pair, for the row softmax -- in a split-row
cluster (its peers' barrier never completes).  The
waits then run out after a short limit, the kernel records
RMSNORM_ERR_TIMEOUT in the device status word, leaves cleanly, and the CUDA
context stays usable: a following clean call must be exact and report OK.
Nothing here traps, faults or spins without a limit.
"""
import ctypes
import time

import pytest
import torch

import oracle
from _parity import SOFTMAX_F32_ATOL, check_bf16, check_f32, compare, oracle_for
from row_wise_rmsnorm_fwd_gb300 import binding, build, workloads

pytestmark = pytest.mark.gpu

LIMIT_NS = 50_000_000      # 50 ms per bounded wait


@pytest.fixture(scope="module")
def flib():
    build.build()
    lib = binding.open_library(build.FAULT_LIB_PATH)
    assert lib.rmsnorm_fault_injection_enabled() == 1
    torch.cuda.init()
    yield lib
    torch.cuda.synchronize()


def call(lib, x, w, y, **opts):
    o = binding.make_options(**opts)
    dt = binding.RMSNORM_DTYPE_F32 if x.dtype == torch.float32 else binding.RMSNORM_DTYPE_BF16
    rows, hidden = x.shape
    return lib.rmsnorm_fwd_ex(dt, x.data_ptr(), w.data_ptr(), y.data_ptr(), rows, hidden,
                              1e-6, ctypes.byref(o),
                              torch.cuda.current_stream().cuda_stream)


def status(lib):
    return lib.rmsnorm_last_device_status(torch.cuda.current_stream().cuda_stream)


def test_product_library_refuses_fault_injection():
    assert binding.load().rmsnorm_fault_injection_enabled() == 0
    x = torch.ones(4, 4096, device="cuda")
    w = torch.ones(4096, device="cuda")
    with pytest.raises(binding.RmsnormError) as ei:
        binding.rmsnorm_fwd_ex(x, w, eps=1e-6, options={"path": "staged", "fault_inject": 1})
    assert ei.value.status == binding.RMSNORM_ERR_UNSUPPORTED


CASES = [
    ("staged withholds a copy", dict(path="staged", fault_inject=1), (64, 4096)),
    ("staged cluster withholds a copy", dict(path="staged", cluster=2, fault_inject=1),
     (16, 8192)),
    ("cluster withholds a partial", dict(path="cluster", cluster=4, fault_inject=2),
     (8, 65536)),
    ("staged cluster withholds a partial", dict(path="staged", cluster=2, fault_inject=2),
     (16, 8192)),
    ("ring-to-register withholds a copy", dict(path="ringreg", fault_inject=1), (64, 16384)),
    ("two-pass cluster withholds a partial", dict(path="twopass", cluster=4, fault_inject=2),
     (8, 65536)),
    ("grid withholds a copy", dict(path="grid", fault_inject=1), (3, 1 << 18)),
    ("grid withholds a partial", dict(path="grid", fault_inject=2), (3, 1 << 18)),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("what,opts,shape", CASES, ids=[c[0] for c in CASES])
def test_bounded_wait_expires_and_context_survives(flib, what, opts, shape, dtype):
    rows, hidden = shape
    x = workloads.make_random(shape, dtype, 5).cuda()
    w = workloads.make_random((hidden,), dtype, 6, ("normal", 1.0, 0.1)).cuda()
    y = torch.empty_like(x)
    assert status(flib) == binding.RMSNORM_OK
    t0 = time.monotonic()
    assert call(flib, x, w, y, wait_timeout_ns=LIMIT_NS, **opts) == binding.RMSNORM_OK
    st = status(flib)                 # synchronises the stream
    elapsed = time.monotonic() - t0
    assert st == binding.RMSNORM_ERR_TIMEOUT, f"{what}: status {st}"
    assert elapsed < 30.0, f"{what}: took {elapsed:.1f} s"
    # the status word was cleared by reading it; the context still works
    assert status(flib) == binding.RMSNORM_OK
    clean = {k: v for k, v in opts.items() if k != "fault_inject"}
    assert call(flib, x, w, y, wait_timeout_ns=LIMIT_NS, **clean) == binding.RMSNORM_OK
    assert status(flib) == binding.RMSNORM_OK
    compare(y, oracle_for(x.cpu(), w.cpu(), 1e-6), f"{what}: clean call after timeout")
    # and so does the product library
    y2 = binding.rmsnorm_fwd_ex(x, w, eps=1e-6, options=clean)
    torch.cuda.synchronize()
    assert torch.equal(y2, y)


def sm_call(lib, x, y, **opts):
    o = binding.make_options(**opts)
    dt = binding.RMSNORM_DTYPE_F32 if x.dtype == torch.float32 else binding.RMSNORM_DTYPE_BF16
    rows, cols = x.shape
    return lib.rowsoftmax_fwd_ex(dt, x.data_ptr(), y.data_ptr(), rows, cols, ctypes.byref(o),
                                 torch.cuda.current_stream().cuda_stream)


def sm_compare(y, x, what):
    x, y = x.cpu(), y.cpu()
    if x.dtype == torch.float32:
        check_f32(y.numpy(), oracle.rowsoftmax_f32(x.numpy()), what, atol=SOFTMAX_F32_ATOL)
    else:
        _, ref16 = oracle.rowsoftmax_bf16(workloads.bf16_bits(x))
        check_bf16(workloads.bf16_bits(y), ref16, what)


SOFTMAX_CASES = [
    ("softmax staged withholds a copy", dict(path="staged", fault_inject=1), (64, 32000)),
    ("softmax staged cluster withholds a copy", dict(path="staged", cluster=4, fault_inject=1),
     (16, 128256)),
    ("softmax cluster withholds a pair", dict(path="cluster", cluster=4, fault_inject=2),
     (8, 65536)),
    ("softmax staged cluster withholds a pair", dict(path="staged", cluster=4, fault_inject=2),
     (16, 128256)),
    ("softmax three-pass cluster withholds a pair",
     dict(path="twopass", cluster=4, fault_inject=2), (8, 65536)),
    ("softmax stream withholds a copy", dict(path="stream", fault_inject=1), (64, 128256)),
    ("softmax stream cluster withholds a copy", dict(path="stream", cluster=2, fault_inject=1),
     (16, 128256)),
    ("softmax stream cluster withholds a pair", dict(path="stream", cluster=2, fault_inject=2),
     (16, 128256)),
    ("softmax grid withholds a copy", dict(path="grid", fault_inject=1), (3, 1 << 18)),
    ("softmax grid withholds a pair", dict(path="grid", fault_inject=2), (3, 1 << 18)),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("what,opts,shape", SOFTMAX_CASES, ids=[c[0] for c in SOFTMAX_CASES])
def test_softmax_bounded_wait_expires_and_context_survives(flib, what, opts, shape, dtype):
    x = workloads.make_random(shape, dtype, 7, ("normal", 0.0, 3.0)).cuda()
    y = torch.empty_like(x)
    assert status(flib) == binding.RMSNORM_OK
    t0 = time.monotonic()
    assert sm_call(flib, x, y, wait_timeout_ns=LIMIT_NS, **opts) == binding.RMSNORM_OK
    st = status(flib)
    elapsed = time.monotonic() - t0
    assert st == binding.RMSNORM_ERR_TIMEOUT, f"{what}: status {st}"
    assert elapsed < 30.0, f"{what}: took {elapsed:.1f} s"
    assert status(flib) == binding.RMSNORM_OK
    clean = {k: v for k, v in opts.items() if k != "fault_inject"}
    assert sm_call(flib, x, y, wait_timeout_ns=LIMIT_NS, **clean) == binding.RMSNORM_OK
    assert status(flib) == binding.RMSNORM_OK
    sm_compare(y, x, f"{what}: clean call after timeout")
    y2 = binding.rowsoftmax_fwd_ex(x, options=clean)
    torch.cuda.synchronize()
    assert torch.equal(y2, y)
