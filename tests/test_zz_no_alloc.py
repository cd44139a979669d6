"""The allocation-free entry point, rmsnorm_fwd_grid_noalloc.

Some callers may not allocate device memory while they run: an engine or
plugin host that owns and accounts for all device memory, or code on a path
where an allocation must not fail or block.  For them the library runs its
whole-grid kernel (every row split over all SMs; few rows of tens of MB) with
the kernel's exchange area in a fixed device array inside the library rather
than memory taken from the pool per call.

This file is collected last (pytest orders files by name), so that a run that
stops at the first failure has already run every other test; it passes on
its own in a fresh process too.  The new call must give what the pooled call
(rmsnorm_fwd_ex with path GRID) gives, within the suite's tolerances, on two
calls in a row: the second one finds the first one's counter and partials in
the array and must clear them.
"""
import ctypes

import numpy as np
import pytest
import torch

from _parity import check_bf16, check_f32
from row_wise_rmsnorm_fwd_gb300 import binding, build, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    build.build()
    lib = binding.load()
    torch.cuda.init()
    yield lib
    torch.cuda.synchronize()


def c_call(lib, x, w, y, eps):
    """rmsnorm_fwd_grid_noalloc through the C ABI."""
    dt = binding.RMSNORM_DTYPE_F32 if x.dtype == torch.float32 else binding.RMSNORM_DTYPE_BF16
    rows, hidden = x.shape
    return lib.rmsnorm_fwd_grid_noalloc(dt, ctypes.c_void_p(x.data_ptr()),
                                        ctypes.c_void_p(w.data_ptr()),
                                        ctypes.c_void_p(y.data_ptr()), rows, hidden, eps,
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def same_within_tolerance(got, want, what):
    """The suite's tolerances, with the pooled call's output as reference:
    fp32 |d| <= max(1e-5 |ref|, 1e-6); bf16 within 1 ulp."""
    got, want = got.cpu(), want.cpu()
    if got.dtype == torch.float32:
        check_f32(got.numpy(), want.double().numpy(), what)
    else:
        check_bf16(workloads.bf16_bits(got), workloads.bf16_bits(want), what)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,hidden", [(3, 1 << 22), (5, 300000 * 4), (1, 4096)])
def test_noalloc_matches_pooled_call_twice(lib, dtype, rows, hidden):
    eps = 1e-6
    outs = []
    for call in range(2):                    # two calls in a row, different inputs
        x = workloads.make_random((rows, hidden), dtype, 100 * call + rows,
                                  ("normal", 0.0, 1.0 + call)).cuda()
        w = workloads.make_random((hidden,), dtype, 7 + call, ("normal", 1.0, 0.1)).cuda()
        ref = binding.rmsnorm_fwd_ex(x, w, eps=eps, options={"path": "grid"})
        y = torch.full_like(x, float("nan"))
        assert c_call(lib, x, w, y, eps) == binding.RMSNORM_OK
        torch.cuda.synchronize()
        same_within_tolerance(y, ref, f"no-alloc call {call + 1} {dtype} {rows}x{hidden}")
        outs.append(y)
    assert binding.rmsnorm_last_device_status() == binding.RMSNORM_OK
    assert not torch.equal(outs[0], outs[1])


def test_noalloc_rejects_what_the_grid_kernel_cannot_serve(lib):
    """Rows that are not 16-byte aligned cannot be streamed by bulk copies:
    refused before any launch, the output left untouched."""
    x = torch.ones(2, 2050, device="cuda")          # 8200-byte rows
    w = torch.ones(2050, device="cuda")
    y = torch.full_like(x, 7.0)
    assert c_call(lib, x, w, y, 1e-6) == binding.RMSNORM_ERR_UNSUPPORTED
    assert c_call(lib, x, w, y, -1.0) == binding.RMSNORM_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())
