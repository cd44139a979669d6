"""Helpers for the GPU parity tests: run the oracle on the same inputs and
compare element by element within the stated tolerances.

Tolerances (fixed by the accuracy targets of the work and derived from the
arithmetic: fp32 sums of at most a few hundred terms per thread plus a
butterfly/tree of at most 10 levels, rsqrtf (a few ulp), two products):
  fp32: |y_gpu - y_ref| <= max(1e-5 * |y_ref|, 1e-6)
  bf16: the GPU's bf16 bits are within 1 ulp of the oracle's single RNE
        rounding of the binary64 result (+0 and -0 are equal).
Row softmax (fp32) takes the same relative bound with an absolute floor of
1e-35 instead of 1e-6: its outputs are probabilities, mostly far below 1e-6,
so the RMSNorm floor would check them to no relative precision at all; below
about 1e-30 an fp32 exponential is near the subnormal range, where relative
precision runs out.
NaN in the reference must be NaN on the GPU and nowhere else.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from row_wise_rmsnorm_fwd_gb300 import workloads

F32_RTOL = 1e-5
F32_ATOL = 1e-6
SOFTMAX_F32_ATOL = 1e-35
BF16_MAX_ULP = 1


def oracle_for(x_cpu: torch.Tensor, w_cpu: torch.Tensor, eps: float,
               epilogue: str = "none", alpha: float = 1.0):
    """Oracle output for host tensors: float64 array (fp32) or uint16 bits (bf16),
    with the fused epilogue applied before the (single) bf16 rounding."""
    if x_cpu.dtype == torch.float32:
        y = oracle.rmsnorm_f32(x_cpu.numpy(), w_cpu.numpy(), eps)
        return y if epilogue == "none" else oracle.apply_epilogue(y, epilogue, alpha)
    if epilogue == "none":
        _, y16 = oracle.rmsnorm_bf16(workloads.bf16_bits(x_cpu), workloads.bf16_bits(w_cpu),
                                     eps)
        return y16
    _, y16 = oracle.rmsnorm_epilogue_bf16(workloads.bf16_bits(x_cpu),
                                          workloads.bf16_bits(w_cpu), eps, epilogue, alpha)
    return y16


def check_f32(y_gpu: np.ndarray, y_ref: np.ndarray, what: str = "", atol: float = F32_ATOL):
    y = y_gpu.astype(np.float64)
    ref_nan = np.isnan(y_ref)
    assert np.array_equal(np.isnan(y), ref_nan), f"{what}: NaN pattern differs"
    ok = ~ref_nan
    err = np.abs(y[ok] - y_ref[ok])
    tol = np.maximum(F32_RTOL * np.abs(y_ref[ok]), atol)
    bad = err > tol
    if bad.any():
        i = np.flatnonzero(bad)[0]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; first at flat "
            f"index {np.flatnonzero(ok)[i]}: gpu {y[ok][i]!r} ref {y_ref[ok][i]!r}")


def _ordered(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def _is_nan_bits(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int32)
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)


def check_bf16(bits_gpu: np.ndarray, bits_ref: np.ndarray, what: str = ""):
    nan_ref = _is_nan_bits(bits_ref)
    assert np.array_equal(_is_nan_bits(bits_gpu), nan_ref), f"{what}: NaN pattern differs"
    ok = ~nan_ref
    d = np.abs(_ordered(bits_gpu[ok]) - _ordered(bits_ref[ok]))
    bad = d > BF16_MAX_ULP
    if bad.any():
        i = np.flatnonzero(bad)[0]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} bf16 values differ by more than "
            f"{BF16_MAX_ULP} ulp; first: gpu 0x{int(bits_gpu[ok][i]):04x} "
            f"ref 0x{int(bits_ref[ok][i]):04x} ({int(d[i])} ulp)")


def compare_every_row(x_dev: torch.Tensor, y_dev: torch.Tensor, w_cpu, eps: float,
                      what: str = "", chunk_rows: int = 16384, piece_elems: int = 1 << 20,
                      threads: int = 0, op: str = "rmsnorm"):
    """Check every row of a full-size GPU result against the oracle (op
    "rmsnorm", or "softmax" with w_cpu and eps unused).

    Rows are copied to the host in chunks of ``chunk_rows``; each chunk is cut
    into pieces of about ``piece_elems`` elements that host threads run
    through the oracle and the comparison at the same time (the oracle is a C
    library called through ctypes, which releases the interpreter lock, and
    numpy's element-wise kernels release it too).  Small pieces keep numpy's
    temporaries in the allocator's reused heap instead of fresh pages."""
    import concurrent.futures as cf
    import os

    import threading

    rows, hidden = x_dev.shape
    piece_rows = max(1, piece_elems // hidden)
    threads = threads or max(1, len(os.sched_getaffinity(0)))
    f32 = x_dev.dtype == torch.float32
    w_host = None
    if op == "rmsnorm":
        w_host = w_cpu.numpy() if f32 else workloads.bf16_bits(w_cpu)
    local = threading.local()

    def piece(args):
        xs, ys, lo = args
        # per-thread output buffers, reused: threads faulting in fresh pages
        # side by side are serialised by the host kernel
        bufs = getattr(local, "bufs", None)
        if bufs is None or bufs[0].shape != tuple(xs.shape):
            bufs = (np.zeros(tuple(xs.shape), np.float64), np.zeros(tuple(xs.shape), np.uint16))
            local.bufs = bufs
        if op == "softmax":
            if f32:
                ref = oracle.rowsoftmax_f32(xs.numpy(), out=bufs[0])
            else:
                _, ref = oracle.rowsoftmax_bf16(workloads.bf16_bits(xs), out64=bufs[0],
                                                out16=bufs[1])
        elif f32:
            ref = oracle.rmsnorm_f32(xs.numpy(), w_host, eps, out=bufs[0])
        else:
            _, ref = oracle.rmsnorm_bf16(workloads.bf16_bits(xs), w_host, eps,
                                         out64=bufs[0], out16=bufs[1])
        compare(ys, ref, f"{what} rows {lo}..{lo + xs.shape[0] - 1}",
                atol=SOFTMAX_F32_ATOL if op == "softmax" else F32_ATOL)

    with cf.ThreadPoolExecutor(threads) as ex:
        for a in range(0, rows, chunk_rows):
            b = min(rows, a + chunk_rows)
            xc, yc = x_dev[a:b].cpu(), y_dev[a:b].cpu()
            jobs = [(xc[p:p + piece_rows], yc[p:p + piece_rows], a + p)
                    for p in range(0, b - a, piece_rows)]
            list(ex.map(piece, jobs))


def compare(y_gpu: torch.Tensor, ref, what: str = "", atol: float = F32_ATOL):
    """Compare a GPU result (any device) with the oracle's output for it
    (``atol``: the fp32 absolute floor, SOFTMAX_F32_ATOL for row softmax)."""
    y = y_gpu.detach().cpu().contiguous()
    if y.dtype == torch.float32:
        check_f32(y.numpy(), ref, what, atol)
    else:
        check_bf16(workloads.bf16_bits(y), ref, what)
