"""Seeded random parity cases: random shapes, element offsets (alignments),
kernel families, launch options and fused epilogues, each checked element by
element against the oracle.  Forced options a family cannot serve are
skipped per case (they must be refused with RMSNORM_ERR_UNSUPPORTED, never
run)."""
from __future__ import annotations

import random

import pytest
import torch

from _parity import SOFTMAX_F32_ATOL, compare, oracle_for
from row_wise_rmsnorm_fwd_gb300 import binding, build, workloads
import oracle

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    binding.load()
    yield
    torch.cuda.synchronize()
    assert binding.rmsnorm_last_device_status() == binding.RMSNORM_OK


def _placed(t: torch.Tensor, offset: int) -> torch.Tensor:
    """A CUDA copy of t that starts `offset` elements into a fresh buffer."""
    flat = torch.zeros(t.numel() + offset + 8, dtype=t.dtype, device="cuda")
    v = flat[offset:offset + t.numel()].view(t.shape)
    v.copy_(t)
    return v


def _offsets(rng: random.Random, dtype: str, n: int):
    """Element offsets: mostly 16-byte aligned (what the bulk-copy kernels
    need), sometimes not (which every family must serve or refuse)."""
    step = 16 // (4 if dtype == "f32" else 2)
    if rng.random() < 0.7:
        return [step * rng.choice([0, 0, 1, 3]) for _ in range(n)]
    return [rng.choice([0, 1, 2, 3, 5]) for _ in range(n)]


def _rms_case(rng: random.Random):
    dtype = rng.choice(["f32", "bf16"])
    hidden = int(2 ** rng.uniform(0, 17.5))
    rows = max(1, min(int(2 ** rng.uniform(0, 12)), (1 << 22) // max(1, hidden)))
    offs = _offsets(rng, dtype, 3)
    path, extra = rng.choice([
        ("auto", {}), ("rowreg", {}), ("rowreg", {"grid": rng.randint(1, 400)}),
        ("staged", {}), ("staged", {"cluster": rng.choice([2, 4])}), ("ringreg", {}),
        ("ringreg", {"stages": rng.randint(2, 6)}), ("cluster", {"cluster": rng.choice([2, 4, 8, 16])}),
        ("twopass", {}), ("page", {}), ("twopass", {"cluster": rng.randint(2, 16)}),
    ])
    epi = rng.choice(["none", "none", "scale", "relu"])
    return dtype, rows, hidden, offs, path, extra, epi


@pytest.mark.parametrize("seed", range(120))
def test_rmsnorm_random_case(seed):
    rng = random.Random(1000 + seed)
    dtype, rows, hidden, offs, path, extra, epi = _rms_case(rng)
    x = workloads.make_random((rows, hidden), dtype, seed, ("normal", 0.0, rng.choice([0.5, 2.0, 30.0])))
    w = workloads.make_random((hidden,), dtype, seed + 1, ("normal", 1.0, 0.2))
    xd, wd = _placed(x, offs[0]), _placed(w, offs[1])
    yd = _placed(torch.zeros_like(x), offs[2])
    opts = dict(extra)
    if path != "auto":
        opts["path"] = path
    if epi != "none":
        opts["epilogue"] = epi
        opts["alpha"] = -0.75
    what = f"seed {seed}: {dtype} {rows}x{hidden} offsets {offs} {path} {extra} {epi}"
    try:
        if opts:
            alpha = opts.pop("alpha", 1.0)
            binding.rmsnorm_fwd_ex(xd, wd, yd, 1e-6, options=binding.make_options(alpha=alpha, **opts))
        elif dtype == "f32":
            binding.rmsnorm_fwd_f32(xd, wd, yd, 1e-6)
        else:
            binding.rmsnorm_fwd_bf16(xd, wd, yd, 1e-6)
    except binding.RmsnormError as e:
        if e.status == binding.RMSNORM_ERR_UNSUPPORTED:
            pytest.skip(f"refused: {what}")
        raise
    torch.cuda.synchronize()
    compare(yd, oracle_for(x, w, 1e-6, epi, -0.75), what)


@pytest.mark.parametrize("seed", range(80))
def test_softmax_random_case(seed):
    rng = random.Random(5000 + seed)
    dtype = rng.choice(["f32", "bf16"])
    cols = int(2 ** rng.uniform(0, 17.5))
    rows = max(1, min(int(2 ** rng.uniform(0, 11)), (1 << 21) // max(1, cols)))
    offs = _offsets(rng, dtype, 2)
    path, extra = rng.choice([
        ("auto", {}), ("rowreg", {}), ("staged", {}), ("staged", {"cluster": rng.choice([2, 4, 8])}),
        ("staged", {"stages": rng.randint(1, 6)}), ("cluster", {"cluster": rng.choice([2, 4, 8, 16])}),
        ("twopass", {}), ("twopass", {"cluster": rng.randint(2, 16)}),
    ])
    x = workloads.make_random((rows, cols), dtype, seed, ("normal", 0.0, rng.choice([1.0, 4.0, 40.0])))
    xd = _placed(x, offs[0])
    yd = _placed(torch.zeros_like(x), offs[1])
    opts = dict(extra)
    if path != "auto":
        opts["path"] = path
    what = f"seed {seed}: {dtype} {rows}x{cols} offsets {offs} {path} {extra}"
    try:
        binding.rowsoftmax_fwd_ex(xd, yd, options=opts)
    except binding.RmsnormError as e:
        if e.status == binding.RMSNORM_ERR_UNSUPPORTED:
            pytest.skip(f"refused: {what}")
        raise
    torch.cuda.synchronize()
    if dtype == "f32":
        ref = oracle.rowsoftmax_f32(x.numpy())
    else:
        _, ref = oracle.rowsoftmax_bf16(workloads.bf16_bits(x))
    compare(yd, ref, what, atol=SOFTMAX_F32_ATOL)
