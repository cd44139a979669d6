"""Seeded synthetic inputs for the RMSNorm forward workloads.

This module draws random numbers and nothing else: it holds none of the
normalisation arithmetic, so the CUDA path and the CPU oracle can both be fed
from it without sharing any of the method.

Shapes and distributions follow the workloads of the page "A hackable Python
ML compiler, part 2" (its RMSNorm example ``torch.nn.RMSNorm(2048)`` on a
``(1,32,2048)`` fp32 input with eps 1e-6, and the TinyLlama / Qwen2.5-7B block
shapes it benchmarks), widened to the bandwidth-bound and bf16 sizes this
library is measured on:

=========  =======================  =====  ================  ===============  ======
name       x shape                  dtype  x distribution    w distribution   eps
=========  =======================  =====  ================  ===============  ======
c1         (1, 32, 2048)            f32    N(0,1)            N(1,0.1)         1e-6
c2         (1, 128, 2048)           f32    N(0,1)            N(1,0.1)         1e-5
c2t        (1, 128, 2050)           f32    N(0,1)            N(1,0.1)         1e-5
c3         (4, 512, 3584)           f32    N(0,1), 36 outlier columns x50     1e-6
c3e        (4, 512, 3584)           f32    N(0,1), 1% of entries x50          1e-6
c4         (65536, 4096)            f32    N(0,1)            U(0.5,1.5)       1e-6
c5a        (262144, 8192)           bf16   N(0,2) (std 2)    N(1,0.1)         1e-6
c5b        (8, 262144)              bf16   N(0,2)            N(1,0.1)         1e-6
w16k       (16384, 16384)           f32    N(0,1)            N(1,0.1)         1e-6
w32k       (8192, 32768)            f32    N(0,1)            N(1,0.1)         1e-6
w64k       (16384, 65536)           bf16   N(0,2)            N(1,0.1)         1e-6
w16m       (8, 16777216)            f32    N(0,1)            N(1,0.1)         1e-6
=========  =======================  =====  ================  ===============  ======

c1..c5b are the measured workloads; w16k (64 KiB rows) and w32k, w64k
(128 KiB rows) are extra wide-row cases, too wide for the register-resident
kernel's sweet spot, used to measure the shared-memory staged, cluster and
two-pass kernels on HBM-sized inputs; w16m (eight rows of 64 MiB) is the
few-rows case too wide for any kernel but the two-pass one.  MODEL_SWEEP
adds the model-shaped batch x seq grid (see below).

Readings: "N(0,2)" is mean 0, standard deviation 2; the Qwen-shaped case's
"1% outlier channels" are round(0.01*3584) = 36 whole columns, picked by a
seeded permutation and multiplied by 50 in every row; c3e is the other
reading of the same phrase, 1% of the entries picked independently (each
with probability 0.01, seeded) and multiplied by 50.  bf16 values are drawn
in fp32 and rounded to bf16 by torch's round-to-nearest-even cast.

Seeds: x uses 1000+k, w uses 2000+k, the outliers 3000+k, where k is
the workload's index in the table.  On the CPU the draws are bit-reproducible;
``device="cuda"`` draws from torch's CUDA generator with the same seed (a
different but equally seeded stream), used where the full tensor is too large
to build on the host.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    shape: tuple
    dtype: str            # "f32" or "bf16"
    x_dist: tuple         # ("normal", mean, std)
    w_dist: tuple         # ("normal", mean, std) or ("uniform", lo, hi)
    eps: float
    outlier_cols: int = 0
    outlier_frac: float = 0.0   # fraction of i.i.d. entries scaled by outlier_scale
    outlier_scale: float = 1.0
    description: str = ""
    op: str = "rmsnorm"   # "rmsnorm" or "softmax" (softmax has no weight)

    @property
    def rows(self) -> int:
        r = 1
        for d in self.shape[:-1]:
            r *= d
        return r

    @property
    def hidden(self) -> int:
        return self.shape[-1]

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def bytes_per_call(self) -> int:
        """Algorithmic bytes: read x once, write y once, read w once (RMSNorm)."""
        w = self.hidden if self.op == "rmsnorm" else 0
        return (2 * self.rows * self.hidden + w) * self.elem_bytes


WORKLOADS = {
    w.name: w for w in [
        Workload("c1", 0, (1, 32, 2048), "f32", ("normal", 0.0, 1.0),
                 ("normal", 1.0, 0.1), 1e-6,
                 description="page example torch.nn.RMSNorm(2048) on (1,32,2048)"),
        Workload("c2", 1, (1, 128, 2048), "f32", ("normal", 0.0, 1.0),
                 ("normal", 1.0, 0.1), 1e-5,
                 description="TinyLlama-shaped (1,128,2048)"),
        Workload("c2t", 1, (1, 128, 2050), "f32", ("normal", 0.0, 1.0),
                 ("normal", 1.0, 0.1), 1e-5,
                 description="ragged row width 2050 (8200-byte row pitch)"),
        Workload("c3", 2, (4, 512, 3584), "f32", ("normal", 0.0, 1.0),
                 ("normal", 1.0, 0.1), 1e-6, outlier_cols=36,
                 outlier_scale=50.0,
                 description="Qwen2.5-7B-shaped (4,512,3584), 36 outlier columns x50"),
        Workload("c3e", 8, (4, 512, 3584), "f32", ("normal", 0.0, 1.0),
                 ("normal", 1.0, 0.1), 1e-6, outlier_frac=0.01,
                 outlier_scale=50.0,
                 description="Qwen2.5-7B-shaped (4,512,3584), 1% of entries x50"),
        Workload("c4", 3, (65536, 4096), "f32", ("normal", 0.0, 1.0),
                 ("uniform", 0.5, 1.5), 1e-6,
                 description="bandwidth-bound fp32 (65536,4096)"),
        Workload("c5a", 4, (262144, 8192), "bf16", ("normal", 0.0, 2.0),
                 ("normal", 1.0, 0.1), 1e-6,
                 description="bandwidth-bound bf16 (262144,8192), 2^31 elements"),
        Workload("c5b", 4, (8, 262144), "bf16", ("normal", 0.0, 2.0),
                 ("normal", 1.0, 0.1), 1e-6,
                 description="few rows, wide bf16 (8,262144)"),
        Workload("w16k", 7, (16384, 16384), "f32", ("normal", 0.0, 1.0),
                 ("normal", 1.0, 0.1), 1e-6,
                 description="wide fp32 rows (16384,16384), 64 KiB per row"),
        Workload("w32k", 5, (8192, 32768), "f32", ("normal", 0.0, 1.0),
                 ("normal", 1.0, 0.1), 1e-6,
                 description="wide fp32 rows (8192,32768), 128 KiB per row"),
        Workload("w64k", 6, (16384, 65536), "bf16", ("normal", 0.0, 2.0),
                 ("normal", 1.0, 0.1), 1e-6,
                 description="wide bf16 rows (16384,65536), 128 KiB per row"),
        Workload("w16m", 9, (8, 1 << 24), "f32", ("normal", 0.0, 1.0),
                 ("normal", 1.0, 0.1), 1e-6,
                 description="few very wide fp32 rows (8,16777216), 64 MiB per row"),
        Workload("w4m", 30, (32, 1 << 22), "f32", ("normal", 0.0, 1.0),
                 ("normal", 1.0, 0.1), 1e-6,
                 description="few wide fp32 rows (32,4194304), 16 MiB per row"),
    ]
}


# Model-shaped sweep: the write-up's model blocks (TinyLlama, hidden 2048;
# Qwen2.5-7B, hidden 3584) at its two sequence lengths (128 and 512) over a
# range of batch sizes; rows = batch * seq.  fp32 as on the page, N(0,1)
# activations, N(1,0.1) weights, eps 1e-5 (TinyLlama) / 1e-6 (Qwen).
MODEL_SWEEP = {}
for _model, _hidden, _eps in (("tinyllama", 2048, 1e-5), ("qwen7b", 3584, 1e-6)):
    for _seq in (128, 512):
        for _batch in (1, 4, 16, 64):
            _name = f"{_model}_b{_batch}_s{_seq}"
            MODEL_SWEEP[_name] = Workload(
                _name, 10 + len(MODEL_SWEEP), (_batch, _seq, _hidden), "f32",
                ("normal", 0.0, 1.0), ("normal", 1.0, 0.1), _eps,
                description=f"{_model}-shaped (batch {_batch}, seq {_seq}, hidden {_hidden})")
WORKLOADS.update(MODEL_SWEEP)

# Row softmax on the same skeleton: attention-score rows (batch 8 x 32 heads x
# seq 512 rows of 512 columns, N(0,2) scores), vocabulary logits (rows of
# 32000, N(0,4)), decode-step logits (few rows of a 128256 vocabulary),
# prefill logits (many rows of a 128256 vocabulary) and few rows of 2^24
# columns (too wide for any kernel but the three-pass one); x only, no weight.
SOFTMAX_WORKLOADS = {
    w.name: w for w in [
        Workload("sm_attn_f32", 40, (8 * 32 * 512, 512), "f32", ("normal", 0.0, 2.0),
                 ("normal", 1.0, 0.0), 0.0, op="softmax",
                 description="softmax over attention scores (131072, 512) fp32"),
        Workload("sm_attn_bf16", 41, (8 * 32 * 512, 512), "bf16", ("normal", 0.0, 2.0),
                 ("normal", 1.0, 0.0), 0.0, op="softmax",
                 description="softmax over attention scores (131072, 512) bf16"),
        Workload("sm_vocab_f32", 42, (4096, 32000), "f32", ("normal", 0.0, 4.0),
                 ("normal", 1.0, 0.0), 0.0, op="softmax",
                 description="softmax over vocabulary logits (4096, 32000) fp32"),
        Workload("sm_vocab_bf16", 43, (8192, 32000), "bf16", ("normal", 0.0, 4.0),
                 ("normal", 1.0, 0.0), 0.0, op="softmax",
                 description="softmax over vocabulary logits (8192, 32000) bf16"),
        Workload("sm_decode_f32", 44, (8, 128256), "f32", ("normal", 0.0, 4.0),
                 ("normal", 1.0, 0.0), 0.0, op="softmax",
                 description="decode-step logits, 8 sequences x 128256 vocabulary, fp32"),
        Workload("sm_decode_bf16", 45, (64, 128256), "bf16", ("normal", 0.0, 4.0),
                 ("normal", 1.0, 0.0), 0.0, op="softmax",
                 description="decode-step logits, 64 sequences x 128256 vocabulary, bf16"),
        Workload("sm_prefill_f32", 46, (1024, 128256), "f32", ("normal", 0.0, 4.0),
                 ("normal", 1.0, 0.0), 0.0, op="softmax",
                 description="prefill logits, 1024 tokens x 128256 vocabulary, fp32"),
        Workload("sm_prefill_bf16", 47, (2048, 128256), "bf16", ("normal", 0.0, 4.0),
                 ("normal", 1.0, 0.0), 0.0, op="softmax",
                 description="prefill logits, 2048 tokens x 128256 vocabulary, bf16"),
        Workload("sm_wide_f32", 48, (8, 1 << 24), "f32", ("normal", 0.0, 4.0),
                 ("normal", 1.0, 0.0), 0.0, op="softmax",
                 description="few very wide rows (8, 16777216) fp32, 64 MiB per row"),
    ]
}
WORKLOADS.update(SOFTMAX_WORKLOADS)


def _torch_dtype(dtype: str):
    return torch.float32 if dtype == "f32" else torch.bfloat16


def _generator(seed: int, device: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _draw(shape, dist, gen, device) -> torch.Tensor:
    kind, a, b = dist
    if kind == "normal":
        t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        return t.mul_(b).add_(a)
    if kind == "uniform":
        t = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
        return t.mul_(b - a).add_(a)
    raise ValueError(f"unknown distribution {kind}")


def outlier_columns(wl: Workload) -> torch.Tensor:
    """The seeded set of outlier columns (empty if the workload has none)."""
    if wl.outlier_cols == 0:
        return torch.empty(0, dtype=torch.long)
    g = _generator(3000 + wl.index, "cpu")
    return torch.randperm(wl.hidden, generator=g)[: wl.outlier_cols].sort().values


def make_x(wl: Workload, device: str = "cpu", rows: int | None = None,
           seed_offset: int = 0) -> torch.Tensor:
    """x for workload ``wl`` with its full shape, or ``rows`` rows of width H.

    ``rows`` draws a prefix-shaped sample (rows x hidden) from the same
    distribution; ``seed_offset`` varies the seed for repeated samples.
    """
    shape = wl.shape if rows is None else (rows, wl.hidden)
    g = _generator(1000 + wl.index + seed_offset, device)
    x = _draw(shape, wl.x_dist, g, device)
    if wl.outlier_cols:
        cols = outlier_columns(wl).to(device)
        x[..., cols] *= wl.outlier_scale
    if wl.outlier_frac:
        go = _generator(3000 + wl.index + seed_offset, device)
        hit = torch.rand(shape, generator=go, device=device) < wl.outlier_frac
        x[hit] *= wl.outlier_scale
    return x.to(_torch_dtype(wl.dtype))


def make_w(wl: Workload, device: str = "cpu") -> torch.Tensor:
    g = _generator(2000 + wl.index, device)
    return _draw((wl.hidden,), wl.w_dist, g, device).to(_torch_dtype(wl.dtype))


def make_random(shape, dtype: str, seed: int, dist=("normal", 0.0, 1.0),
                device: str = "cpu") -> torch.Tensor:
    """A seeded tensor of any shape (for sweeps over widths and row counts)."""
    g = _generator(seed, device)
    return _draw(tuple(shape), dist, g, device).to(_torch_dtype(dtype))


def make_sign_row(n: int, dtype: str, seed: int, device: str = "cuda",
                  w_dist=("normal", 1.0, 0.1), chunk: int = 1 << 27):
    """One row of n entries +1 or -1 (each sign with probability 1/2) and a
    weight vector of n entries from ``w_dist`` (none if ``w_dist`` is None),
    drawn chunk by chunk from generators seeded with ``seed`` (x) and
    ``seed + 1`` (w), so rows of up to 2^31 - 1 entries need no full-size
    temporaries.  Returns (x of shape (1, n), w of shape (n,) or None)."""
    gx, gw = _generator(seed, device), _generator(seed + 1, device)
    x = torch.empty((1, n), dtype=_torch_dtype(dtype), device=device)
    w = None if w_dist is None else torch.empty((n,), dtype=_torch_dtype(dtype), device=device)
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        u = torch.rand(b - a, generator=gx, device=device)
        x[0, a:b] = torch.where(u < 0.5, -1.0, 1.0).to(x.dtype)
        del u
        if w is not None:
            w[a:b] = _draw((b - a,), w_dist, gw, device).to(w.dtype)
    return x, w


def bf16_bits(t: torch.Tensor):
    """bfloat16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def from_bf16_bits(bits) -> torch.Tensor:
    """numpy uint16 bit patterns -> bfloat16 tensor (host)."""
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
