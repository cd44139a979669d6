"""The every-row checker used on the full-size workloads, exercised on the
CPU: with the oracle's own result it passes, and one planted bad element in
any chunk or piece (including the ragged last ones) is found and located."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from _parity import compare_every_row
from row_wise_rmsnorm_fwd_gb300 import workloads


def _case(dtype, rows=300, hidden=257, seed=11):
    x = workloads.make_random((rows, hidden), dtype, seed)
    w = workloads.make_random((hidden,), dtype, seed + 1, ("normal", 1.0, 0.1))
    if dtype == "f32":
        y = torch.from_numpy(oracle.rmsnorm_f32(x.numpy(), w.numpy(), 1e-6).astype(np.float32))
    else:
        _, y16 = oracle.rmsnorm_bf16(workloads.bf16_bits(x), workloads.bf16_bits(w), 1e-6)
        y = workloads.from_bf16_bits(y16)
    return x, w, y


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_every_row_passes_on_the_oracle_result(dtype):
    x, w, y = _case(dtype)
    compare_every_row(x, y, w, 1e-6, "clean", chunk_rows=128, piece_elems=40 * 257, threads=3)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("row", [0, 127, 128, 255, 299])
def test_every_row_finds_one_bad_element(dtype, row):
    x, w, y = _case(dtype)
    y[row, 200] = y[row, 200] * 1.25 + 0.5
    with pytest.raises(AssertionError) as e:
        compare_every_row(x, y, w, 1e-6, "planted", chunk_rows=128, piece_elems=40 * 257,
                          threads=3)
    lo = int(str(e.value).split("rows ")[1].split("..")[0])
    hi = int(str(e.value).split("..")[1].split(":")[0])
    assert lo <= row <= hi


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_every_row_softmax_mode(dtype):
    x = workloads.make_random((300, 257), dtype, 5, ("normal", 0.0, 3.0))
    if dtype == "f32":
        y = torch.from_numpy(oracle.rowsoftmax_f32(x.numpy()).astype(np.float32))
    else:
        _, y16 = oracle.rowsoftmax_bf16(workloads.bf16_bits(x))
        y = workloads.from_bf16_bits(y16)
    compare_every_row(x, y, None, 0.0, "clean", chunk_rows=128, piece_elems=40 * 257,
                      threads=3, op="softmax")
    y[131, 7] = y[131, 7] * 1.5 + 0.01
    with pytest.raises(AssertionError):
        compare_every_row(x, y, None, 0.0, "planted", chunk_rows=128, piece_elems=40 * 257,
                          threads=3, op="softmax")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sign_row_pieces_reproduce_the_whole_row(dtype):
    """The widest-row parity test checks a row of 2^31 - 1 elements piece by
    piece, running the oracle on each piece as a row of its own.  That is
    exact only because every entry is +1 or -1: the mean square of the row
    and of any piece is then exactly 1.  Checked here on a small row drawn by
    the same generator: the entries are +-1 with both signs present, and the
    oracle's per-piece outputs equal its whole-row outputs bit for bit."""
    n, piece = 10_007, 1_000
    x, w = workloads.make_sign_row(n, dtype, seed=4242, device="cpu", chunk=3_000)
    xf = x.float()
    assert bool((xf.abs() == 1).all()) and 0 < int((xf > 0).sum()) < n
    if dtype == "f32":
        whole = oracle.rmsnorm_f32(x.numpy(), w.numpy(), 1e-6)
        parts = [oracle.rmsnorm_f32(x[:, a:a + piece].numpy(), w[a:a + piece].numpy(), 1e-6)
                 for a in range(0, n, piece)]
    else:
        xb, wb = workloads.bf16_bits(x), workloads.bf16_bits(w)
        _, whole = oracle.rmsnorm_bf16(xb, wb, 1e-6)
        parts = [oracle.rmsnorm_bf16(xb[:, a:a + piece], wb[a:a + piece], 1e-6)[1]
                 for a in range(0, n, piece)]
    assert np.array_equal(np.concatenate(parts, axis=1), whole)


def test_sign_row_softmax_closed_form_matches_the_oracle():
    """The widest-row softmax test compares every output against
    v+ = e / S or v- = e^-1 / S, S = n+ e + n- e^-1, instead of running the
    oracle over 2^31 - 1 columns.  That formula is the definition for a row
    of +-1 entries; checked here against the oracle on a small row drawn by
    the same generator, in binary64 and after the single bf16 rounding."""
    import math

    n = 10_007
    x, _ = workloads.make_sign_row(n, "f32", seed=4343, device="cpu", w_dist=None, chunk=3_000)
    xs = x.numpy()
    n_pos = int((xs > 0).sum())
    s = n_pos * math.e + (n - n_pos) / math.e
    v = np.array([math.e / s, 1.0 / (math.e * s)])
    closed = np.where(xs > 0, v[0], v[1])
    ref = oracle.rowsoftmax_f64(xs.astype(np.float64))
    assert np.allclose(ref, closed, rtol=1e-13, atol=0)
    xb = workloads.bf16_bits(x.to(torch.bfloat16))
    _, ref16 = oracle.rowsoftmax_bf16(xb)
    assert np.array_equal(ref16, np.where(xs > 0, oracle.f64_to_bf16(v)[0],
                                          oracle.f64_to_bf16(v)[1]))
