"""Pins for the row-softmax oracle (CPU only), independent of the oracle:
closed forms with exact exponentials, invariants of the definition, extreme
values that an unstabilised formula would overflow, IEEE special cases, and
torch's float64 softmax as an independent library routine."""
import math

import numpy as np
import pytest
import torch

import oracle


def test_closed_form_exp_values_1_3_6():
    """exp(0), exp(ln 3), exp(ln 6) = 1, 3, 6: y = [0.1, 0.3, 0.6]."""
    y = oracle.rowsoftmax_f64(np.array([[0.0, math.log(3.0), math.log(6.0)]]))
    np.testing.assert_allclose(y[0], [0.1, 0.3, 0.6], rtol=4e-16)


def test_closed_form_quarter_quarter_half():
    y = oracle.rowsoftmax_f64(np.array([[0.0, 0.0, math.log(2.0)]]))
    np.testing.assert_allclose(y[0], [0.25, 0.25, 0.5], rtol=4e-16)


@pytest.mark.parametrize("cols", [1, 2, 7, 512, 32000])
def test_uniform_row_is_one_over_n(cols):
    y = oracle.rowsoftmax_f64(np.full((2, cols), -3.25))
    np.testing.assert_array_equal(y, np.full((2, cols), 1.0 / cols))


def test_large_values_do_not_overflow():
    """x = [1000, 1001]: exp(1000) overflows binary64, the stabilised form
    gives [1/(1+e), e/(1+e)]."""
    y = oracle.rowsoftmax_f64(np.array([[1000.0, 1001.0], [-1000.0, -1001.0]]))
    e = math.e
    np.testing.assert_allclose(y[0], [1 / (1 + e), e / (1 + e)], rtol=1e-15)
    np.testing.assert_allclose(y[1], [e / (1 + e), 1 / (1 + e)], rtol=1e-15)


def test_wide_spread_uses_the_maximum():
    """x = [0, 800]: exp(-800) underflows to 0 and the result is [0, 1]; a
    shift by anything but the maximum overflows exp (800 > log(DBL_MAX))."""
    y = oracle.rowsoftmax_f64(np.array([[0.0, 800.0]]))
    assert y[0, 0] == 0.0 and y[0, 1] == 1.0


def test_shift_invariance_and_normalisation():
    rng = np.random.default_rng(40)
    x = rng.normal(0, 3, (6, 333))
    y = oracle.rowsoftmax_f64(x)
    np.testing.assert_allclose(oracle.rowsoftmax_f64(x + 17.5), y, rtol=1e-13)
    np.testing.assert_allclose(y.sum(axis=1), 1.0, rtol=1e-13)
    assert (y > 0).all()
    # order preserving within a row
    for r in range(6):
        assert np.array_equal(np.argsort(x[r], kind="stable"), np.argsort(y[r], kind="stable"))


def test_rows_are_independent_and_permutation_equivariant():
    rng = np.random.default_rng(41)
    x = rng.normal(0, 1, (5, 40))
    y = oracle.rowsoftmax_f64(x)
    for r in range(5):
        np.testing.assert_array_equal(oracle.rowsoftmax_f64(x[r:r + 1]), y[r:r + 1])
    p = rng.permutation(40)
    np.testing.assert_allclose(oracle.rowsoftmax_f64(x[:, p]), y[:, p], rtol=1e-15)


def test_ieee_special_cases():
    with np.errstate(all="ignore"):
        y = oracle.rowsoftmax_f64(np.array([
            [0.0, -np.inf, math.log(3.0)],     # masked entry -> exactly 0
            [-np.inf, -np.inf, -np.inf],       # fully masked -> NaN row
            [1.0, np.nan, 2.0],                # NaN -> NaN row
            [1.0, np.inf, 2.0],                # +inf -> NaN row
        ]))
    np.testing.assert_allclose(y[0], [0.25, 0.0, 0.75], rtol=4e-16)
    assert y[0, 1] == 0.0
    assert np.isnan(y[1]).all() and np.isnan(y[2]).all() and np.isnan(y[3]).all()


@pytest.mark.parametrize("shape", [(3, 5), (64, 512), (4, 32000), (1, 1)])
def test_against_torch_softmax_float64(shape):
    g = torch.Generator().manual_seed(sum(shape))
    x = torch.randn(shape, generator=g, dtype=torch.float64) * 4
    ref = torch.softmax(x, dim=-1).numpy()
    np.testing.assert_allclose(oracle.rowsoftmax_f64(x.numpy()), ref, rtol=1e-13, atol=1e-300)


def test_f32_and_bf16_entries():
    g = torch.Generator().manual_seed(42)
    x = torch.randn(9, 300, generator=g) * 3
    np.testing.assert_array_equal(oracle.rowsoftmax_f32(x.numpy()),
                                  oracle.rowsoftmax_f64(x.double().numpy()))
    xb = x.to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    y64, y16 = oracle.rowsoftmax_bf16(bits)
    np.testing.assert_array_equal(y64, oracle.rowsoftmax_f64(xb.double().numpy()))
    np.testing.assert_array_equal(y16, oracle.f64_to_bf16(y64))


def test_large_magnitude_rows_closed_forms():
    """Rows far from zero: softmax depends only on differences, so 2^24 + k
    (exact in binary32 and binary64 for small integers k) gives softmax(k);
    entries near +-FLT_MAX give 1/count at the maxima and exact zeros
    elsewhere (their differences, up to 6.8e38, underflow exp); two equal
    maxima of any magnitude share 1/2 each."""
    k = np.array([0.0, -1.0, -2.0, -3.0])
    e = np.exp(k)
    y = oracle.rowsoftmax_f32(np.array([2.0 ** 24 + k], dtype=np.float32))
    np.testing.assert_allclose(y[0], e / e.sum(), rtol=1e-15)
    fmax = float(np.finfo(np.float32).max)
    x = np.array([[fmax, -fmax, fmax, 0.0],
                  [-fmax, -fmax, -3.0e38, -fmax],
                  [1.0e10, 1.0e10 - 1024.0, -1.0e10, 1.0e10]], dtype=np.float32)
    y = oracle.rowsoftmax_f32(x)
    np.testing.assert_array_equal(y[0], [0.5, 0.0, 0.5, 0.0])
    np.testing.assert_array_equal(y[1], [0.0, 0.0, 1.0, 0.0])
    np.testing.assert_array_equal(y[2], [0.5, 0.0, 0.0, 0.5])
    # bf16: the largest finite bf16 twice -> 0.5 each (bf16 0x3F00)
    bits = np.array([[0x7F7F, 0x7F7F, 0xFF7F]], dtype=np.uint16)
    y64, y16 = oracle.rowsoftmax_bf16(bits)
    np.testing.assert_array_equal(y64[0], [0.5, 0.5, 0.0])
    np.testing.assert_array_equal(y16[0], [0x3F00, 0x3F00, 0x0000])
