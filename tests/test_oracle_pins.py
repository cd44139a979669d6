"""Pins for the CPU oracle, independent of the oracle itself (CPU only).

Each test checks the oracle against something it does not compute: hand-worked
closed forms (tests/golden/worked_examples.json), exact algebraic identities of
the definition, an independent library routine (torch's float64 CPU
``rms_norm``), and an exhaustive search over bfloat16 for the rounding step.
The definition pinned is the one of the page "A hackable Python ML compiler,
part 2" (RMSNorm Loop IR and generated-kernel epilogue):
``y[r,j] = (x[r,j] * 1/sqrt(mean_j x[r,j]^2 + eps)) * w[j]``.

Each plausible slip in the oracle -- a dropped 1/H, eps outside the root, a
wrong weight index, a wrong sign, rows mixed, a double rounding in the bf16
encoder -- fails at least one test here.
"""
import ast
import json
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")
getcontext().prec = 50


# ---------------------------------------------------------------- helpers --

def _eval_closed_form(expr: str) -> Decimal:
    """Evaluate +, -, *, /, sqrt() over decimal literals at 50 digits."""
    def ev(node):
        if isinstance(node, ast.Expression):
            return ev(node.body)
        if isinstance(node, ast.Constant):
            return Decimal(repr(node.value)) if isinstance(node.value, float) \
                else Decimal(node.value)
        if isinstance(node, ast.UnaryOp) and isinstance(node.op, ast.USub):
            return -ev(node.operand)
        if isinstance(node, ast.BinOp):
            a, b = ev(node.left), ev(node.right)
            if isinstance(node.op, ast.Add):
                return a + b
            if isinstance(node.op, ast.Sub):
                return a - b
            if isinstance(node.op, ast.Mult):
                return a * b
            if isinstance(node.op, ast.Div):
                return a / b
        if (isinstance(node, ast.Call) and isinstance(node.func, ast.Name)
                and node.func.id == "sqrt" and len(node.args) == 1):
            return ev(node.args[0]).sqrt()
        raise ValueError(f"unsupported closed form: {ast.dump(node)}")
    return ev(ast.parse(expr, mode="eval"))


def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


# ------------------------------------------------ hand-worked closed forms --

@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_worked_examples(case):
    x = np.array(case["x"], dtype=np.float64)
    w = np.array(case["w"], dtype=np.float64)
    y = oracle.rmsnorm_f64(x, w, case["eps"])
    expect = np.array([[float(_eval_closed_form(e)) for e in row]
                       for row in case["y"]])
    np.testing.assert_allclose(y, expect, rtol=4e-16, atol=0)


def test_worked_example_intermediates():
    """mean of squares and rstd of the 1x4 ramp: 15/2 and sqrt(2/15)."""
    ms, rstd = oracle.rmsnorm_stats_f64(np.array([[1.0, 2, 3, 4]]), 0.0)
    assert ms[0] == 7.5
    assert abs(rstd[0] - float(Decimal(2 / Decimal(15)).sqrt())) <= 1e-16


# ------------------------------------------------------------ closed forms --

@pytest.mark.parametrize("hidden", [1, 2, 7, 64, 1000])
@pytest.mark.parametrize("c,eps", [(0.5, 1e-6), (-3.0, 1e-5), (1e-3, 1e-6),
                                   (7.25, 0.0), (2.0, 4.0)])
def test_constant_row(hidden, c, eps):
    """A constant row c gives c/sqrt(c^2+eps)*w, independent of H."""
    rng = np.random.default_rng(7)
    w = rng.normal(1.0, 0.1, hidden)
    y = oracle.rmsnorm_f64(np.full((1, hidden), c), w, eps)
    expect = c / math.sqrt(c * c + eps) * w
    # sequential binary64 sum of H equal terms: relative error <= (H-1)u,
    # halved by the root; plus a few roundings in the epilogue
    rtol = (hidden + 6) * 2.0 ** -53
    np.testing.assert_allclose(y[0], expect, rtol=rtol, atol=0)


def test_zero_rows_give_zero():
    x = np.zeros((3, 17))
    x[1] = np.arange(17)          # a non-zero row between zero rows
    y = oracle.rmsnorm_f64(x, np.linspace(-2, 2, 17), 1e-6)
    assert np.all(y[0] == 0) and np.all(y[2] == 0)
    assert np.any(y[1] != 0)


def test_eps_zero_zero_row_is_nan():
    """eps = 0 and a zero row: 0 * (1/sqrt(0)) = 0 * inf = NaN, as defined."""
    with np.errstate(all="ignore"):
        y = oracle.rmsnorm_f64(np.zeros((1, 4)), np.ones(4), 0.0)
    assert np.all(np.isnan(y))


# -------------------------------------------------------------- invariants --

@pytest.mark.parametrize("k", [-6, -1, 1, 3, 10])
def test_scale_invariance_power_of_two(k):
    """y_eps(a x) == y_{eps/a^2}(x) bit for bit when a = 2^k."""
    rng = np.random.default_rng(11)
    x = rng.normal(0, 1, (5, 33))
    w = rng.normal(1, 0.1, 33)
    a = 2.0 ** k
    eps = 1e-6
    np.testing.assert_array_equal(oracle.rmsnorm_f64(a * x, w, eps),
                                  oracle.rmsnorm_f64(x, w, eps / (a * a)))


def test_scale_invariance_eps0_any_scale():
    rng = np.random.default_rng(12)
    x = rng.normal(0, 1, (4, 50))
    w = rng.normal(1, 0.1, 50)
    for a in (0.37, 3.1, 1234.5):
        np.testing.assert_allclose(oracle.rmsnorm_f64(a * x, w, 0.0),
                                   oracle.rmsnorm_f64(x, w, 0.0), rtol=1e-14)


def test_sign_symmetry_exact():
    rng = np.random.default_rng(13)
    x = rng.normal(0, 1, (6, 40))
    w = rng.normal(1, 0.1, 40)
    np.testing.assert_array_equal(oracle.rmsnorm_f64(-x, w, 1e-6),
                                  -oracle.rmsnorm_f64(x, w, 1e-6))


def test_joint_column_permutation():
    """Permuting columns of x and w together permutes y; w is indexed by j."""
    rng = np.random.default_rng(14)
    x = rng.normal(0, 1, (3, 64))
    w = rng.uniform(0.5, 1.5, 64)
    p = rng.permutation(64)
    np.testing.assert_allclose(oracle.rmsnorm_f64(x[:, p], w[p], 1e-6),
                               oracle.rmsnorm_f64(x, w, 1e-6)[:, p], rtol=1e-15)
    # permuting only w must change the result (the weight is per column)
    assert not np.allclose(oracle.rmsnorm_f64(x, w[p], 1e-6),
                           oracle.rmsnorm_f64(x, w, 1e-6)[:, :])


def test_row_independence_exact():
    rng = np.random.default_rng(15)
    x = rng.normal(0, 1, (7, 31))
    w = rng.normal(1, 0.1, 31)
    full = oracle.rmsnorm_f64(x, w, 1e-5)
    for r in range(7):
        np.testing.assert_array_equal(oracle.rmsnorm_f64(x[r:r + 1], w, 1e-5),
                                      full[r:r + 1])


@pytest.mark.parametrize("eps", [0.0, 1e-6, 0.3])
def test_mean_square_identity(eps):
    """mean_j (y_j / w_j)^2 = ms / (ms + eps)."""
    rng = np.random.default_rng(16)
    x = rng.normal(0, 2, (5, 129))
    w = rng.uniform(0.5, 1.5, 129)
    y = oracle.rmsnorm_f64(x, w, eps)
    ms = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.mean((y / w) ** 2, axis=1), ms / (ms + eps),
                               rtol=1e-13)


def test_brute_force_exact_sum_tiny():
    """The sum of squares of small integers is exact; compare against an
    exact rational mean and a 50-digit root for every element."""
    rng = np.random.default_rng(17)
    x = rng.integers(-20, 21, (4, 9)).astype(np.float64)
    w = rng.integers(-5, 6, 9).astype(np.float64) / 4.0
    eps = 0.125
    y = oracle.rmsnorm_f64(x, w, eps)
    for r in range(4):
        ms = Fraction(int(sum(int(v) ** 2 for v in x[r])), 9) + Fraction(1, 8)
        rstd = 1 / (Decimal(ms.numerator) / Decimal(ms.denominator)).sqrt()
        for j in range(9):
            exact = Decimal(int(x[r, j])) * rstd * Decimal(repr(float(w[j])))
            assert abs(y[r, j] - float(exact)) <= 2.5e-16 * max(1.0, abs(float(exact)))


# ---------------------------------------------- independent library routine --

@pytest.mark.parametrize("shape,eps", [((1, 32, 2048), 1e-6), ((3, 5, 7), 1e-5),
                                       ((64, 3584), 1e-6), ((2, 2050), 0.1)])
def test_against_torch_rms_norm_float64(shape, eps):
    g = torch.Generator().manual_seed(sum(shape))
    x = torch.randn(shape, generator=g, dtype=torch.float64) * 3
    w = torch.randn(shape[-1], generator=g, dtype=torch.float64) * 0.1 + 1
    ref = torch.nn.functional.rms_norm(x, (shape[-1],), w, eps).numpy()
    y = oracle.rmsnorm_f64(x.numpy(), w.numpy(), eps)
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-300)


def test_f32_entry_widens_exactly():
    rng = np.random.default_rng(18)
    x = rng.normal(0, 1, (9, 77)).astype(np.float32)
    w = rng.normal(1, 0.1, 77).astype(np.float32)
    np.testing.assert_array_equal(
        oracle.rmsnorm_f32(x, w, 1e-6),
        oracle.rmsnorm_f64(x.astype(np.float64), w.astype(np.float64), 1e-6))


# ----------------------------------------------------------------- bfloat16 --

def _all_bf16_bits():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def test_bf16_decode_matches_torch_for_all_patterns():
    bits = _all_bf16_bits()
    ours = oracle.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    # signed zeros survive
    assert math.copysign(1.0, ours[0x8000]) == -1.0


def _finite_bf16_table():
    """All finite bf16 values as exact Fractions with their bit patterns,
    decoded from the definition (sign, biased exponent, 7 fraction bits)."""
    table = []
    for b in range(65536):
        s, e, f = b >> 15, (b >> 7) & 0xFF, b & 0x7F
        if e == 0xFF:
            continue
        mag = (Fraction(f, 128) * Fraction(2) ** -126 if e == 0
               else (1 + Fraction(f, 128)) * Fraction(2) ** (e - 127))
        table.append((-mag if s else mag, b))
    return table


_TABLE = None


def _nearest_even_bf16(v: float) -> int:
    """Exhaustive round-to-nearest-even over all finite bf16 values."""
    global _TABLE
    if _TABLE is None:
        pos = sorted((m, b) for m, b in _finite_bf16_table() if m > 0 or b == 0)
        _TABLE = pos
    a = Fraction(abs(v))
    sign = 0x8000 if math.copysign(1.0, v) < 0 else 0
    # largest finite and the overflow threshold (halfway to 2^128, ties to even -> inf)
    vals = [m for m, _ in _TABLE]
    lo = 0
    hi = len(vals) - 1
    if a >= vals[-1] + (Fraction(2) ** 128 - vals[-1]) / 2:
        return sign | 0x7F80
    while lo < hi:                 # first index with vals[idx] >= a
        mid = (lo + hi) // 2
        if vals[mid] < a:
            lo = mid + 1
        else:
            hi = mid
    cands = [i for i in (lo - 1, lo) if 0 <= i < len(vals)]
    best = min(cands, key=lambda i: (abs(vals[i] - a), _TABLE[i][1] & 1))
    return sign | _TABLE[best][1]


def test_bf16_encode_round_trips_every_finite_value():
    bits = np.array([b for _, b in _finite_bf16_table()], dtype=np.uint16)
    vals = oracle.bf16_to_f64(bits)
    np.testing.assert_array_equal(oracle.f64_to_bf16(vals), bits)


def test_bf16_encode_ties_go_to_even_exhaustively():
    """Every exact midpoint between neighbouring positive finite bf16 values
    rounds to the one with the even fraction (ties-to-even)."""
    table = sorted((m, b) for m, b in _finite_bf16_table() if m > 0)
    mids, want = [], []
    for (m0, b0), (m1, b1) in zip(table, table[1:]):
        mids.append(float((m0 + m1) / 2))    # exact in binary64
        want.append(b0 if b0 % 2 == 0 else b1)
    got = oracle.f64_to_bf16(np.array(mids))
    np.testing.assert_array_equal(got, np.array(want, dtype=np.uint16))


def test_bf16_encode_just_off_midpoints():
    """A value a hair above (below) a midpoint goes to the upper (lower)
    neighbour.  A hair is 2^-40 relative: far below binary32 resolution, so an
    encoder that rounded through binary32 first (double rounding) would land
    on the midpoint and then on the even neighbour, and fail here."""
    table = sorted((m, b) for m, b in _finite_bf16_table() if m > 0)
    above, below, up, down = [], [], [], []
    for i in range(0, len(table) - 1, 97):
        (m0, b0), (m1, b1) = table[i], table[i + 1]
        mid = (m0 + m1) / 2
        above.append(float(mid * (1 + Fraction(1, 2 ** 40))))
        below.append(float(mid * (1 - Fraction(1, 2 ** 40))))
        up.append(b1)
        down.append(b0)
    np.testing.assert_array_equal(oracle.f64_to_bf16(np.array(above)),
                                  np.array(up, dtype=np.uint16))
    np.testing.assert_array_equal(oracle.f64_to_bf16(np.array(below)),
                                  np.array(down, dtype=np.uint16))


def test_bf16_encode_matches_exhaustive_search_random():
    rng = np.random.default_rng(19)
    vals = np.concatenate([
        rng.normal(0, 1, 300),
        rng.normal(0, 1, 100) * 2.0 ** rng.integers(-140, 130, 100),
        np.array([0.0, -0.0, 1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 2 ** -133,
                  2 ** -134, 3 * 2 ** -135, 2 ** -126 * (1 - 2 ** -9),
                  3.3895313892515355e38, 3.4e38, -1e300, 1e-300]),
    ])
    got = oracle.f64_to_bf16(vals)
    want = np.array([_nearest_even_bf16(float(v)) for v in vals], dtype=np.uint16)
    np.testing.assert_array_equal(got, want)


def test_bf16_encode_agrees_with_torch_on_float32_values():
    """For values exactly representable in binary32 a single RNE rounding to
    bf16 is also what torch's float32->bfloat16 cast does."""
    g = torch.Generator().manual_seed(20)
    v = torch.randn(20000, generator=g) * torch.exp2(
        torch.randint(-100, 100, (20000,), generator=g).float())
    ref = v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_bf16(v.double().numpy())
    np.testing.assert_array_equal(got, ref)


def test_bf16_specials():
    got = oracle.f64_to_bf16(np.array([np.inf, -np.inf, np.nan]))
    assert got[0] == 0x7F80 and got[1] == 0xFF80 and (got[2] & 0x7FFF) == 0x7FC0


def test_bf16_oracle_is_f64_oracle_rounded_once():
    g = torch.Generator().manual_seed(21)
    x = (torch.randn(6, 300, generator=g) * 2).to(torch.bfloat16)
    w = (torch.randn(300, generator=g) * 0.1 + 1).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    wb = w.view(torch.int16).numpy().view(np.uint16)
    y64, y16 = oracle.rmsnorm_bf16(xb, wb, 1e-6)
    np.testing.assert_array_equal(
        y64, oracle.rmsnorm_f64(x.double().numpy(), w.double().numpy(), 1e-6))
    np.testing.assert_array_equal(y16, oracle.f64_to_bf16(y64))


# --------------------------------------------------------- argument checks --

def test_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.rmsnorm_f64(np.ones((2, 3)), np.ones(4), 1e-6)
    with pytest.raises(ValueError):
        oracle.rmsnorm_f64(np.ones((2, 0)), np.ones(0), 1e-6)


def test_empty_rows_ok():
    y = oracle.rmsnorm_f64(np.ones((0, 5)), np.ones(5), 1e-6)
    assert y.shape == (0, 5)


# ------------------------------------------------------------- epilogues --
# The fused epilogue (CuTe DSL JIT-argument page, section 2.3: a compile-time
# epilogue_op such as an optional ReLU, applied to each output before the store).

def test_epilogue_scale_power_of_two_is_exact():
    rng = np.random.default_rng(30)
    x = rng.normal(0, 1, (4, 65)).astype(np.float32)
    w = rng.normal(1, 0.1, 65).astype(np.float32)
    base = oracle.rmsnorm_f32(x, w, 1e-6)
    for a in (0.25, 2.0, -8.0):
        np.testing.assert_array_equal(oracle.rmsnorm_epilogue_f32(x, w, 1e-6, "scale", a),
                                      a * base)


def test_epilogue_relu_definition():
    y = np.array([-2.0, -0.0, 0.0, 1e-300, 3.5, np.nan, -np.inf, np.inf])
    got = oracle.apply_epilogue(y, "relu")
    assert got[0] == 0 and got[1] == 0 and np.signbit(got[1]) == False  # noqa: E712
    assert got[2] == 0 and got[3] == 1e-300 and got[4] == 3.5
    assert np.isnan(got[5]) and got[6] == 0 and got[7] == np.inf


def test_epilogue_relu_matches_torch_float64():
    g = torch.Generator().manual_seed(31)
    x = torch.randn(7, 300, generator=g, dtype=torch.float64)
    w = torch.randn(300, generator=g, dtype=torch.float64) * 0.5 + 0.2
    ref = torch.relu(torch.nn.functional.rms_norm(x, (300,), w, 1e-5)).numpy()
    got = oracle.apply_epilogue(oracle.rmsnorm_f64(x.numpy(), w.numpy(), 1e-5), "relu")
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=0)
    assert (got >= 0).all()


def test_epilogue_none_is_identity_and_bf16_rounds_once():
    g = torch.Generator().manual_seed(32)
    x = (torch.randn(5, 200, generator=g) * 2).to(torch.bfloat16)
    w = (torch.randn(200, generator=g) * 0.1 + 1).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    wb = w.view(torch.int16).numpy().view(np.uint16)
    y64, y16 = oracle.rmsnorm_bf16(xb, wb, 1e-6)
    e64, e16 = oracle.rmsnorm_epilogue_bf16(xb, wb, 1e-6, "none")
    np.testing.assert_array_equal(e64, y64)
    np.testing.assert_array_equal(e16, y16)
    s64, s16 = oracle.rmsnorm_epilogue_bf16(xb, wb, 1e-6, "scale", 3.0)
    np.testing.assert_array_equal(s64, 3.0 * y64)
    np.testing.assert_array_equal(s16, oracle.f64_to_bf16(3.0 * y64))


def test_vectorised_encoder_matches_scalar_encoder():
    rng = np.random.default_rng(33)
    v = rng.normal(0, 1, 5000) * 2.0 ** rng.integers(-130, 128, 5000)
    np.testing.assert_array_equal(oracle.f64_to_bf16_fast(v), oracle.f64_to_bf16(v))
