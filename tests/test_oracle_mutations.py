"""The oracle's pins catch planted mistakes (CPU only).

Each case copies the oracle's C source, plants one plausible slip, compiles the
copy into a temporary directory and runs a subset of the pins against it.  The
pins must reject every mutant; the unmodified copy must pass.  Nothing here
touches the real oracle build or the CUDA library.
"""
import ctypes
import json
import os
import shutil
import subprocess

import numpy as np
import pytest

from test_oracle_pins import GOLDEN, _eval_closed_form

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "rmsnorm_oracle.c")
SOFTMAX_SRC = os.path.join(os.path.dirname(SRC), "rowsoftmax_oracle.c")

MUTANTS = {
    "unmodified": None,
    "sum_not_mean": ("double ms = acc / (double)hidden;", "double ms = acc;"),
    "eps_outside_root": ("double rstd = 1.0 / sqrt(ms + eps);",
                         "double rstd = 1.0 / sqrt(ms) + eps;"),
    "eps_dropped": ("double rstd = 1.0 / sqrt(ms + eps);",
                    "double rstd = 1.0 / sqrt(ms);"),
    "weight_index": ("yr[j] = (xr[j] * rstd) * w[j];",
                     "yr[j] = (xr[j] * rstd) * w[hidden - 1 - j];"),
    "lost_sign": ("yr[j] = (xr[j] * rstd) * w[j];",
                  "yr[j] = (fabs(xr[j]) * rstd) * w[j];"),
    "sqrt_not_rsqrt": ("double rstd = 1.0 / sqrt(ms + eps);",
                       "double rstd = sqrt(ms + eps);"),
    "row_offset": ("rms_row_f64(x + r * hidden, w, y + r * hidden, hidden, eps);",
                   "rms_row_f64(x, w, y + r * hidden, hidden, eps);"),
    "bf16_truncate": ("double r = round_half_even(n);", "double r = floor(n);"),
    "bf16_double_round": ("double n = ldexp(a, -(int)q_exp);",
                          "double n = ldexp((double)(float)a, -(int)q_exp);"),
    "bf16_ties_away": ("return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;",
                       "return fl + 1.0;"),
    "epilogue_relu_drops_nan": ("v = (v > 0.0 || isnan(v)) ? v : 0.0;",
                                "v = (v > 0.0) ? v : 0.0;"),
    "epilogue_relu_keeps_negative_zero": ("v = (v > 0.0 || isnan(v)) ? v : 0.0;",
                                          "v = (v >= 0.0 || isnan(v)) ? v : 0.0;"),
    "epilogue_scale_ignored": ("v = alpha * v;", "v = v;"),
}


def _build(tmp_path, name, mutation):
    src = open(SRC).read()
    if mutation is not None:
        old, new = mutation
        assert src.count(old) >= 1, f"mutation site for {name} not found"
        src = src.replace(old, new)
    c = tmp_path / f"{name}.c"
    c.write_text(src)
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                    "-ffp-contract=off", "-o", str(so), str(c), "-lm"],
                   check=True)
    lib = ctypes.CDLL(str(so))
    vp, i64, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
    lib.oracle_rmsnorm_f64.argtypes = [vp, vp, vp, i64, i64, dbl]
    lib.oracle_f64_to_bf16_rne.argtypes = [dbl]
    lib.oracle_f64_to_bf16_rne.restype = ctypes.c_uint16
    lib.oracle_apply_epilogue_f64.argtypes = [vp, i64, ctypes.c_int, dbl]
    return lib


def _pins_pass(lib) -> bool:
    """A compact subset of the pins: worked examples and bf16 rounding."""
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        x = np.ascontiguousarray(case["x"], dtype=np.float64)
        w = np.ascontiguousarray(case["w"], dtype=np.float64)
        y = np.empty_like(x)
        lib.oracle_rmsnorm_f64(x.ctypes.data, w.ctypes.data, y.ctypes.data,
                               x.shape[0], x.shape[1], case["eps"])
        expect = np.array([[float(_eval_closed_form(e)) for e in row]
                           for row in case["y"]])
        if not np.allclose(y, expect, rtol=4e-16, atol=0):
            return False
    # bf16: a tie (1 + 2^-8 -> 1.0), a tie to the odd side's even neighbour
    # (1 + 3*2^-8 -> 0x3F82), and a hair above a tie (must round up)
    probes = {1.0 + 2.0 ** -8: 0x3F80, 1.0 + 3 * 2.0 ** -8: 0x3F82,
              (1.0 + 2.0 ** -8) * (1 + 2.0 ** -40): 0x3F81, 1.0: 0x3F80}
    if not all(lib.oracle_f64_to_bf16_rne(v) == b for v, b in probes.items()):
        return False
    # epilogue definition: ReLU keeps NaN and maps -0 to +0; scale multiplies
    v = np.array([-2.0, -0.0, 3.0, np.nan])
    lib.oracle_apply_epilogue_f64(v.ctypes.data, v.size, 2, 0.0)
    if not (v[0] == 0 and not np.signbit(v[1]) and v[2] == 3.0 and np.isnan(v[3])):
        return False
    v = np.array([1.5, -2.0])
    lib.oracle_apply_epilogue_f64(v.ctypes.data, v.size, 1, 4.0)
    return bool(v[0] == 6.0 and v[1] == -8.0)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(tmp_path, name):
    lib = _build(tmp_path, name, MUTANTS[name])
    if name == "unmodified":
        assert _pins_pass(lib)
    else:
        assert not _pins_pass(lib), f"pins did not catch mutant {name}"


# ---------------------------------------------------------- row softmax --

SOFTMAX_MUTANTS = {
    "unmodified": None,
    "no_max_shift": ("y[j] = exp(x[j] - m);", "y[j] = exp(x[j]);"),
    "min_not_max": ("if (x[j] > m) m = x[j];", "if (x[j] < m) m = x[j];"),
    "divide_by_count": ("for (int64_t j = 0; j < cols; ++j) y[j] = y[j] / s;",
                        "for (int64_t j = 0; j < cols; ++j) y[j] = y[j] / (double)cols;"),
    "first_element_skipped": ("    double s = 0.0;\n    for (int64_t j = 0; j < cols; ++j) {",
                              "    double s = 0.0;\n    for (int64_t j = 1; j < cols; ++j) {"),
}


def _build_softmax(tmp_path, name, mutation):
    src = open(SOFTMAX_SRC).read()
    if mutation is not None:
        old, new = mutation
        assert src.count(old) >= 1, f"mutation site for {name} not found"
        src = src.replace(old, new)
    c = tmp_path / f"sm_{name}.c"
    c.write_text(src)
    so = tmp_path / f"libsm_{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(so), SRC, str(c), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    lib.oracle_rowsoftmax_f64.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_int64, ctypes.c_int64]
    return lib


def _softmax_pins_pass(lib) -> bool:
    import math

    def sm(rows):
        x = np.ascontiguousarray(rows, dtype=np.float64)
        y = np.empty_like(x)
        lib.oracle_rowsoftmax_f64(x.ctypes.data, y.ctypes.data, x.shape[0], x.shape[1])
        return y
    with np.errstate(all="ignore"):
        y = sm([[0.0, math.log(3.0), math.log(6.0)]])
        if not np.allclose(y[0], [0.1, 0.3, 0.6], rtol=4e-16, atol=0):
            return False
        y = sm([[1000.0, 1001.0]])
        e = math.e
        if not np.allclose(y[0], [1 / (1 + e), e / (1 + e)], rtol=1e-15, atol=0):
            return False
        y = sm([[0.0, 800.0]])
        return bool(y[0, 0] == 0.0 and y[0, 1] == 1.0)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(SOFTMAX_MUTANTS))
def test_softmax_pins_reject_mutant(tmp_path, name):
    lib = _build_softmax(tmp_path, name, SOFTMAX_MUTANTS[name])
    if name == "unmodified":
        assert _softmax_pins_pass(lib)
    else:
        assert not _softmax_pins_pass(lib), f"pins did not catch mutant {name}"
