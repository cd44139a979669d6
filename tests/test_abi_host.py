"""The C ABI loads, exports what include/rmsnorm.h declares, and rejects bad
arguments on the host before touching any device (CPU only: every call here
returns before the library makes its first CUDA runtime call)."""
import ctypes
import subprocess

import pytest

from row_wise_rmsnorm_fwd_gb300 import binding, build

OK, INVALID = binding.RMSNORM_OK, binding.RMSNORM_ERR_INVALID_ARG


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_every_declared_function_is_exported(lib):
    names = binding.declared_functions()
    assert {"rmsnorm_fwd_f32", "rmsnorm_fwd_bf16", "rmsnorm_fwd_ex", "rmsnorm_plan",
            "rmsnorm_last_device_status", "rmsnorm_status_string",
            "rmsnorm_abi_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_exports_are_plain_c_symbols(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for n in binding.declared_functions():
        assert n in exported, f"{n} is not an unmangled exported symbol"


def test_status_strings(lib):
    for code in range(5):
        s = binding.rmsnorm_status_string(code)
        assert isinstance(s, str) and s
    assert binding.rmsnorm_status_string(99) == "unknown status"
    assert binding.rmsnorm_abi_version() == 10200


def test_struct_sizes_match_header():
    # int32 x 11 + float + uint64 = 56 bytes; int32 x 12 + char[48] = 96 bytes
    assert ctypes.sizeof(binding.rmsnorm_options_t) == 56
    assert ctypes.sizeof(binding.rmsnorm_plan_t) == 96


A = 0x10000000     # fake, 256-byte aligned "device" addresses: never dereferenced
B = 0x20000000
W = 0x30000000


@pytest.mark.parametrize("fn", ["rmsnorm_fwd_f32", "rmsnorm_fwd_bf16"])
def test_rejects_bad_arguments_before_launch(lib, fn):
    f = getattr(binding.raw, fn)
    assert f(0, W, B, 4, 8, 1e-6) == INVALID                 # x NULL
    assert f(A, 0, B, 4, 8, 1e-6) == INVALID                 # w NULL
    assert f(A, W, 0, 4, 8, 1e-6) == INVALID                 # y NULL
    assert f(A, W, B, -1, 8, 1e-6) == INVALID                # rows < 0
    assert f(A, W, B, 4, 0, 1e-6) == INVALID                 # hidden == 0
    assert f(A, W, B, 4, -3, 1e-6) == INVALID                # hidden < 0
    assert f(A, W, B, 4, 2 ** 31, 1e-6) == INVALID           # hidden too large
    assert f(A, W, B, 2 ** 62, 2 ** 20, 1e-6) == INVALID     # size overflow
    assert f(A, W, B, 4, 8, float("nan")) == INVALID         # eps NaN
    assert f(A, W, B, 4, 8, float("inf")) == INVALID         # eps inf
    assert f(A, W, B, 4, 8, -1e-6) == INVALID                # eps < 0
    assert f(A, W, A + 4, 4, 8, 1e-6) == INVALID             # x/y partial overlap
    assert f(A, B + 8, B, 4, 8, 1e-6) == INVALID             # w inside y
    assert f(A + 1, W, B, 4, 8, 1e-6) == INVALID             # misaligned element


def test_zero_rows_is_ok_without_launch(lib):
    assert binding.raw.rmsnorm_fwd_f32(A, W, B, 0, 8, 1e-6) == OK
    assert binding.raw.rmsnorm_fwd_bf16(A, W, A, 0, 8, 1e-6) == OK   # in place


def test_ex_rejects_bad_dtype(lib):
    assert binding.raw.rmsnorm_fwd_ex(7, A, W, B, 4, 8, 1e-6) == INVALID


def test_plan_rejects_null_plan(lib):
    lib_ = binding.load()
    assert lib_.rmsnorm_plan(0, A, W, B, 4, 8, None, None) == INVALID


def test_product_path_has_no_fallback(monkeypatch, tmp_path):
    """With the library missing the binding raises instead of computing."""
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        binding.load()


@pytest.mark.parametrize("fn", ["rowsoftmax_fwd_f32", "rowsoftmax_fwd_bf16"])
def test_softmax_rejects_bad_arguments_before_launch(lib, fn):
    f = getattr(binding.raw, fn)
    assert f(0, B, 4, 8) == INVALID                  # x NULL
    assert f(A, 0, 4, 8) == INVALID                  # y NULL
    assert f(A, B, -1, 8) == INVALID                 # rows < 0
    assert f(A, B, 4, 0) == INVALID                  # cols == 0
    assert f(A, B, 4, 2 ** 31) == INVALID            # cols too large
    assert f(A, A + 4, 4, 8) == INVALID              # partial overlap
    assert f(A + 1, B, 4, 8) == INVALID              # misaligned element
    assert f(A, B, 0, 8) == OK                       # no rows: nothing to do
    assert f(A, A, 0, 8) == OK                       # in place, no rows


def test_softmax_ex_rejects_rmsnorm_only_options(lib):
    for field, value in (("cluster", 2), ("chunk_bytes", 4096), ("stages", 3), ("weights", 1),
                         ("epilogue", 1), ("path", 5), ("path", 6)):
        o = binding.make_options()
        setattr(o, field, value)
        assert binding.raw.rowsoftmax_fwd_ex(0, A, B, 4, 8, o) == INVALID, field


def test_softmax_fault_injection_is_test_build_only(lib):
    """The product library refuses fault injection at every site (1: the
    staged ring's first copy, 2: a split row's first pair) and where no site
    exists; values outside 0..2 are invalid.  No CUDA call is made."""
    unsupported = binding.RMSNORM_ERR_UNSUPPORTED
    for opts in (dict(path="staged", fault_inject=1), dict(path="staged", cluster=2, fault_inject=1),
                 dict(path="staged", cluster=2, fault_inject=2),
                 dict(path="cluster", cluster=2, fault_inject=2),
                 dict(fault_inject=1), dict(path="rowreg", fault_inject=2),
                 dict(path="twopass", fault_inject=1), dict(path="stream", fault_inject=1),
                 dict(path="stream", cluster=2, fault_inject=2),
                 dict(path="stream", fault_inject=2)):
        o = binding.make_options(**opts)
        assert binding.raw.rowsoftmax_fwd_ex(0, A, B, 4, 8, o) == unsupported, opts
    for v in (-1, 3):
        o = binding.make_options(path="staged", fault_inject=v)
        assert binding.raw.rowsoftmax_fwd_ex(0, A, B, 4, 8, o) == INVALID, v


def test_softmax_ex_staged_shape_options_are_checked(lib):
    """chunk_bytes and stages shape only the staged kernel; bad values are
    rejected before any CUDA call."""
    for path in ("rowreg", "twopass", "cluster"):
        for field in ("chunk_bytes", "stages"):
            o = binding.make_options(path=path)
            setattr(o, field, 32)
            assert binding.raw.rowsoftmax_fwd_ex(0, A, B, 4, 8, o) == INVALID, (path, field)
    for field, value in (("chunk_bytes", 4100), ("chunk_bytes", -16), ("stages", -1)):
        o = binding.make_options(path="staged")
        setattr(o, field, value)
        assert binding.raw.rowsoftmax_fwd_ex(0, A, B, 4, 8, o) == INVALID, (field, value)


def test_softmax_cluster_sizes_are_checked(lib):
    """A split over a cluster takes 2..16 CTAs: any size for the three-pass
    and streamed kernels (RMSNORM_PATH_TWOPASS, RMSNORM_PATH_STREAM), powers
    of two for the register and staged kernels; anything else is refused
    before any CUDA call."""
    for path, cluster in (("cluster", 3), ("cluster", 12), ("staged", 6), ("twopass", 17),
                          ("twopass", -1), ("stream", 17), ("stream", -2), ("rowreg", 2),
                          ("auto", 2)):
        o = binding.make_options(path=path)
        o.cluster = cluster
        assert binding.raw.rowsoftmax_fwd_ex(0, A, B, 4, 8, o) == INVALID, (path, cluster)
