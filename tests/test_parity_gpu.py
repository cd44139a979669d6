"""GPU parity: librmsnorm's kernels against the fp64 CPU oracle, element by
element, through the C ABI (ctypes binding).  Needs a GB300 (sm_103a)."""
from __future__ import annotations

import zlib

import numpy as np
import pytest
import torch

from _parity import compare, compare_every_row, oracle_for
from row_wise_rmsnorm_fwd_gb300 import binding, build, workloads

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    binding.load()
    torch.cuda.init()
    yield
    torch.cuda.synchronize()
    assert binding.rmsnorm_last_device_status() == binding.RMSNORM_OK


def sms() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count


def run(x, w, eps, y=None, **opts):
    """One call through the C ABI; forced options go through rmsnorm_fwd_ex."""
    if y is None:
        y = torch.empty_like(x)
    if opts:
        binding.rmsnorm_fwd_ex(x, w, y, eps, options=opts)
    elif x.dtype == torch.float32:
        binding.rmsnorm_fwd_f32(x, w, y, eps)
    else:
        binding.rmsnorm_fwd_bf16(x, w, y, eps)
    torch.cuda.synchronize()
    return y


def rand_case(rows, hidden, dtype, seed, xdist=("normal", 0.0, 1.0)):
    x = workloads.make_random((rows, hidden), dtype, seed, xdist)
    w = workloads.make_random((hidden,), dtype, seed + 1, ("normal", 1.0, 0.1))
    return x, w


def check_case(x_cpu, w_cpu, eps, what, **opts):
    y = run(x_cpu.cuda(), w_cpu.cuda(), eps, **opts)
    compare(y, oracle_for(x_cpu, w_cpu, eps), what)
    return y


# ------------------------------------------------------------- workloads --

@pytest.mark.parametrize("name", ["c1", "c2", "c2t", "c3", "c3e", "c5b"])
def test_workload_full(name):
    wl = workloads.WORKLOADS[name]
    x, w = workloads.make_x(wl), workloads.make_w(wl)
    check_case(x, w, wl.eps, name)


@pytest.mark.parametrize("name", ["c1", "c2", "c2t", "c3", "c3e"])
def test_workload_page_schedule(name):
    """The write-up's own schedule, rebuilt as a comparison kernel, on the
    workloads it fits (the page's example is c1)."""
    wl = workloads.WORKLOADS[name]
    x, w = workloads.make_x(wl), workloads.make_w(wl)
    check_case(x.reshape(-1, wl.hidden), w, wl.eps, f"page schedule {name}", path="page")


@pytest.mark.parametrize("name", ["c4", "c5a", "w16m", "w4m"])
def test_workload_full_size_every_row(name):
    """Full-size workload in the bench's launch configuration (automatic
    path, current stream, inputs drawn on the device); every row is checked
    against the oracle, 16384 rows at a time, on all host cores."""
    wl = workloads.WORKLOADS[name]
    x = workloads.make_x(wl, device="cuda")
    w = workloads.make_w(wl, device="cuda")
    y = run(x, w, wl.eps)
    rows, hidden = wl.rows, wl.hidden
    compare_every_row(x.view(rows, hidden), y.view(rows, hidden), w.cpu(), wl.eps,
                      f"{name} full size")
    del x, y
    torch.cuda.empty_cache()


# ----------------------------------------------------------------- sweeps --

WIDTHS = [1, 2, 3, 4, 7, 8, 31, 32, 33, 127, 128, 255, 256, 1000, 2047, 2048, 2049,
          2050, 4095, 4096, 8191, 8192, 8193, 16384, 65536]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("hidden", WIDTHS)
def test_width_sweep(dtype, hidden):
    rows = 37 if hidden <= 8193 else 9
    x, w = rand_case(rows, hidden, dtype, seed=hidden)
    check_case(x, w, 1e-6, f"{dtype} H={hidden}")


@pytest.mark.parametrize("dtype,hidden", [("f32", 4096), ("bf16", 8192), ("f32", 3584)])
def test_row_sweep(dtype, hidden):
    n = sms()
    for rows in [1, 2, 7, 31, 32, 33, n - 1, n, n + 1, 4096]:
        x, w = rand_case(rows, hidden, dtype, seed=rows)
        check_case(x, w, 1e-5, f"{dtype} H={hidden} rows={rows}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,hidden", [(1, 262144), (8, 262144), (3, 100000), (2, 1 << 20),
                                         (1, (1 << 22) + 3), (3, 3 << 20)])
def test_wide_rows(dtype, rows, hidden):
    x, w = rand_case(rows, hidden, dtype, seed=rows + hidden, xdist=("normal", 0.0, 2.0))
    check_case(x, w, 1e-6, f"{dtype} {rows}x{hidden}")


MAX_HIDDEN = (1 << 31) - 1      # the widest row the ABI accepts


@pytest.mark.parametrize("dtype,opts", [("f32", {}), ("bf16", {}),
                                        ("bf16", {"path": "twopass", "cluster": 2})],
                         ids=["f32-auto", "bf16-auto", "bf16-twopass-cluster-2"])
def test_maximum_row_width(dtype, opts):
    """One row of 2^31 - 1 elements.  The width is odd, so every vector is a
    single element and the row holds 2^31 - 1 of them: the vector indices
    reach the top of their range.  x is +-1 with random signs, so the row's
    mean square is exactly 1 whatever its length, and any contiguous piece of
    the row has the same mean square: the oracle, run on the row piece by
    piece (each piece as a row of its own), gives every element's expected
    value.  The automatic choice splits the row over a cluster of two-pass
    CTAs (of the size that fills the most SMs), the forced one over two; the
    unsplit two-pass kernel refuses a row this wide without launching."""
    import concurrent.futures as cf
    import os

    x, w = workloads.make_sign_row(MAX_HIDDEN, dtype, seed=4242)
    with pytest.raises(binding.RmsnormError) as ei:
        binding.rmsnorm_plan(x, w, options={"path": "twopass"})
    assert ei.value.status == binding.RMSNORM_ERR_UNSUPPORTED
    y = run(x, w, 1e-6, **opts)
    plan = binding.rmsnorm_plan(x, w, y, options=opts or None)
    assert plan["vec_bytes"] == x.element_size(), plan
    piece = 1 << 22

    def check(a):
        b = min(MAX_HIDDEN, a + piece)
        xs, ws = x[:, a:b].cpu(), w[a:b].cpu()
        compare(y[:, a:b], oracle_for(xs, ws, 1e-6), f"{dtype} {opts} elements {a}..{b - 1}")

    with cf.ThreadPoolExecutor(max(1, min(8, len(os.sched_getaffinity(0))))) as ex:
        list(ex.map(check, range(0, MAX_HIDDEN, piece)))
    del x, w, y
    torch.cuda.empty_cache()


# ----------------------------------------------------------- forced paths --

FORCED = [
    ("rowreg", {}), ("twopass", {}), ("staged", {}), ("staged", {"chunk_bytes": 4096}),
    ("staged", {"cluster": 2}), ("staged", {"cluster": 4}), ("staged", {"threads": 128}),
    ("staged", {"weights": 1}), ("staged", {"weights": 2, "chunk_bytes": 2048}),
    ("staged", {"stages": 32, "chunk_bytes": 1024}), ("staged", {"cluster": 2, "weights": 1}),
    ("cluster", {"cluster": 2}), ("cluster", {"cluster": 4}), ("cluster", {"cluster": 8}),
    ("cluster", {"cluster": 16}), ("page", {}), ("ringreg", {}), ("ringreg", {"stages": 2}),
    ("ringreg", {"threads": 256}), ("ringreg", {"grid": 2}),
    ("twopass", {"cluster": 2}), ("twopass", {"cluster": 16}),
    ("twopass", {"cluster": 4, "threads": 96}), ("twopass", {"cluster": 3}),
    ("twopass", {"cluster": 12}), ("grid", {}), ("grid", {"grid": 5}), ("grid", {"stages": 2}),
    ("grid", {"threads": 64, "grid": 100}),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path,extra", FORCED, ids=lambda v: str(v))
@pytest.mark.parametrize("rows,hidden", [(5, 4096), (300, 2048), (3, 16384), (2, 8200),
                                         (40, 1000)])
def test_forced_paths(dtype, path, extra, rows, hidden):
    x, w = rand_case(rows, hidden, dtype, seed=7 * rows + hidden)
    opts = dict(path=path, **extra)
    try:
        y = run(x.cuda(), w.cuda(), 1e-6, **opts)
    except binding.RmsnormError as e:
        if e.status == binding.RMSNORM_ERR_UNSUPPORTED:
            pytest.skip(f"{path} {extra} cannot serve {rows}x{hidden}")
        raise
    compare(y, oracle_for(x, w, 1e-6), f"{path} {extra} {dtype} {rows}x{hidden}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,hidden", [(41, 32768), (37, 18432), (9, 16384), (300, 1024),
                                         (5, 8200)])
@pytest.mark.parametrize("extra", [{}, {"stages": 2}, {"stages": 8, "grid": 3}, {"m2": 1},
                                   {"m2": 1, "stages": 2, "grid": 1}, {"m2": 1, "stages": 7},
                                   {"grid": 7}],
                         ids=lambda v: str(v))
def test_ringreg_shapes(dtype, rows, hidden, extra):
    """The ring-to-register kernel over ring depths (2 to 8 slots, fewer or
    more than a row's chunks), both chunk sizes (4 and 2 vectors per consumer
    thread) and CTA counts that give every CTA many rows."""
    if dtype == "bf16" and hidden == 32768:
        hidden = 65536                       # 128 KB rows in both dtypes
    x, w = rand_case(rows, hidden, dtype, seed=rows * 3 + hidden)
    xc, wc = x.cuda(), w.cuda()
    opts = dict(path="ringreg", **{k: v for k, v in extra.items() if k != "m2"})
    if extra.get("m2"):
        plan = binding.rmsnorm_plan(xc, wc, torch.empty_like(xc), options={"path": "ringreg"})
        opts["chunk_bytes"] = 2 * plan["threads_per_row"] * 16
    try:
        y = run(xc, wc, 1e-6, **opts)
    except binding.RmsnormError as e:
        if e.status == binding.RMSNORM_ERR_UNSUPPORTED:
            pytest.skip(f"ringreg {extra} cannot serve {rows}x{hidden}")
        raise
    compare(y, oracle_for(x, w, 1e-6), f"ringreg {extra} {dtype} {rows}x{hidden}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_forced_launch_shapes(dtype):
    """Grid and group sizes that leave some CTAs with no rows, or many."""
    x, w = rand_case(333, 2048, dtype, seed=11)
    ref = oracle_for(x, w, 1e-6)
    xc, wc = x.cuda(), w.cuda()
    for grid in (1, 3, 152, 1000):
        compare(run(xc, wc, 1e-6, path="rowreg", grid=grid), ref, f"grid {grid}")
    for threads in (64, 96, 128, 256, 512):
        compare(run(xc, wc, 1e-6, path="rowreg", threads=threads), ref, f"G {threads}")
    for vb in (4, 8, 16):
        compare(run(xc, wc, 1e-6, path="rowreg", vec_bytes=vb), ref, f"vb {vb}")
    compare(run(xc, wc, 1e-6, path="twopass", threads=96), ref, "twopass 96")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("hidden", [1, 4, 24, 64, 100, 128, 200, 256])
def test_sub_warp_row_groups(dtype, hidden):
    """Rows of fewer than 32 vectors: 1-16 lanes per row, several rows per
    warp; the group reduction must not mix neighbouring rows (rows of very
    different scale sit next to each other)."""
    rows = 1000
    x, w = rand_case(rows, hidden, dtype, seed=hidden + 17)
    x = x * torch.logspace(-3, 3, rows).to(x.dtype).unsqueeze(1)
    ref = oracle_for(x, w, 1e-6)
    xc, wc = x.cuda(), w.cuda()
    compare(run(xc, wc, 1e-6), ref, f"auto {dtype} H={hidden}")
    for g in (1, 2, 4, 8, 16):
        try:
            y = run(xc, wc, 1e-6, path="rowreg", threads=g, grid=77)
        except binding.RmsnormError as e:
            assert e.status == binding.RMSNORM_ERR_UNSUPPORTED
            continue
        compare(y, ref, f"G={g} {dtype} H={hidden}")


# ----------------------------------------------------- layout edge cases --

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("offset", [1, 2, 3, 4, 5])
def test_misaligned_pointers(dtype, offset):
    """x, y and w at element offsets that rule out 16-byte (or any) vectors."""
    rows, hidden = 19, 2050
    x, w = rand_case(rows, hidden, dtype, seed=offset)
    n = rows * hidden
    xb = torch.zeros(n + 16, dtype=DT[dtype], device="cuda")
    yb = torch.zeros(n + 16, dtype=DT[dtype], device="cuda")
    wb = torch.zeros(hidden + 16, dtype=DT[dtype], device="cuda")
    xv = xb[offset:offset + n].view(rows, hidden)
    yv = yb[offset + 1:offset + 1 + n].view(rows, hidden)
    wv = wb[offset + 2:offset + 2 + hidden]
    xv.copy_(x)
    wv.copy_(w)
    run(xv, wv, 1e-6, y=yv)
    compare(yv, oracle_for(x, w, 1e-6), f"offset {offset}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,hidden", [(64, 4096), (8, 65536), (4, 262144), (33, 1000)])
def test_in_place(dtype, rows, hidden):
    x, w = rand_case(rows, hidden, dtype, seed=99)
    xc = x.cuda()
    run(xc, w.cuda(), 1e-6, y=xc)
    compare(xc, oracle_for(x, w, 1e-6), "in place")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path", ["auto", "rowreg", "staged", "cluster", "twopass", "page",
                                  "ringreg", "grid"])
def test_guard_regions_untouched(dtype, path):
    """Sentinels before and after y stay intact (no out-of-bounds stores)."""
    rows, hidden = 21, 4104
    x, w = rand_case(rows, hidden, dtype, seed=3)
    guard = 4096
    n = rows * hidden
    sentinel = -12345.0
    buf = torch.full((guard + n + guard,), sentinel, dtype=DT[dtype], device="cuda")
    y = buf[guard:guard + n].view(rows, hidden)
    opts = {} if path == "auto" else {"path": path}
    try:
        run(x.cuda(), w.cuda(), 1e-6, y=y, **opts)
    except binding.RmsnormError as e:
        if e.status == binding.RMSNORM_ERR_UNSUPPORTED:
            pytest.skip("path cannot serve this shape")
        raise
    assert bool((buf[:guard] == sentinel).all()) and bool((buf[guard + n:] == sentinel).all())
    compare(y, oracle_for(x, w, 1e-6), f"guarded {path}")


# --------------------------------------------------- numerics edge cases --

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_special_rows(dtype):
    """Zero rows, constant rows, NaN and Inf propagation, tiny and huge rows."""
    hidden = 2048
    x = workloads.make_random((8, hidden), "f32", 77)
    x[0] = 0.0
    x[1] = 0.5
    x[2, 5] = float("nan")
    x[3, 7] = float("inf")
    x[4] *= 1e-20
    x[5] *= 1e17   # large but inside the fp32 range of the squared sum
    x[6, :] = -3.0
    x = x.to(DT[dtype])
    w = workloads.make_random((hidden,), dtype, 78, ("normal", 1.0, 0.1))
    check_case(x, w, 1e-6, "special rows")
    check_case(x[:2].contiguous(), w, 0.25, "special rows, large eps")


def test_eps_zero_zero_row_is_nan():
    x = torch.zeros(3, 512)
    x[1] = 1.0
    w = torch.ones(512)
    y = run(x.cuda(), w.cuda(), 0.0).cpu()
    assert torch.isnan(y[0]).all() and torch.isnan(y[2]).all()
    assert torch.allclose(y[1], torch.ones(512))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path", ["auto", "rowreg", "staged", "cluster", "twopass", "page",
                                  "ringreg", "grid"])
def test_deterministic(dtype, path):
    x, w = rand_case(64, 8192, dtype, seed=123)
    xc, wc = x.cuda(), w.cuda()
    opts = {} if path == "auto" else {"path": path}
    try:
        a = run(xc, wc, 1e-6, **opts)
    except binding.RmsnormError as e:
        if e.status == binding.RMSNORM_ERR_UNSUPPORTED:
            pytest.skip("path cannot serve this shape")
        raise
    for _ in range(3):
        assert torch.equal(run(xc, wc, 1e-6, **opts), a)


def test_non_default_stream():
    x, w = rand_case(500, 4096, "f32", seed=1)
    xc, wc = x.cuda(), w.cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = binding.rmsnorm_fwd_f32(xc, wc, eps=1e-6)
    s.synchronize()
    compare(y, oracle_for(x, w, 1e-6), "side stream")


def test_plan_reports_families():
    x = torch.empty(65536, 4096, device="cuda")
    w = torch.empty(4096, device="cuda")
    p = binding.rmsnorm_plan(x, w)
    assert p["path_name"] == "rowreg" and p["vec_bytes"] == 16
    xb = torch.empty(8, 262144, device="cuda", dtype=torch.bfloat16)
    wb = torch.empty(262144, device="cuda", dtype=torch.bfloat16)
    p = binding.rmsnorm_plan(xb, wb)
    assert p["cluster"] > 1


@pytest.mark.parametrize("shape,dtype,kernel,lanes,nv", [
    ((262144, 8192), "bf16", "rowreg", 256, 4),      # c5a
    ((65536, 4096), "f32", "rowreg", 256, 4),        # c4
    ((4096, 128), "bf16", "rowreg", 4, 4),           # per-head QK norm: 8 rows per warp
    ((4096, 1536), "bf16", "rowreg", 64, 3),         # 3 vectors leave no lane idle
    ((1024, 16384), "f32", "staged_bulk", 256, 0),   # fp32 rows of 64 KB
    ((1024, 12288), "f32", "ringreg", 384, 8),       # fp32 rows of 48 KB
    ((1024, 32768), "f32", "ringreg", 512, 16),      # fp32 rows of 128 KB
    ((1024, 24576), "f32", "twopass", 1024, 0),      # fp32 rows of 96 KB
    ((8, 262144), "bf16", "cluster_rowreg", 512, 8), # c5b: few wide rows
    ((2, 1 << 20), "f32", "twopass_cluster", 1024, 0),   # few rows of 4 MB
    ((8, 1 << 24), "f32", "twopass_cluster", 1024, 0),   # w16m: rows of 64 MiB over clusters
    ((12, 10 << 20), "f32", "grid_stream", 448, 2),      # rows of 40 MiB: phased, 14 KB chunks
    ((11, 11 << 20), "f32", "twopass_cluster", 1024, 0), # rows of 44 MiB over clusters
    ((32, 1 << 22), "f32", "grid_stream", 448, 4),       # rows of 16 MiB over the whole grid
    ((16, 1 << 23), "bf16", "grid_stream", 448, 4),      # the same in bf16
    ((40, 5 << 19), "f32", "grid_stream", 448, 4),       # rows of 10 MiB
    ((64, 1 << 21), "f32", "twopass_cluster", 1024, 0),  # rows of 8 MiB: clusters again
])
def test_automatic_choice(shape, dtype, kernel, lanes, nv):
    """The automatic kernel choice for representative shapes (a guard on the
    measured selection rules; no launch)."""
    x = torch.empty(shape, dtype=DT[dtype], device="cuda")
    w = torch.empty(shape[-1], dtype=DT[dtype], device="cuda")
    p = binding.rmsnorm_plan(x, w)
    assert p["kernel"] == kernel, p
    assert p["threads_per_row"] == lanes and p["vecs_per_thread"] == nv, p


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_automatic_whole_grid_rows(dtype):
    """Rows of 16 MiB that the automatic choice spreads over the whole grid
    (cooperative launch, pool scratch), against the oracle; in place too."""
    hidden = (1 << 22) if dtype == "f32" else (1 << 23)
    x, w = rand_case(3, hidden, dtype, seed=41)
    ref = oracle_for(x, w, 1e-6)
    xc, wc = x.cuda(), w.cuda()
    assert binding.rmsnorm_plan(xc, wc)["kernel"] == "grid_stream"
    compare(run(xc, wc, 1e-6), ref, f"auto whole grid {dtype}")
    run(xc, wc, 1e-6, y=xc)
    compare(xc, ref, f"auto whole grid in place {dtype}")


def test_few_very_wide_rows_split_over_clusters():
    """Rows too wide for any cluster's registers or shared memory still spread
    over rows x 16 SMs: the two-pass kernel, each row over a cluster."""
    x = torch.empty(2, 1 << 20, device="cuda")
    w = torch.empty(1 << 20, device="cuda")
    p = binding.rmsnorm_plan(x, w)
    assert p["kernel"] == "twopass_cluster" and p["cluster"] >= 8, p
    assert p["grid"] == 2 * p["cluster"], p
    x = torch.empty(300, 1 << 20, device="cuda")   # many rows: one CTA per row
    p = binding.rmsnorm_plan(x, w)
    assert p["kernel"] == "twopass" and p["cluster"] == 1, p


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,hidden,extra", [
    (3, 1 << 22, {}),                     # rows of 16 / 8 MB over the whole grid
    (2, 4 * 300007 + 4, {"grid": 37}),    # ragged last slice, few CTAs
    (5, 1 << 20, {"stages": 2, "chunk_bytes": 2 * 16 * 448}),
    (1, 1024, {}),                        # a row shorter than the grid: most slices empty
])
def test_rows_over_the_whole_grid(dtype, rows, hidden, extra):
    """Every row split over the whole (cooperatively launched) grid, the CTAs'
    sums of squares meeting in global scratch; in place too."""
    x, w = rand_case(rows, hidden, dtype, seed=rows + hidden % 1000)
    ref = oracle_for(x, w, 1e-6)
    xc, wc = x.cuda(), w.cuda()
    compare(run(xc, wc, 1e-6, path="grid", **extra), ref, f"grid {extra} {dtype} {rows}x{hidden}")
    run(xc, wc, 1e-6, y=xc, path="grid", **extra)
    compare(xc, ref, f"grid in place {extra} {dtype} {rows}x{hidden}")


@pytest.mark.parametrize("dtype,rows,hidden", [
    ("f32", 2, 7 << 20),      # rows of 28 MiB: phased (second read, then the next first read)
    ("f32", 2, 10 << 20),     # rows of 40 MiB: phased, second read reversed
    ("bf16", 2, 14 << 20),    # rows of 28 MiB
    ("bf16", 3, 20 << 20),    # rows of 40 MiB, three rows
])
def test_whole_grid_row_schedules(dtype, rows, hidden):
    """The whole-grid kernel's phased row schedules (chosen for rows wider than
    24 MiB), against the oracle; in place too."""
    x, w = rand_case(rows, hidden, dtype, seed=hidden % 997 + rows)
    ref = oracle_for(x, w, 1e-6)
    xc, wc = x.cuda(), w.cuda()
    compare(run(xc, wc, 1e-6, path="grid"), ref, f"grid schedule {dtype} {rows}x{hidden}")
    run(xc, wc, 1e-6, y=xc, path="grid")
    compare(xc, ref, f"grid schedule in place {dtype} {rows}x{hidden}")


def test_row_kernel_grid_has_about_three_row_blocks_per_cta():
    x = torch.empty(262144, 8192, dtype=torch.bfloat16, device="cuda")
    w = torch.empty(8192, dtype=torch.bfloat16, device="cuda")
    p = binding.rmsnorm_plan(x, w)
    blocks = 262144 // p["rows_per_cta"]
    assert 3 <= blocks / p["grid"] < 4, p


def test_unsupported_forced_option_launches_nothing():
    x = torch.ones(4, 2050, device="cuda")   # 8200-byte rows: no 16-byte pitch
    w = torch.ones(2050, device="cuda")
    y = torch.full_like(x, 7.0)
    with pytest.raises(binding.RmsnormError) as ei:
        binding.rmsnorm_fwd_ex(x, w, y, 1e-6, options={"path": "staged"})
    assert ei.value.status == binding.RMSNORM_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())


# --------------------------------------------------------- fused epilogue --

EPI_PATHS = [("auto", {}), ("rowreg", {}), ("staged", {}), ("ringreg", {}),
             ("cluster", {"cluster": 2}),
             ("cluster", {"cluster": 8}), ("twopass", {}), ("rowreg", {"vec_bytes": 4}),
             ("grid", {})]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("epi,alpha", [("scale", 0.37), ("scale", -4.0), ("relu", 1.0)])
@pytest.mark.parametrize("path,extra", EPI_PATHS, ids=lambda v: str(v))
def test_fused_epilogue(dtype, epi, alpha, path, extra):
    """y = epilogue(RMSNorm(x) * w) in every kernel family, against the oracle's
    epilogue in binary64 (bf16 rounded once, after the epilogue)."""
    rows, hidden = (23, 4096) if path != "cluster" else (5, 16384)
    x, w = rand_case(rows, hidden, dtype, seed=zlib.crc32(f"{epi}{path}".encode()) % 1000)
    opts = {} if path == "auto" else {"path": path, **extra}
    y = torch.empty(rows, hidden, dtype=DT[dtype], device="cuda")
    binding.rmsnorm_fwd_ex(x.cuda(), w.cuda(), y, 1e-6,
                           options={**opts, "epilogue": epi, "alpha": alpha})
    torch.cuda.synchronize()
    compare(y, oracle_for(x, w, 1e-6, epi, alpha), f"{epi} {path} {extra} {dtype}")
    if epi == "relu":
        assert bool((y >= 0).all())


def test_epilogue_rejected_where_unsupported():
    x = torch.ones(4, 512, device="cuda")
    w = torch.ones(512, device="cuda")
    with pytest.raises(binding.RmsnormError) as ei:
        binding.rmsnorm_fwd_ex(x, w, eps=1e-6, options={"path": "page", "epilogue": "relu"})
    assert ei.value.status == binding.RMSNORM_ERR_UNSUPPORTED
    with pytest.raises(binding.RmsnormError) as ei:
        binding.rmsnorm_fwd_ex(x, w, eps=1e-6, options={"epilogue": 9})
    assert ei.value.status == binding.RMSNORM_ERR_INVALID_ARG
    with pytest.raises(binding.RmsnormError) as ei:
        binding.rmsnorm_fwd_ex(x, w, eps=1e-6,
                               options={"epilogue": "scale", "alpha": float("inf")})
    assert ei.value.status == binding.RMSNORM_ERR_INVALID_ARG


# ------------------------------------------------------ model-shaped sweep --

@pytest.mark.parametrize("name", sorted(workloads.MODEL_SWEEP))
def test_model_sweep(name):
    """TinyLlama / Qwen2.5-7B shapes, batch 1..64 x seq 128/512, automatic path:
    every row against the oracle."""
    wl = workloads.MODEL_SWEEP[name]
    x = workloads.make_x(wl, device="cuda").reshape(-1, wl.hidden)
    w = workloads.make_w(wl, device="cuda")
    y = run(x, w, wl.eps)
    compare_every_row(x, y, w.cpu(), wl.eps, name)
