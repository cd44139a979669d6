"""GPU parity of the row-wise softmax against the fp64 CPU oracle (C ABI via
the ctypes binding).  Tolerances (tests/_parity.py): fp32 |d| <= max(1e-5
|ref|, 1e-35), a relative bound down to outputs near the subnormal range;
bf16 within 1 ulp of the single rounding."""
import numpy as np
import pytest
import torch

import oracle
from _parity import SOFTMAX_F32_ATOL, check_bf16, check_f32, compare_every_row
from row_wise_rmsnorm_fwd_gb300 import binding, build, workloads

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    binding.load()
    yield
    torch.cuda.synchronize()


def ref_for(x_cpu):
    if x_cpu.dtype == torch.float32:
        return oracle.rowsoftmax_f32(x_cpu.numpy())
    _, y16 = oracle.rowsoftmax_bf16(workloads.bf16_bits(x_cpu))
    return y16


def compare(y, ref, what):
    y = y.detach().cpu().contiguous()
    if y.dtype == torch.float32:
        check_f32(y.numpy(), ref, what, atol=SOFTMAX_F32_ATOL)
    else:
        check_bf16(workloads.bf16_bits(y), ref, what)


def run(x, y=None, **opts):
    if y is None:
        y = torch.empty_like(x)
    if opts:
        binding.rowsoftmax_fwd_ex(x, y, options=opts)
    elif x.dtype == torch.float32:
        binding.rowsoftmax_fwd_f32(x, y)
    else:
        binding.rowsoftmax_fwd_bf16(x, y)
    torch.cuda.synchronize()
    return y


def case(rows, cols, dtype, seed, std=3.0):
    return workloads.make_random((rows, cols), dtype, seed, ("normal", 0.0, std))


@pytest.mark.parametrize("name", sorted(workloads.SOFTMAX_WORKLOADS))
def test_softmax_workloads_every_row(name):
    """Every softmax workload at full size in the bench's launch configuration
    (automatic path, inputs drawn on the device): every row against the
    oracle, on all host cores."""
    wl = workloads.SOFTMAX_WORKLOADS[name]
    x = workloads.make_x(wl, device="cuda")
    y = run(x)
    compare_every_row(x.view(wl.rows, wl.hidden), y.view(wl.rows, wl.hidden), None, 0.0,
                      f"{name} full size", op="softmax")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", [1, 2, 3, 31, 32, 33, 127, 512, 1000, 2049, 4096, 8193,
                                  16384, 32000, 65536, 100000])
def test_width_sweep(dtype, cols):
    rows = 37 if cols <= 16384 else 5
    x = case(rows, cols, dtype, cols)
    compare(run(x.cuda()), ref_for(x), f"{dtype} cols={cols}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path,cluster", [("rowreg", 0), ("twopass", 0), ("staged", 0),
                                          ("stream", 0), ("grid", 0),
                                          ("cluster", 2), ("cluster", 4), ("cluster", 8),
                                          ("cluster", 16), ("twopass", 2), ("twopass", 16),
                                          ("twopass", 5), ("twopass", 12)])
@pytest.mark.parametrize("rows,cols", [(300, 512), (7, 4096), (3, 32000), (64, 1000),
                                       (5, 128256), (2, 262144)])
def test_forced_paths(dtype, path, cluster, rows, cols):
    x = case(rows, cols, dtype, rows + cols)
    try:
        y = run(x.cuda(), path=path, cluster=cluster)
    except binding.RmsnormError as e:
        if e.status == binding.RMSNORM_ERR_UNSUPPORTED:
            pytest.skip("path cannot serve this shape")
        raise
    compare(y, ref_for(x), f"{path} C={cluster} {dtype} {rows}x{cols}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path", ["cluster", "twopass"])
def test_cluster_special_values(dtype, path):
    """Masked, fully masked, NaN and +inf rows through the cluster splits of
    the register and the three-pass kernels (the maximum and the sum cross
    the cluster); row 4 has one slice of -inf and finite slices elsewhere."""
    cols = 65536
    x = case(5, cols, "f32", 19)
    x[0, ::7] = -float("inf")
    x[1] = -float("inf")
    x[2, 60000] = float("nan")
    x[3, 3] = float("inf")
    x[4, :cols // 8] = -float("inf")
    x = x.to(DT[dtype])
    y = run(x.cuda(), path=path, cluster=8)
    compare(y, ref_for(x), f"{path} cluster special {dtype}")


def large_magnitude_rows(cols, seed):
    """Rows whose maximum is far from zero, where an exponent offset
    bias - m*log2(e) rounded to fp32 is off by more than exp2 can absorb
    (hundreds at |m| = 1e10) or overflows (|m| > FLT_MAX / log2(e)):
    0: 2^22 + multiples of 1/2 (exact in fp32; real spread of exponentials),
    1: 1e10 + N(0, 3000), 2: -1e10 + N(0, 3000), 3: uniform in [3e38,
    3.38e38], 4: its negation, 5: a mix of both, 6: 3e6 + N(0, 4) (just above
    the fused form's bound), 7: 2e6 + N(0, 4) (just below it)."""
    g = torch.Generator().manual_seed(seed)
    n = lambda std: torch.randn(cols, generator=g, dtype=torch.float64) * std  # noqa: E731
    u = torch.rand(cols, generator=g, dtype=torch.float64)
    rows = [
        2.0 ** 22 + torch.round(n(4.0) * 2) / 2,
        1e10 + n(3000.0),
        -1e10 + n(3000.0),
        3.0e38 + u * 0.38e38,
        -(3.0e38 + u * 0.38e38),
        torch.where(torch.rand(cols, generator=g) < 0.5, 1.0, -1.0).double() * (3.0e38 + u * 0.38e38),
        3e6 + n(4.0),
        2e6 + n(4.0),
    ]
    return torch.stack(rows).float()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path,cluster,cols", [
    ("auto", 0, 4096), ("auto", 0, 32000), ("rowreg", 0, 4096), ("staged", 0, 32000),
    ("cluster", 4, 65536), ("twopass", 0, 65536), ("twopass", 4, 65536),
    ("staged", 2, 128256), ("staged", 4, 128256), ("stream", 0, 65536),
    ("stream", 0, 128256), ("stream", 2, 128256), ("stream", 3, 100000), ("grid", 0, 128256),
    ("grid", 0, 1 << 20)])
def test_large_magnitude_rows(dtype, path, cluster, cols):
    """Rows with maxima from 2e6 to 3.38e38 (either sign) through every
    softmax kernel: finite results equal to the oracle's, no NaN rows."""
    x = large_magnitude_rows(cols, 50 + cols).to(DT[dtype])
    try:
        y = run(x.cuda(), **({} if path == "auto" else {"path": path, "cluster": cluster}))
    except binding.RmsnormError as e:
        if e.status == binding.RMSNORM_ERR_UNSUPPORTED:
            pytest.skip("path cannot serve this shape")
        raise
    assert not torch.isnan(y.float()).any()
    compare(y, ref_for(x), f"large magnitudes {path} C={cluster} {dtype} cols={cols}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols,cluster,stages,grid", [
    (300, 128256, 2, 0, 0),           # prefill-logit rows over clusters of two
    (77, 262144, 4, 0, 0),            # clusters of four
    (100, 262144, 2, 0, 0),           # rows in flight beyond the read-ahead bound
    (9, 100000, 3, 2, 6),             # odd cluster, two-slot ring, two clusters
    (5, 4104, 2, 0, 0),               # slices shorter than one chunk
    (3, 24, 2, 0, 0),                 # three vectors per row split over two CTAs
])
def test_stream_cluster_split(dtype, rows, cols, cluster, stages, grid):
    """The streamed kernel with each row split over a thread-block cluster
    (one (maximum, sum) exchange per row through distributed shared memory)."""
    x = case(rows, cols, dtype, rows * 11 + cols + cluster)
    try:
        y = run(x.cuda(), path="stream", cluster=cluster, stages=stages, grid=grid)
    except binding.RmsnormError as e:
        assert e.status == binding.RMSNORM_ERR_UNSUPPORTED
        nvec = cols * x.element_size() // 16
        assert (cols * x.element_size()) % 16 != 0 or (cluster - 1) * (-(-nvec // cluster)) >= nvec
        return
    compare(y, ref_for(x), f"stream split C={cluster} {dtype} {rows}x{cols} S={stages} grid={grid}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols,chunk,stages,grid,threads", [
    (300, 128256, 0, 0, 0, 0),        # prefill-logit rows, automatic ring
    (7, 8, 0, 0, 0, 0),               # a row shorter than one vector per thread
    (40, 2056, 0, 0, 0, 0),           # one partial chunk per row
    (33, 7684, 0, 0, 0, 0),           # fp32: one full 30720-byte chunk and a 16-byte one
    (160, 100000, 0, 0, 0, 0),        # more rows than SMs, ragged last chunk
    (19, 262144, 0, 2, 5, 0),         # a two-slot ring, five CTAs, many rows each
    (25, 77780, 0, 3, 0, 64),         # 64 consumer threads, three slots (bf16: refused)
    (12, 50000, 16 * 2 * 480, 0, 0, 480),    # two vectors per thread and chunk, 15 warps
])
def test_stream_ring_shapes(dtype, rows, cols, chunk, stages, grid, threads):
    """The two-read streamed kernel over ragged widths, ring depths, grid
    sizes (several rows per CTA) and consumer counts; widths whose rows are
    not a multiple of 16 bytes are refused."""
    x = case(rows, cols, dtype, rows * 7 + cols)
    try:
        y = run(x.cuda(), path="stream", chunk_bytes=chunk, stages=stages, grid=grid,
                threads=threads)
    except binding.RmsnormError as e:
        assert e.status == binding.RMSNORM_ERR_UNSUPPORTED
        assert (cols * x.element_size()) % 16 != 0
        return
    compare(y, ref_for(x), f"stream {dtype} {rows}x{cols} chunk={chunk} S={stages} "
                           f"grid={grid} threads={threads}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_stream_special_values(dtype):
    """Masked entries, a fully masked row, NaN and +inf rows, and a row whose
    first 40000 entries are -inf (whole chunks of it, so some threads see only
    -inf before the finite part) through the streamed kernel; in place too."""
    cols = 128256
    x = case(6, cols, "f32", 23)
    x[0, ::7] = -float("inf")
    x[1] = -float("inf")
    x[2, 60000] = float("nan")
    x[3, 3] = float("inf")
    x[4, :40000] = -float("inf")
    x[5, 100000:] = -float("inf")
    x = x.to(DT[dtype])
    ref = ref_for(x)
    for path, cl in (("stream", 0), ("stream", 2), ("stream", 4), ("grid", 0)):
        compare(run(x.cuda(), path=path, cluster=cl), ref, f"{path} C={cl} special {dtype}")
        xd = x.cuda()
        run(xd, xd, path=path, cluster=cl)
        compare(xd, ref, f"{path} C={cl} special in place {dtype}")


@pytest.mark.parametrize("dtype,rows,cols", [
    ("f32", 3, 1 << 23),      # rows of 32 MiB: the second read interleaved with the next first read
    ("f32", 2, 1 << 24),      # rows of 64 MiB: phased
    ("bf16", 2, 1 << 25),     # rows of 64 MiB
])
def test_whole_grid_row_schedules(dtype, rows, cols):
    """Both row schedules of the whole-grid kernel against the oracle."""
    x = case(rows, cols, dtype, rows + cols % 991)
    compare(run(x.cuda(), path="grid"), ref_for(x), f"grid schedule {dtype} {rows}x{cols}")


MAX_COLS = (1 << 31) - 1      # the widest row the ABI accepts


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_maximum_row_width(dtype):
    """One row of 2^31 - 1 columns (odd: one-element vectors, so the vector
    indices reach the top of their range), split over a cluster of three-pass
    CTAs; the unsplit three-pass kernel refuses it without launching.  x is
    +-1 with random signs, so by the definition every output is one of two
    values, v+ = e / S and v- = e^-1 / S with S = n+ e + n- e^-1 (n+, n- the
    counts of each sign), evaluated in binary64 (and rounded once to bf16);
    every element is compared against its value, piece by piece."""
    import concurrent.futures as cf
    import math
    import os

    x, _ = workloads.make_sign_row(MAX_COLS, dtype, seed=4343, w_dist=None)
    y = torch.empty_like(x)
    with pytest.raises(binding.RmsnormError) as ei:
        binding.rowsoftmax_plan(x, y, options={"path": "twopass"})
    assert ei.value.status == binding.RMSNORM_ERR_UNSUPPORTED
    p = binding.rowsoftmax_plan(x, y)
    assert p["kernel"] == "softmax_cluster_threepass" and p["vec_bytes"] == x.element_size(), p
    run(x, y=y)
    n_pos = int((x > 0).sum())
    n_neg = MAX_COLS - n_pos
    assert 0 < n_pos < MAX_COLS
    s = n_pos * math.e + n_neg / math.e
    v = np.array([math.e / s, 1.0 / (math.e * s)])          # v+, v-
    ref_vals = v if dtype == "f32" else oracle.f64_to_bf16(v)
    piece = 1 << 22

    def check(a):
        b = min(MAX_COLS, a + piece)
        pos = (x[0, a:b] > 0).cpu().numpy()
        ref = np.where(pos, ref_vals[0], ref_vals[1])
        compare(y[:, a:b], ref[None, :], f"{dtype} softmax columns {a}..{b - 1}")

    with cf.ThreadPoolExecutor(max(1, min(8, len(os.sched_getaffinity(0))))) as ex:
        list(ex.map(check, range(0, MAX_COLS, piece)))
    del x, y
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols", [(1, (1 << 22) + 3), (3, 3 << 20), (2, 1 << 20)])
def test_few_very_wide_rows(dtype, rows, cols):
    """Rows too wide for the register and staged kernels, few of them: the
    automatic choice splits each over a cluster of three-pass CTAs."""
    x = case(rows, cols, dtype, rows * 7 + cols)
    xd = x.cuda()
    p = binding.rowsoftmax_plan(xd, torch.empty_like(xd))
    assert p["kernel"] == "softmax_cluster_threepass" and p["cluster"] >= 8, p
    compare(run(xd), ref_for(x), f"{dtype} {rows}x{cols}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols,chunk,stages,grid,threads", [
    (300, 512, 0, 0, 0, 0),            # one chunk per row, the ring holds many rows
    (300, 512, 0, 0, 3, 0),            # 100 rows per CTA: the ring wraps many times
    (41, 32000, 0, 0, 5, 0),           # vocabulary rows, several rows per CTA
    (41, 32000, 4096, 0, 4, 512),      # 16 chunks, a short last chunk
    (41, 32000, 4096, 16, 4, 0),       # ring of exactly one row (no lookahead)
    (41, 32000, 4096, 17, 2, 0),       # one slot of lookahead: slot index drifts per row
    (9, 8200, 1024, 32, 2, 256),       # the largest ring, 17 chunks per row, 256 threads
    (17, 40, 0, 0, 0, 0),              # a row shorter than one vector per consumer thread
    (5, 5000, 16384, 3, 0, 128),       # row of 10/20 KB in one chunk (not a power of two)
])
def test_staged_ring_shapes(dtype, rows, cols, chunk, stages, grid, threads):
    """The shared-memory staged softmax over ring sizes, chunk sizes and CTA
    counts that make every slot-reuse pattern occur.  `chunk` is in bytes of
    bf16 rows; fp32 rows use twice as many bytes, so both dtypes cut a row
    into the same number of chunks."""
    x = case(rows, cols, dtype, rows * 7 + cols)
    chunk_bytes = chunk * (2 if dtype == "f32" else 1)
    y = run(x.cuda(), path="staged", chunk_bytes=chunk_bytes, stages=stages, grid=grid,
            threads=threads)
    compare(y, ref_for(x), f"staged {dtype} {rows}x{cols} chunk={chunk} S={stages} g={grid}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols,cluster,chunk,stages,grid", [
    (37, 128256, 4, 0, 0, 0),          # prefill logits: the automatic split
    (37, 128256, 8, 0, 0, 16),         # two clusters: many rows each
    (9, 65536, 2, 0, 0, 0),
    (300, 20000, 2, 8192, 0, 0),       # several chunks per slice
    (300, 20000, 4, 0, 2, 8),          # a two-slot ring, a row per cluster at a time
    (50, 1928, 16, 64, 0, 0),          # 16-CTA clusters; the last slice is short, so
                                       # some of its chunks are empty
    (5, 8200, 8, 1024, 0, 0),
    (41, 32808, 2, 0, 0, 4),           # two clusters of 20 and 21 rows: odd and even
                                       # row counts through the double-buffered exchange
    (7, 128256, 4, 0, 3, 8),           # clusters of 4 and 3 rows
    (64, 100000, 8, 16384, 0, 8),      # one cluster, 64 rows, two chunks per slice;
                                       # short last slice
])
def test_staged_cluster_split(dtype, rows, cols, cluster, chunk, stages, grid):
    """Rows split over a cluster of CTAs, each staging its slice through its
    own ring into registers; maximum and sum cross the cluster."""
    x = case(rows, cols, dtype, rows + cols + cluster)
    chunk_bytes = chunk * (2 if dtype == "f32" else 1)
    try:
        y = run(x.cuda(), path="staged", cluster=cluster, chunk_bytes=chunk_bytes,
                stages=stages, grid=grid)
    except binding.RmsnormError as e:
        if e.status == binding.RMSNORM_ERR_UNSUPPORTED:
            pytest.skip("this split cannot serve the shape")
        raise
    compare(y, ref_for(x), f"staged C={cluster} {dtype} {rows}x{cols}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_staged_cluster_special_values(dtype):
    """Masked, fully masked, NaN and +inf rows through the cluster-split
    staged kernel (special values in different slices)."""
    x = case(6, 128256, "f32", 29)
    x[0, ::5] = -float("inf")
    x[1] = -float("inf")
    x[2, 128000] = float("nan")        # in the last slice
    x[3, 10] = float("inf")            # in the first slice
    x[4] = 2.0                         # uniform row
    x = x.to(DT[dtype])
    y = run(x.cuda(), path="staged", cluster=4)
    compare(y, ref_for(x), f"staged cluster special {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", [1, 3, 16, 64, 100, 128, 255])
def test_sub_warp_row_groups(dtype, cols):
    """Rows of fewer than 32 vectors: 1-16 lanes per row, several rows per
    warp; the group maximum and sum must not mix neighbouring rows."""
    rows = 700
    x = case(rows, cols, dtype, cols + 5)
    x = (x.float() + torch.linspace(-50, 50, rows).unsqueeze(1)).to(DT[dtype])
    ref = ref_for(x)
    xc = x.cuda()
    compare(run(xc), ref, f"auto {dtype} cols={cols}")
    for g in (1, 2, 4, 8, 16):
        try:
            y = run(xc, path="rowreg", threads=g, grid=53)
        except binding.RmsnormError as e:
            assert e.status == binding.RMSNORM_ERR_UNSUPPORTED
            continue
        compare(y, ref, f"G={g} {dtype} cols={cols}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_staged_special_values(dtype):
    """Masked, fully masked, NaN and +inf rows through the staged kernel
    (each row's maximum and sum cross its consumer warps)."""
    x = case(5, 32000, "f32", 23)
    x[0, ::7] = -float("inf")
    x[1] = -float("inf")
    x[2, 31999] = float("nan")
    x[3, 0] = float("inf")
    x[4] = -3.5
    x = x.to(DT[dtype])
    y = run(x.cuda(), path="staged", grid=2)
    compare(y, ref_for(x), f"staged special {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_special_values(dtype):
    cols = 640
    x = case(6, cols, "f32", 9)
    x[0, ::3] = -float("inf")          # masked entries -> exactly 0
    x[1] = -float("inf")               # fully masked row -> NaN
    x[2, 17] = float("nan")            # NaN -> NaN row
    x[3, 5] = float("inf")             # +inf -> NaN row
    x[4] *= 40.0                       # wide spread: most outputs underflow to 0
    x[5] = 7.25                        # uniform row -> 1/cols
    x = x.to(DT[dtype])
    y = run(x.cuda())
    compare(y, ref_for(x), f"special {dtype}")
    assert bool((y[0].cpu()[::3] == 0).all())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,cols", [(64, 512), (5, 32000), (3, 100000)])
def test_in_place_and_misaligned(dtype, rows, cols):
    x = case(rows, cols, dtype, 3)
    xc = x.cuda()
    run(xc, y=xc)
    compare(xc, ref_for(x), "in place")
    n = rows * cols
    buf = torch.zeros(n + 8, dtype=DT[dtype], device="cuda")
    out = torch.zeros(n + 8, dtype=DT[dtype], device="cuda")
    xv = buf[1:1 + n].view(rows, cols)
    yv = out[3:3 + n].view(rows, cols)
    xv.copy_(x)
    run(xv, y=yv)
    compare(yv, ref_for(x), "misaligned")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_guards_and_determinism(dtype):
    rows, cols = 33, 4104
    x = case(rows, cols, dtype, 4).cuda()
    guard = 2048
    buf = torch.full((guard + rows * cols + guard,), -5.0, dtype=DT[dtype], device="cuda")
    y = buf[guard:guard + rows * cols].view(rows, cols)
    run(x, y=y)
    assert bool((buf[:guard] == -5.0).all()) and bool((buf[-guard:] == -5.0).all())
    for _ in range(3):
        assert torch.equal(run(x), y)


@pytest.mark.parametrize("shape,dtype,kernel", [
    ((131072, 512), "f32", "softmax_rowreg"),
    ((131072, 512), "bf16", "softmax_rowreg"),
    ((4096, 32000), "f32", "softmax_staged"),
    ((8192, 32000), "bf16", "softmax_staged"),
    ((16384, 16384), "bf16", "softmax_rowreg"),          # eight vectors per thread
    ((1024, 128256), "f32", "softmax_cluster_stream"),   # prefill logits, fp32: slices of 2
    ((2048, 128256), "bf16", "softmax_stream"),          # prefill logits, bf16: rows of 256 KB
    ((2048, 262144), "bf16", "softmax_cluster_stream"),  # rows of 512 KB over 2 CTAs
    ((5368, 100000), "bf16", "softmax_stream"),          # rows of 195 KB
    ((8192, 65536), "bf16", "softmax_stream"),           # rows of 128 KB
    ((8192, 49152), "bf16", "softmax_threepass"),        # rows of 96 KB: L2 serves the re-reads
    ((5592, 48000), "f32", "softmax_stream"),            # rows of 188 KB
    ((4096, 65536), "f32", "softmax_stream"),            # rows of 256 KB
    ((1024, 1 << 20), "f32", "softmax_cluster_stream"),  # rows of 4 MB over 8 CTAs
    ((64, 128256), "bf16", "softmax_cluster_stream"),    # decode logits, 64 sequences
    ((8, 128256), "f32", "softmax_cluster_rowreg"),      # decode logits, 8 sequences
    ((2, 1 << 20), "f32", "softmax_cluster_threepass"),  # few rows of 4 MB
    ((8, 1 << 24), "f32", "softmax_grid_stream"),        # rows of 64 MiB over the whole grid
    ((2048, 128255), "f32", "softmax_threepass"),        # rows not a multiple of 16 bytes
])
def test_automatic_choice(shape, dtype, kernel):
    """The automatic kernel choice for representative shapes (no launch)."""
    x = torch.empty(shape, dtype=DT[dtype], device="cuda")
    p = binding.rowsoftmax_plan(x, torch.empty_like(x))
    assert p["kernel"] == kernel, p


def test_plans_report_each_kernels_own_launch():
    """Each plan reports the launch of the kernel it chose and nothing of the
    others: the streamed kernel its ring and no cluster, the three-pass kernel
    (forced) no ring, the staged split (forced) its cluster and ring."""
    x = torch.empty((3533, 151936), dtype=torch.bfloat16, device="cuda")
    p = binding.rowsoftmax_plan(x, torch.empty_like(x))
    assert p["kernel"] == "softmax_stream", p
    assert p["cluster"] == 1 and p["smem_bytes"] > 0 and p["stages"] >= 2, p
    assert p["block_threads"] == 480 and p["grid"] == torch.cuda.get_device_properties(0).multi_processor_count, p
    t = binding.rowsoftmax_plan(x, torch.empty_like(x), options={"path": "twopass"})
    assert t["kernel"] == "softmax_threepass", t
    assert t["cluster"] == 1 and t["smem_bytes"] == 0 and t["stages"] == 0, t
    q = binding.rowsoftmax_plan(x, torch.empty_like(x), options={"path": "staged", "cluster": 8})
    assert q["cluster"] == 8 and q["smem_bytes"] > 0 and q["stages"] >= 1, q


def test_rows_sum_to_one_and_match_torch():
    x = case(1000, 512, "f32", 5).cuda()
    y = run(x)
    torch.testing.assert_close(y.sum(-1), torch.ones(1000, device="cuda"), rtol=0, atol=2e-6)
    torch.testing.assert_close(y, torch.softmax(x, -1), rtol=1e-5, atol=1e-7)
