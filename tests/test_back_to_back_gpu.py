"""Back-to-back calls on one stream.  Every kernel is launched so that it may
start while the previous kernel in the stream still runs (programmatic
dependent launch) and waits for that kernel's memory before touching its own;
these tests check that no call reads an input before the previous call has
written it, or writes an output before the previous call has read it.  Each
chain runs twice -- once with a host synchronisation after every call (no
overlap possible), once back to back -- and the results must agree bit for
bit (every kernel is deterministic)."""
from __future__ import annotations

import pytest
import torch

from row_wise_rmsnorm_fwd_gb300 import binding, build, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    binding.load()
    torch.cuda.init()
    yield
    torch.cuda.synchronize()
    assert binding.rmsnorm_last_device_status() == binding.RMSNORM_OK


DT = {"f32": torch.float32, "bf16": torch.bfloat16}

# (op, dtype, rows, hidden, forced options): one case per kernel family
CASES = [
    ("rn", "bf16", 8, 262144, {}),                                  # cluster split, registers
    ("rn", "f32", 4096, 4096, {}),                                  # register-resident rows
    ("rn", "f32", 512, 16384, {"path": "staged"}),                  # bulk-copy staged
    ("rn", "f32", 512, 12288, {"path": "ringreg"}),                 # ring to registers
    ("rn", "f32", 256, 24576, {"path": "twopass"}),                 # two-pass
    ("rn", "f32", 4, 1 << 20, {"path": "twopass", "cluster": 8}),   # two-pass over clusters
    ("rn", "bf16", 256, 2048, {"path": "page"}),                    # page schedule replica
    ("rn", "f32", 3, 1 << 22, {"path": "grid"}),                    # whole grid (cooperative)
    ("sm", "f32", 1024, 8192, {}),                                  # softmax in registers
    ("sm", "f32", 256, 128256, {"path": "stream", "cluster": 2}),   # streamed, split
    ("sm", "bf16", 512, 32000, {"path": "staged"}),                 # staged
    ("sm", "f32", 64, 1 << 20, {"path": "twopass"}),                # three-pass
]


def call(op, x, w, y, opts):
    if op == "rn":
        binding.rmsnorm_fwd_ex(x, w, y, 1e-6, options=opts or None)
    else:
        binding.rowsoftmax_fwd_ex(x, y, options=opts or None)


def ids(c):
    return f"{c[0]}-{c[1]}-{c[2]}x{c[3]}-{c[4].get('path', 'auto')}{c[4].get('cluster', '')}"


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_chained_calls_read_the_previous_output(case):
    """y1 = f(x), y2 = f(y1), y3 = f(y2), ...: each call reads what the call
    before it wrote."""
    op, dt, rows, hidden, opts = case
    x = workloads.make_random((rows, hidden), dt, 11, ("normal", 0.0, 1.0), device="cuda")
    w = workloads.make_random((hidden,), dt, 12, ("normal", 1.0, 0.1), device="cuda")
    steps = 6

    def chain(sync):
        bufs = [x.clone()] + [torch.empty_like(x) for _ in range(steps)]
        for i in range(steps):
            call(op, bufs[i], w, bufs[i + 1], opts)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return bufs[-1]

    ref = chain(True)
    for _ in range(3):
        assert torch.equal(chain(False), ref), f"{ids(case)}: back-to-back chain differs"


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_next_call_overwrites_the_previous_input(case):
    """Call A reads x and writes y; call B, right behind it, writes into x: A
    must have read all of x before B's first store."""
    op, dt, rows, hidden, opts = case
    x = workloads.make_random((rows, hidden), dt, 21, ("normal", 0.0, 1.0), device="cuda")
    z = workloads.make_random((rows, hidden), dt, 22, ("normal", 0.0, 1.0), device="cuda")
    w = workloads.make_random((hidden,), dt, 23, ("normal", 1.0, 0.1), device="cuda")
    ya_ref, yb_ref = torch.empty_like(x), torch.empty_like(x)
    call(op, x, w, ya_ref, opts)
    call(op, z, w, yb_ref, opts)
    torch.cuda.synchronize()
    for _ in range(3):
        xa = x.clone()
        ya = torch.empty_like(x)
        torch.cuda.synchronize()
        call(op, xa, w, ya, opts)      # reads xa
        call(op, z, w, xa, opts)       # overwrites xa
        torch.cuda.synchronize()
        assert torch.equal(ya, ya_ref), f"{ids(case)}: the first call saw its input overwritten"
        assert torch.equal(xa, yb_ref), f"{ids(case)}: the second call's output differs"
