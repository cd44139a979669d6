"""Concurrency and CUDA-graph behaviour of the C ABI (GPU).

- Several host threads call the library at once, each on its own stream
  (per-device set-up runs once under a lock; launches carry no shared state).
- Calls captured into a CUDA graph replay with the same results: the launch
  path makes no host-synchronising call once a shape has been planned.
"""
import threading

import pytest
import torch

from _parity import compare, oracle_for
from row_wise_rmsnorm_fwd_gb300 import binding, build, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    binding.load()
    yield
    torch.cuda.synchronize()


def test_concurrent_host_threads():
    shapes = [(300, 4096, "f32"), (77, 8192, "bf16"), (5, 65536, "f32"), (1000, 512, "bf16"),
              (40, 16384, "f32"), (9, 262144, "bf16")]
    cases = []
    for i, (r, h, dt) in enumerate(shapes):
        x = workloads.make_random((r, h), dt, 100 + i)
        w = workloads.make_random((h,), dt, 200 + i, ("normal", 1.0, 0.1))
        cases.append((x, w, x.cuda(), w.cuda()))
    outs = [None] * len(cases)
    errors = []

    def work(i):
        try:
            s = torch.cuda.Stream()
            _, _, xd, wd = cases[i]
            with torch.cuda.stream(s):
                y = None
                for _ in range(20):
                    y = binding.rmsnorm_fwd_ex(xd, wd, eps=1e-6)
                    sm = binding.rowsoftmax_fwd_ex(xd)
            s.synchronize()
            outs[i] = (y, sm)
        except Exception as e:  # noqa: BLE001 -- collected and re-raised below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, (x, w, _, _) in enumerate(cases):
        compare(outs[i][0], oracle_for(x, w, 1e-6), f"thread {i}")
    assert binding.rmsnorm_last_device_status() == binding.RMSNORM_OK


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_cuda_graph_capture_and_replay(dtype):
    """Small, launch-bound calls (a TinyLlama-shaped block has two RMSNorms)
    captured once into a graph and replayed."""
    H = 2048
    xs = [workloads.make_random((128, H), dtype, 300 + k) for k in range(4)]
    w = workloads.make_random((H,), dtype, 310, ("normal", 1.0, 0.1))
    xd = [x.cuda() for x in xs]
    wd = w.cuda()
    ys = [torch.empty_like(x) for x in xd]
    fwd = binding.rmsnorm_fwd_f32 if dtype == "f32" else binding.rmsnorm_fwd_bf16
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):                       # plan each shape before capture
        for x, y in zip(xd, ys):
            fwd(x, wd, y, 1e-5)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for x, y in zip(xd, ys):
            fwd(x, wd, y, 1e-5)
    for y in ys:
        y.zero_()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for k, (x, y) in enumerate(zip(xs, ys)):
        compare(y, oracle_for(x, w, 1e-5), f"graph replay {k}")
    # new inputs in the same buffers are picked up by the next replay
    xd[0].copy_(workloads.make_random((128, H), dtype, 399).cuda())
    g.replay()
    torch.cuda.synchronize()
    compare(ys[0], oracle_for(xd[0].cpu(), w, 1e-5), "graph replay after new input")
