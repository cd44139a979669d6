"""bench.py's reference arm runs the oracle on the host (CPU only) and prints
one JSON line with the contract's keys; its helpers read the committed
profiles correctly."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "c1",
                          "--steps", "3", "--warmup", "3"], cwd=ROOT, capture_output=True,
                         text=True, timeout=600, check=True).stdout.strip().splitlines()
    assert len(out) == 1
    d = json.loads(out[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["steps"] == 3 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["cores"] == bench.host_cores()
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("c1")


def test_cpu_baseline_is_row_parallel_with_single_thread_beside_it():
    from row_wise_rmsnorm_fwd_gb300 import workloads
    d = bench.cpu_baseline_line(workloads.WORKLOADS["c1"])
    assert d["kind"] == "oracle" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cores"] == bench.host_cores() and "seconds" not in d
    one = d["single_thread"]
    assert one["cores"] == 1 and one["value"] > 0 and "single-thread" in one["sample"]


def test_reference_arm_softmax_workload():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                          "sm_attn_f32", "--steps", "3", "--warmup", "3"], cwd=ROOT,
                         capture_output=True, text=True, timeout=600, check=True).stdout
    d = json.loads(out.strip().splitlines()[-1])
    assert d["metric"].startswith("row softmax") and d["value"] > 0


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--warmup", "2"],
                       cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0


def test_committed_profiles_parse():
    """Every committed per-kernel summary names its source files, and the
    traffic of a profile is returned only while their hash matches."""
    pdir = os.path.join(ROOT, "profiles")
    found = 0
    for name in os.listdir(pdir):
        if not name.endswith(".txt") or name.startswith("launches"):
            continue
        text = open(os.path.join(pdir, name)).read()
        head = text.splitlines()[0].split()      # "ncu summary: <kernel> on workload <w>"
        kernel, workload = head[2], head[-1]
        assert name == f"{kernel}_{workload}.txt"
        assert "kernel_source_files:" in text and "traffic_bytes_per_launch:" in text
        assert "ncu " in text and "--clock-control none" in text
        found += 1
        t = bench.profiled_traffic(workload, kernel)
        assert t is None or t > 0
    assert found >= 6


def _args(**kw):
    import argparse
    base = dict(workload="c5a", rows=0, secondary=None, path="auto", cluster=0, grid=0,
                threads=0, chunk=0, stages=0, epilogue="none")
    base.update(kw)
    return argparse.Namespace(**base)


def test_secondary_workloads_only_on_the_default_run():
    from row_wise_rmsnorm_fwd_gb300 import workloads
    names = bench.secondary_names(_args())
    assert names == list(bench.SECONDARY_DEFAULT)
    assert {"c4", "c5b"} <= set(names)
    assert all(n in workloads.WORKLOADS for n in names)
    assert bench.secondary_names(_args(workload="c4")) == []
    assert bench.secondary_names(_args(rows=1024)) == []
    assert bench.secondary_names(_args(path="twopass")) == []
    assert bench.secondary_names(_args(secondary="none")) == []
    assert bench.secondary_names(_args(workload="c1", secondary="c4,c5b")) == ["c4", "c5b"]


def test_roofline_block_labels_the_copy_peak_and_the_nominal_fraction():
    r = bench.roofline_block(6000.0, 6768.8, "measured", None)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["frac"] - 6000.0 / 6768.8) < 1e-12
    assert abs(r["frac_of_nominal"] - 6000.0 / bench.NOMINAL_HBM_GBS) < 1e-12
    assert "copy peak" in r["peak_source"]
