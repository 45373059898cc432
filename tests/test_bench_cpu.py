"""Host-side logic of bench.py (no GPU): the roofline each workload is
judged against, the algorithmic work per launch it is computed from, and
the DRAM traffic it reports, which must come from an ncu capture of the
kernel source the workload's plan runs now."""
from __future__ import annotations

import os
import sys

import pytest

import synth
import tiled_gemm_codegen_gb300 as tg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

PEAKS = {"hbm_gbs": 6769.4, "bf16_tflops": 1978.8, "bf16_tflops_sustained": 1700.0}


@pytest.fixture(scope="module")
def lib():
    tg.load()
    return True


def test_algorithmic_work_per_launch():
    for w in synth.WORKLOADS.values():
        assert w.flops == 2 * w.batch * w.M * w.N * w.K
        assert w.bytes_moved == w.batch * (2 * w.M * w.K + 2 * w.K * w.N + 4 * w.M * w.N)


def test_roofline_bound_of_each_workload():
    """HBM when the algorithmic flop per byte is below the ridge point of
    the measured peaks (~292), else the bf16 tensor peak."""
    want = {"square_4096": "tensor", "ragged_4097x4095x4100": "tensor", "batched_64x384x640x1000": "hbm",
            "skinny_64x28672x8192": "hbm", "ragged_197x131x77": "hbm"}
    for name, w in synth.WORKLOADS.items():
        r = bench.roofline_of(w, 0.1, PEAKS, "measured")
        assert r["bound"] == want[name], name
        # (the line rounds TFLOP/s to 0.01, GB/s to 0.1 and fractions to 1e-4)
        if r["bound"] == "tensor":
            tf = w.flops / 1e-4 / 1e12
            assert r["achieved"] == pytest.approx(tf, rel=1e-3, abs=0.006)
            assert r["frac"] == pytest.approx(tf / PEAKS["bf16_tflops"], rel=1e-3, abs=6e-5)
        else:
            gbs = w.bytes_moved / 1e-4 / 1e9
            assert r["achieved"] == pytest.approx(gbs, rel=1e-3, abs=0.06)
            assert r["frac"] == pytest.approx(gbs / PEAKS["hbm_gbs"], rel=1e-3, abs=6e-5)


def test_traffic_comes_from_a_capture_of_the_current_kernel(lib):
    """Every workload's DRAM traffic is on file for the source hash of the
    kernel its default plan runs (the direct-load kernel for the small one),
    so the bench line never reports a figure taken on other code."""
    for name, w in synth.WORKLOADS.items():
        lead = w.batch
        info = tg.plan(w.M, w.N, w.K, lead, sm_count=152)
        direct = info["direct"] == 2
        traffic = bench.measured_traffic(name, direct)
        assert isinstance(traffic, int) and traffic > 0, (name, direct)
        # a capture keyed to the other kernel's sources does not count
        assert bench.measured_traffic(name, not direct) is None, name


def test_profile_named_in_the_traffic_file_exists():
    with open(bench.TRAFFIC_FILE) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            assert len(parts) == 4, line
            assert os.path.exists(os.path.join(ROOT, "profiles", parts[3])), parts[3]
