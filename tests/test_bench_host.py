"""Host-side parts of bench.py that need no GPU: the oracle's CPU baseline sampler, its
single-thread run and the BLAS thread report."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from ragged_grouped_gemm_device_gb300 import workloads as W  # noqa: E402


def test_oracle_sampler_counts_the_rows_it_timed():
    wl = W.make("toy")
    flops, elapsed, desc = bench.OracleSampler(wl).run(10.0)
    # the toy workload is small enough to be sampled whole: all 10 rows, forward + backward
    assert flops == 18.0 * 10 * wl.d * wl.h and elapsed > 0
    assert "4 of 4 experts (10 of 10 rows)" in desc


def test_single_thread_sample_runs_with_one_blas_thread():
    r = bench.oracle_single_thread("toy", 0.1)
    assert "error" not in r, r
    assert r["blas_threads"] == 1 and r["value"] > 0
    assert bench.blas_threads() >= 1


def test_oracle_rates_time_forward_and_backward_separately():
    r = bench.oracle_rates(W.make("toy"), 10.0)
    assert set(r) == {"fwd", "fwd_bwd"}
    for mode in r.values():
        assert mode["experts"] == 4 and mode["rows"] == 10 and mode["tflops"] > 0


def test_kernel_rooflines_bound_by_intensity_against_the_ridge():
    peaks = {"bf16_tflops": 2000.0, "hbm_gbs": 8000.0}      # ridge 250 FLOP/B
    work = {"gemm": (1e12, 1e9, 1e12),                     # 1000 FLOP/B: tensor-bound
            "wgrad": (8e11, 5e9, 1.6e12),                  # 160 FLOP/B: memory-bound
            "gather": (0, 6e8, 0)}
    per_call = {"gemm": 1.0, "wgrad": 1.25, "gather": 0.1}
    br, dom, roof = bench.kernel_rooflines(per_call, work, peaks, "test")
    assert br["gemm"]["bound"] == "tensor" and br["wgrad"]["bound"] == "hbm" and br["gather"]["bound"] == "hbm"
    assert dom == "wgrad" and roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert abs(roof["achieved"] - 5e9 / 1.25e-3 / 1e9) < 1e-6 and abs(roof["frac"] - 0.5) < 1e-9
    assert abs(roof["mma_executed_tflops"] - 1280.0) < 1e-6       # both halves executed
    assert abs(br["gemm"]["floor_ms"] - 0.5) < 1e-9 and abs(br["gemm"]["frac"] - 0.5) < 1e-9
    w = bench.kernel_work(131072, 16384, 8, 256, 2048, 512)
    assert w["wgrad_dual"][0] == 6.0 * 131072 * 2048 * 512 and w["wgrad_dual"][2] == 2 * w["wgrad_dual"][0]


def test_traffic_is_taken_only_from_captures_of_the_current_sources():
    t = bench.load_traffic()
    assert set(t) <= {"up_swiglu", "down", "down_dgrad_swiglu", "up_dgrad", "wgrad_dual"}
    assert all(v > 0 for v in t.values())
