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
