"""bench.py's CPU baseline: the oracle timed on the host's cores, and for the
small workloads also on one core with single-threaded BLAS.  CPU only."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_small_workload_adds_a_one_core_run():
    import bench
    from exact_attention_24_gb300.workloads import C1
    rec = bench.cpu_baseline(C1, 0.3)
    assert rec["kind"] == "oracle" and rec["value"] > 0
    assert rec["cores"] == len(os.sched_getaffinity(0))
    one = rec["one_core"]
    assert "error" not in one, one
    assert one["cores"] == 1 and one["value"] > 0 and "one_core" not in one
    assert one["host"]["blas_threads"] == {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1",
                                           "MKL_NUM_THREADS": "1"}


def test_large_workload_has_no_one_core_run():
    import bench
    from exact_attention_24_gb300.workloads import C3
    assert C3.flops() >= bench.ONE_CORE_MAX_FLOPS
    rec = bench.cpu_baseline(C3, 0.2)
    assert "one_core" not in rec
