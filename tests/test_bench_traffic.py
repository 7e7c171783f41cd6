"""bench.py's traffic record: DRAM bytes summed from an ncu --csv capture,
stored under the source digest, and read back only while that digest holds.
CPU only; the capture is a small hand-written CSV in ncu's layout."""

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

HEADER = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
          '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
          '"Metric Value"\n')


def _row(launch, kernel, metric, unit, value):
    return (f'"{launch}","1","python3","127.0.0.1","{kernel}","1","13","(320, 1, 1)",'
            f'"(152, 1, 1)","0","10.3","Command line profiler metrics","{metric}","{unit}",'
            f'"{value}"\n')


@pytest.fixture
def bench_in_tmp(tmp_path, monkeypatch):
    import bench
    os.makedirs(tmp_path / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return bench, tmp_path


def test_one_launch_is_recorded_and_read_back(bench_in_tmp):
    bench, tmp = bench_in_tmp
    csv = tmp / "cap.csv"
    csv.write_text("==PROF== noise line\n" + HEADER +
                   _row(0, "fa_tc_kernel<128, 0, 0>", "dram__bytes_read.sum", "byte", "1,000,000") +
                   _row(0, "fa_tc_kernel<128, 0, 0>", "dram__bytes_write.sum", "Kbyte", "250") +
                   _row(0, "fa_tc_kernel<128, 0, 0>", "gpu__time_duration.sum", "ns", "5000"))
    e = bench.record_traffic(str(csv), "fa_tc", "W1", "ncu ...")
    assert (e["dram_bytes_read"], e["dram_bytes_write"]) == (1_000_000, 250_000)
    assert e["dram_bytes_per_launch"] == 1_250_000 and e["launches_summed"] == 1
    assert bench.load_traffic("fa_tc", "W1") == 1_250_000
    assert bench.load_traffic("fa_tc", "other") is None


def test_backward_step_sums_its_launches(bench_in_tmp):
    bench, tmp = bench_in_tmp
    csv = tmp / "cap.csv"
    body = HEADER
    for i, (r, w) in enumerate([(10, 1), (200, 30), (100, 20)]):
        body += _row(i, f"bwd_kernel_{i}", "dram__bytes_read.sum", "Mbyte", r)
        body += _row(i, f"bwd_kernel_{i}", "dram__bytes_write.sum", "Mbyte", w)
    csv.write_text(body)
    e = bench.record_traffic(str(csv), "fa_bwd", "W2", "")
    assert e["launches_summed"] == 3
    assert e["dram_bytes_per_launch"] == 361_000_000


def test_stale_digest_reads_as_unknown(bench_in_tmp):
    bench, tmp = bench_in_tmp
    csv = tmp / "cap.csv"
    csv.write_text(HEADER + _row(0, "k", "dram__bytes_read.sum", "byte", "8"))
    bench.record_traffic(str(csv), "fa_tc", "W3", "")
    path = tmp / "profiles" / "traffic.json"
    rec = json.loads(path.read_text())
    rec["fa_tc/W3"]["source_digest"] = "0" * 16
    path.write_text(json.dumps(rec))
    assert bench.load_traffic("fa_tc", "W3") is None


def test_capture_without_dram_metrics_is_rejected(bench_in_tmp):
    bench, tmp = bench_in_tmp
    csv = tmp / "cap.csv"
    csv.write_text(HEADER + _row(0, "k", "gpu__time_duration.sum", "ns", "8"))
    with pytest.raises(ValueError):
        bench.record_traffic(str(csv), "fa_tc", "W4", "")


def test_kernel_digest_follows_only_its_own_sources(tmp_path, monkeypatch):
    """Editing one kernel family's source leaves the other families'
    measurements valid; editing a shared header invalidates them all."""
    import shutil
    from exact_attention_24_gb300 import build
    csrc = tmp_path / "csrc"
    shutil.copytree(build.CSRC, csrc)
    monkeypatch.setattr(build, "CSRC", str(csrc))
    before = {k: build.kernel_digest(k) for k in build.KERNEL_SOURCES}
    with open(csrc / "fa_simt.cu", "a") as f:
        f.write("\n// edit\n")
    after = {k: build.kernel_digest(k) for k in build.KERNEL_SOURCES}
    assert after["fa_simt"] != before["fa_simt"]
    assert after["fa_tc"] == before["fa_tc"] and after["fa_bwd"] == before["fa_bwd"]
    with open(csrc / "device_common.cuh", "a") as f:
        f.write("\n// edit\n")
    shared = {k: build.kernel_digest(k) for k in build.KERNEL_SOURCES}
    assert all(shared[k] != after[k] for k in build.KERNEL_SOURCES)


def test_kernel_digest_does_not_depend_on_the_checkout_location(tmp_path, monkeypatch):
    """A copy of the tree at another path (as on another machine) has the same
    digests, so measurements recorded in one place stay valid in another."""
    import shutil
    from exact_attention_24_gb300 import build
    here = {k: build.kernel_digest(k) for k in build.KERNEL_SOURCES}
    csrc, inc = tmp_path / "pkg" / "csrc", tmp_path / "include"
    shutil.copytree(build.CSRC, csrc)
    shutil.copytree(build.INCLUDE, inc)
    monkeypatch.setattr(build, "CSRC", str(csrc))
    monkeypatch.setattr(build, "INCLUDE", str(inc))
    monkeypatch.setattr(build, "NVCC_FLAGS", [f.replace(build.ROOT + "/include", str(inc))
                                              for f in build.NVCC_FLAGS])
    assert any(str(inc) in f for f in build.NVCC_FLAGS)
    assert {k: build.kernel_digest(k) for k in build.KERNEL_SOURCES} == here
