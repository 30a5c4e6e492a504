"""bench.py's host logic, on CPU: the byte accounting behind every roofline
figure, the workload table, and the source hash that ties a recorded ncu
DRAM-traffic figure to the code it was measured on."""
from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

PN3T, PN4T = 124, 125
LAYER = [(PN3T, 5120, 6144), (PN3T, 5120, 17408), (PN3T, 5120, 17408), (PN4T, 5120, 1024),
         (PN4T, 5120, 1024), (PN4T, 6144, 5120), (PN4T, 17408, 5120)]      # (type, K, N)


def test_algorithmic_bytes_at_the_pages_widths():
    # a PN row is K / bpb blocks of 34 bytes: 2176 B (pn3t, K = 5120) and
    # 9248 B (pn4t, K = 17408); x is fp16 [M][K] and y fp32 [M][N]
    assert bench.algorithmic_bytes([(PN3T, 5120, 17408)], 1) == 17408 * 2176 + 2 * 5120 + 4 * 17408
    assert bench.algorithmic_bytes([(PN4T, 17408, 5120)], 1) == 5120 * 9248 + 2 * 17408 + 4 * 5120
    # the layer's packed weights alone: 158,760,960 bytes
    assert bench.algorithmic_bytes(LAYER, 0) == 158_760_960
    # bits per weight 3.40 / 4.25: 34 bytes per 80 / 64 weights
    assert bench.algorithmic_bytes([(PN3T, 80, 1)], 0) * 8 / 80 == 3.4
    assert bench.algorithmic_bytes([(PN4T, 64, 1)], 0) * 8 / 64 == 4.25
    # x and y scale with M
    one, eight = bench.algorithmic_bytes(LAYER, 1), bench.algorithmic_bytes(LAYER, 8)
    assert eight - one == 7 * sum(2 * K + 4 * N for _, K, N in LAYER)


def test_workloads_and_their_kernels():
    assert bench.workload(1)[1:] == ([(PN3T, 5120, 17408)], 1)
    assert bench.workload(4)[1:] == (LAYER, 8)
    assert bench.workload(5)[2] == 16
    # --m runs a workload's tensors at another M; the prefill workload keeps its own
    name, tensors, M = bench.workload(4, 2)
    assert tensors == LAYER and M == 2 and "M=2" in name
    assert bench.workload(6, 8)[2] == 4096
    for bad in (17, -1):
        with pytest.raises(SystemExit):
            bench.workload(3, bad)
    assert [bench.kernel_of(c) for c in range(7)] == ["stream"] * 4 + ["tc"] * 2 + ["prefill"]


def test_code_only_ignores_comments_and_layout():
    a = 'int f(int x) {  // the answer\n    return x + 42; /* block\n comment */ }\n'
    b = 'int f(int x) {\n  return x + 42;\n}  // another comment\n'
    assert bench.code_only(a) == bench.code_only(b)
    # a change to the code is seen; comment markers inside string literals are code
    assert bench.code_only(a) != bench.code_only(a.replace("42", "43"))
    s = 'const char* p = "http://x /* y */"; // z\n'
    assert bench.code_only(s) == 'const char* p = "http://x /* y */";'


def test_kernel_source_hash_is_stable_and_per_kernel():
    h = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    assert h == {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    assert len(set(h.values())) == len(h)
    assert all(len(v) == 16 and int(v, 16) >= 0 for v in h.values())


def test_recorded_traffic_only_for_the_current_sources(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(
        '{"records": ['
        '{"config": 1, "kernel": "gemv_stream_kernel<8>", "bytes_per_launch": 111, "source": "aaaa"},'
        '{"config": 4, "kernel": "gemv_tc_kernel<1>", "bytes_per_launch": 444, "source": "bbbb"}]}')
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: {"stream": "aaaa", "tc": "cccc"}.get(k, "x"))
    assert bench.recorded_traffic(1) == 111          # taken on the current stream sources
    assert bench.recorded_traffic(4) is None         # the batch kernel changed since
    assert bench.recorded_traffic(2) is None         # never captured
    (tmp_path / "profiles" / "traffic.json").write_text("not json")
    assert bench.recorded_traffic(1) is None


def test_committed_traffic_records_are_well_formed():
    import json
    with open(os.path.join(ROOT, bench.TRAFFIC_FILE)) as fh:
        records = json.load(fh)["records"]
    assert records
    for r in records:
        assert set(r) >= {"config", "kernel", "bytes_per_launch", "source"}
        assert r["config"] in range(7)
        assert int(r["bytes_per_launch"]) > 0 and len(r["source"]) == 16


def test_measured_peak_reads_the_driver_file(tmp_path, monkeypatch):
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6123.4, "bf16_tflops": 1800.0}')
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peak() == (pytest.approx(6123.4), "measured")
    (tmp_path / "MEASURED_PEAKS.json").unlink()
    assert bench.measured_peak() == (bench.FALLBACK_HBM_GBS, "fallback")
