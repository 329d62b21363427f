"""Host logic of bench.py that needs no GPU: the recorded ncu traffic is used only for the
kernel code it was measured on."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _sources(tmp_path, monkeypatch, body):
    """Kernel "k" made of one file k.cu with this body."""
    (tmp_path / "k.cu").write_text(body)
    monkeypatch.setattr(bench, "CSRC", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", {"k": ("k.cu",)})


def test_source_hash_ignores_comments_and_spacing(tmp_path, monkeypatch):
    _sources(tmp_path, monkeypatch, "int a = 1;  // one\nint b = 2;\n")
    h0 = bench.kernel_source_hash("k")
    _sources(tmp_path, monkeypatch, "// header\nint  a = 1;\n\nint b = 2;   // two\n")
    assert bench.kernel_source_hash("k") == h0
    _sources(tmp_path, monkeypatch, "int a = 1;\nint b = 3;\n")
    assert bench.kernel_source_hash("k") != h0


def test_recorded_traffic_needs_matching_code(tmp_path, monkeypatch):
    _sources(tmp_path, monkeypatch, "int a = 1;\n")
    rec = {"entries": {"k@w": {"dram_bytes_per_launch": 123, "source_hash": bench.kernel_source_hash("k")}}}
    f = tmp_path / "t.json"
    f.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("w", "k") == 123
    assert bench.recorded_traffic("other", "k") is None
    _sources(tmp_path, monkeypatch, "int a = 2;\n")
    assert bench.recorded_traffic("w", "k") is None


def test_committed_traffic_record_is_consistent():
    """The committed launch-list record: read + write = total per launch, and the bench reports
    it exactly when it was taken on the kernel code as it is now (else null)."""
    with open(bench.TRAFFIC_FILE) as fh:
        rec = json.load(fh)
    for key, e in rec["entries"].items():
        # per-launch averages, each truncated to whole bytes
        assert abs(e["dram_bytes_per_launch"] - e["dram_read_bytes_per_launch"] - e["dram_write_bytes_per_launch"]) <= 1
        kernel, workload = key.split("@")
        want = e["dram_bytes_per_launch"] if e["source_hash"] == bench.kernel_source_hash(kernel) else None
        assert bench.recorded_traffic(workload, kernel) == want
