"""Host-side pieces of the benchmark that decide what a bench line reports:
the kernel-source hash that ties the committed DRAM-traffic figures to the
code they were measured on, the traffic lookup, and the dense peaks."""

import json
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

SRC = """// header comment
__global__ void k(int* x) {  /* block
  comment */ x[0] = 1;  // trailing
}
"""


def test_code_only_drops_comments_and_layout():
    reworded = SRC.replace("header comment", "another header").replace("trailing", "other")
    relaid = SRC.replace("x[0] = 1;", "x[0]  =\n    1;")
    assert bench._code_only(SRC) == bench._code_only(reworded) == bench._code_only(relaid)
    assert bench._code_only(SRC) != bench._code_only(SRC.replace("x[0] = 1", "x[0] = 2"))
    assert "comment" not in bench._code_only(SRC)


@pytest.fixture()
def fake_root(tmp_path, monkeypatch):
    for f in bench.KERNEL_SOURCES:
        os.makedirs(tmp_path / os.path.dirname(f), exist_ok=True)
        shutil.copy(os.path.join(ROOT, f), tmp_path / f)
    os.makedirs(tmp_path / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def _write_traffic(root, entries):
    with open(root / "profiles" / "traffic.json", "w") as f:
        json.dump(entries, f)


def test_traffic_is_reported_only_for_the_source_it_was_measured_on(fake_root):
    h = bench.kernel_hash()
    _write_traffic(fake_root, {"w": {"bytes_per_launch": 123.0, "kernel_hash": h},
                               "old": {"bytes_per_launch": 456.0, "kernel_hash": "0" * 16}})
    assert bench.load_traffic("w") == 123.0
    assert bench.load_traffic("old") is None       # measured on other code
    assert bench.load_traffic("missing") is None
    # A comment-only edit keeps the figure; a code edit voids it.
    src = fake_root / bench.KERNEL_SOURCES[0]
    text = src.read_text()
    src.write_text("// a new comment line\n" + text)
    assert bench.kernel_hash() == h and bench.load_traffic("w") == 123.0
    src.write_text(text + "\nstatic int zyfa_extra_symbol;\n")
    assert bench.kernel_hash() != h and bench.load_traffic("w") is None


def test_no_traffic_file_means_no_figure(fake_root):
    assert bench.load_traffic("w") is None


def test_committed_traffic_entries_are_sums_of_read_and_write():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    for name, e in t.items():
        total = (e["dram_read_MB"] + e["dram_write_MB"]) * 1e6
        assert abs(e["bytes_per_launch"] - total) <= 1.0, name


def test_dense_peaks():
    peaks = {"bf16_tflops": 1915.0}
    assert bench.tensor_peak("bf16", peaks) == 1915.0
    assert bench.tensor_peak("fp8", peaks) == 3830.0
