"""Host-side pieces of the benchmark that need no GPU: the DRAM-traffic field
taken from the committed ncu captures, which must go null once a source file of
the captured kernel changes, and the integrity of those committed entries."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _tree(tmp_path, files):
    csrc = tmp_path / "tensor_core_dense_tn_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name, text in files.items():
        (csrc / name).write_text(text)
    (tmp_path / "profiles").mkdir()
    return csrc


def test_traffic_follows_the_hash_of_its_own_sources(tmp_path, monkeypatch):
    """An entry stays valid while its own sources are unchanged and goes null
    when one of them changes; a change to a file it does not list leaves it."""
    csrc = _tree(tmp_path, {"a.cu": "kernel a\n", "b.cu": "kernel b\n", "common.cuh": "shared\n"})
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    entries = {
        "workload A": {"sources": ["a.cu", "common.cuh"], "dram_bytes_per_launch": 111},
        "workload B": {"sources": ["b.cu", "common.cuh"], "dram_bytes_per_launch": 222},
    }
    for e in entries.values():
        e["source_hash"] = bench.kernel_source_hash(tuple(e["sources"]))
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(entries))

    assert bench.profiled_traffic("workload A") == 111
    assert bench.profiled_traffic("workload B") == 222
    assert bench.profiled_traffic("no such workload") is None

    (csrc / "b.cu").write_text("kernel b, changed\n")
    assert bench.profiled_traffic("workload A") == 111
    assert bench.profiled_traffic("workload B") is None

    (csrc / "common.cuh").write_text("shared, changed\n")
    assert bench.profiled_traffic("workload A") is None


def test_missing_or_broken_capture_file_gives_null(tmp_path, monkeypatch):
    _tree(tmp_path, {"a.cu": "x\n"})
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("anything") is None
    (tmp_path / "profiles" / "ncu_traffic.json").write_text("{not json")
    assert bench.profiled_traffic("anything") is None


def test_committed_entries_are_consistent():
    """Every committed capture names sources that exist, a hash of the right
    form, and a per-launch total equal to its read + write bytes."""
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        d = json.load(f)
    entries = {k: v for k, v in d.items() if isinstance(v, dict)}
    assert entries
    for name, e in entries.items():
        assert e["sources"], name
        for src in e["sources"]:
            assert os.path.exists(os.path.join(ROOT, "tensor_core_dense_tn_gb300", "csrc", src)), (name, src)
        assert len(e["source_hash"]) == 16 and int(e["source_hash"], 16) >= 0, name
        assert e["dram_bytes_per_launch"] == e["dram_read_bytes"] + e["dram_write_bytes"], name
        assert "--clock-control none" in e["command"], name


def test_clock_summary_reads_only_the_timed_window():
    """Median SM clock, the maximum clock and every active slowdown reason of
    the samples inside [t0, t1]; samples outside it and malformed lines do not
    count."""
    c = bench.ClockSampler(0)
    na, a = "Not Active", "Active"
    c.lines = [
        (9.0, f"0, 1000, 2070, 500.0, 0x1, {na}, {na}, {a}, {na}"),        # before the window
        (10.0, f"0, 2070, 2070, 1300.5, 0x0, {na}, {na}, {na}, {na}"),
        (10.1, f"0, 1965, 2070, 1398.0, 0x4, {na}, {na}, {na}, {a}"),
        (10.2, "0, [N/A], 2070, 1390.0, 0x4, Not Active"),                  # malformed
        (10.3, f"0, 1950, 2070, 1401.0, 0x4, {na}, {na}, {na}, {a}"),
        (12.0, f"0, 900, 2070, 300.0, 0x8, {a}, {na}, {na}, {na}"),         # after the window
    ]
    s = c.summary(10.0, 10.3)
    assert s == {"sm_mhz": 1965.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert c.summary(20.0, 21.0) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
