"""bench.py's roofline traffic lookup, on CPU: a committed ncu DRAM figure is
reported only while the kernel sources still hash to the value stored with
it, so a figure taken on an older kernel is never reported for a newer one."""
from __future__ import annotations

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_figure_is_used_only_with_a_matching_source_hash(tmp_path, monkeypatch):
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps({
        "fresh": {"kernel_source_hash": bench.kernel_source_hash(bench.KERNEL_FILES), "dram_bytes_per_launch": 123},
        "stale": {"kernel_source_hash": "0000000000000000", "dram_bytes_per_launch": 456},
        "wide": {"kernel_source_hash": bench.kernel_source_hash(bench.WIDE_KERNEL_FILES), "dram_bytes_per_launch": 789},
    }))
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(path))
    assert bench.traffic_per_launch("fresh") == 123
    assert bench.traffic_per_launch("stale") is None
    assert bench.traffic_per_launch("absent") is None
    assert bench.traffic_per_launch("wide", bench.fwd_kernel_files(256)) == 789
    assert bench.traffic_per_launch("wide", bench.fwd_kernel_files(128)) is None  # another kernel's hash


def test_missing_or_broken_file_gives_no_figure(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "none.json"))
    assert bench.traffic_per_launch("target") is None
    bad = tmp_path / "bad.json"
    bad.write_text("{not json")
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(bad))
    assert bench.traffic_per_launch("target") is None


def test_hash_covers_every_listed_source():
    # each file the hash claims to cover exists and changes the hash
    for files in (bench.KERNEL_FILES, bench.WIDE_KERNEL_FILES, bench.BWD_KERNEL_FILES):
        for f in files:
            assert os.path.exists(os.path.join(bench.KERNEL_SOURCES, f)), f
        assert bench.kernel_source_hash(files) != bench.kernel_source_hash(files[1:])


def test_committed_figures_were_taken_on_the_kernels_as_they_stand():
    # every entry in the committed file still matches its kernel's sources, so
    # the bench reports each figure; reads + writes add up to the total
    with open(bench.PROFILE_TRAFFIC) as f:
        table = json.load(f)
    entries = {k: v for k, v in table.items() if isinstance(v, dict)}
    assert {"target", "bwd:target"} <= set(entries)
    for name, e in entries.items():
        if name.startswith("bwd:"):
            files = bench.BWD_KERNEL_FILES
        else:
            files = bench.fwd_kernel_files(bench.workloads.WORKLOADS[name].D)
        assert e["kernel_source_hash"] == bench.kernel_source_hash(files), name
        assert e["dram_bytes_per_launch"] == e["dram_bytes_read_per_launch"] + e["dram_bytes_write_per_launch"], name
        assert bench.traffic_per_launch(name, files) == e["dram_bytes_per_launch"], name
