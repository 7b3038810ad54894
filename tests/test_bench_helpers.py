"""The bench's bookkeeping, on the CPU: the key under which a workload's
per-launch DRAM bytes are recorded, the rule that a record counts only while
the kernel sources still hash to the digest it was taken on (else the bench
reports no traffic), the scaling of a record taken on a scaled-down
instance, and the shape of the committed records."""
import json
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DEFAULT_WORKLOADS = ("pr1_fp32", "llama3_8b", "long_context", "ragged_slots", "paged")


def test_traffic_key_names_the_operation():
    assert bench.traffic_key("paged", False, False, 0, {}) == "paged"
    assert bench.traffic_key("llama3_8b", True, False, 0, {}) == "llama3_8b/attend"
    assert bench.traffic_key("paged", False, True, 3, {}) == "paged/e4m3/q3"
    assert bench.traffic_key("llama3_8b", False, False, 0, {"window": 64}) == "llama3_8b/mods"


def _fake_root(tmp_path, entries, sources):
    csrc = tmp_path / "gqa_kv_cache_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name, text in sources.items():
        (csrc / name).write_text(text)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(entries))
    return str(tmp_path)


def test_traffic_record_counts_only_on_its_own_sources(tmp_path, monkeypatch):
    sources = {"k.cuh": "kernel body v1\n", "k.cu": "launch\n"}
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _fake_root(tmp_path, {}, sources)
    sha = bench.sources_sha(["k.cuh", "k.cu"])
    entries = {"tc_decode_kernel": {
        "whole": {"sources": ["k.cuh", "k.cu"], "sources_sha": sha, "bytes_per_launch": 1234},
        "scaled": {"sources": ["k.cuh", "k.cu"], "sources_sha": sha, "bytes_over_algorithmic": 1.5},
        "stale": {"sources": ["k.cuh", "k.cu"], "sources_sha": "0" * 16, "bytes_per_launch": 99}}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(entries))
    assert bench.traffic_for("tc_decode_kernel", "whole", 10_000) == 1234
    # a capture of a scaled-down instance scales by the launch's algorithmic bytes
    assert bench.traffic_for("tc_decode_kernel", "scaled", 10_000) == 15_000
    assert bench.traffic_for("tc_decode_kernel", "stale", 10_000) is None
    assert bench.traffic_for("tc_decode_kernel", "missing", 10_000) is None
    assert bench.traffic_for("unit_decode_kernel", "whole", 10_000) is None
    # any change to a listed source retires the record
    (tmp_path / "gqa_kv_cache_gb300" / "csrc" / "k.cuh").write_text("kernel body v2\n")
    assert bench.traffic_for("tc_decode_kernel", "whole", 10_000) is None


def test_committed_records_cover_the_default_workloads():
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    have = {key for kern in d.values() for key in kern}
    for w in DEFAULT_WORKLOADS:
        assert w in have, w
    csrc = os.path.join(ROOT, "gqa_kv_cache_gb300", "csrc")
    for kern, recs in d.items():
        for key, e in recs.items():
            assert e["sources"] and all(os.path.exists(os.path.join(csrc, n)) for n in e["sources"]), (kern, key)
            assert len(e["sources_sha"]) == 16
            assert ("bytes_per_launch" in e) != ("bytes_over_algorithmic" in e), (kern, key)
            # a launch moves at least its algorithmic bytes, and never many times them
            ratio = e["capture_bytes"] / e["capture_algorithmic_bytes"]
            assert 1.0 <= ratio < 2.5, (kern, key, ratio)
            if "bytes_over_algorithmic" in e:
                assert e["bytes_over_algorithmic"] == pytest.approx(ratio, rel=1e-4)
