"""The committed ncu evidence matches the sources: every traffic.json entry
names an existing summary under profiles/ and carries the sha256 of the
current sources of its mode's kernel (bench.py reports an entry's DRAM
traffic only then), and each summary gives the command that made it."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def _entries():
    d = json.load(open(os.path.join(PROFILES, "traffic.json")))
    return {k: v for k, v in d.items() if isinstance(v, dict)}


def _mode(key):
    for m in ("greedy", "ragged", "truncated", "draft_logits"):
        if key.endswith("_" + m):
            return key[: -len(m) - 1], m
    return key, "sampled"


def test_traffic_entries_match_current_sources():
    entries = _entries()
    assert entries
    for key, e in entries.items():
        workload, mode = _mode(key)
        assert workload in bench.workloads.CONFIGS, key
        assert e["kernel_source_sha256"] == bench.kernel_source_hash(mode), (
            f"{key}: captured on other sources of the {mode} kernel; re-capture it")
        assert bench.profile_traffic(workload, mode) == float(e["dram_bytes_per_launch"])
        assert 0.9 < e["dram_bytes_per_launch"] / e["algorithmic_bytes"] < 2.0, key


def test_summaries_exist_and_give_their_command():
    for key, e in _entries().items():
        path = os.path.join(PROFILES, e["summary"])
        text = open(path).read()
        assert "ncu " in text and "--clock-control none" in text, e["summary"]
        assert "bench.py" in text, e["summary"]
