"""The committed ncu summaries describe the kernels as they are built now.

profiles/traffic.json records, per profiled kernel, the DRAM bytes of one
launch and a hash of the source files that kernel is compiled from; the
benchmark reports that traffic only while the hash matches.  These checks
keep the summaries from going stale silently: every entry names existing
sources whose hash matches, and every entry has its markdown summary.
"""
import hashlib
import json
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def _entries():
    with open(os.path.join(PROFILES, "traffic.json")) as f:
        return json.load(f)


def test_traffic_entries_match_the_sources():
    stale = []
    for key, e in _entries().items():
        digest = hashlib.sha256()
        for rel in e["source_files"]:
            with open(os.path.join(ROOT, rel), "rb") as f:
                digest.update(f.read())
        if digest.hexdigest()[:16] != e["source_sha256_16"]:
            stale.append(key)
    assert not stale, f"re-profile these kernels (sources changed since the capture): {stale}"


def test_traffic_entries_are_sane():
    for key, e in _entries().items():
        assert e["dram_bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_write"], key
        assert e["dram_bytes_per_launch"] > 0 and e["gpu_time_ns_cold"] > 0, key
        assert "--clock-control none" in e["command"], key


def test_every_entry_has_its_summary():
    names = set(os.listdir(PROFILES))
    for key in _entries():
        assert f"{key}.md" in names, f"profiles/{key}.md is missing"


def test_summaries_are_text_and_small():
    for name in os.listdir(PROFILES):
        path = os.path.join(PROFILES, name)
        assert name.endswith((".md", ".txt", ".json")), name
        assert os.path.getsize(path) < 64 * 1024, name
