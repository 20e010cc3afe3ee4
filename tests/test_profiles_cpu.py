"""The committed measurement evidence is consistent with itself: every DRAM
traffic record that bench.py reports names an ncu summary under profiles/
that exists, quotes the record's source hash and the command that made it,
and reads + writes add up to the bytes per launch.  (Whether a record is
current is decided at run time: bench.py reports traffic only while the
kernel's sources still hash the same.)"""
from __future__ import annotations

import json
import os

import pytest

import bench

PROFILES = os.path.join(bench.ROOT, "profiles")


def _records():
    with open(os.path.join(PROFILES, "traffic.json")) as f:
        d = json.load(f)
    return {k: v for k, v in d.items() if not k.startswith("_")}


def test_every_record_is_for_a_known_kernel():
    for kernel in _records():
        assert kernel in bench.KERNEL_SOURCES, kernel


@pytest.mark.parametrize("kernel", sorted(_records()))
def test_record_matches_its_summary(kernel):
    rec = _records()[kernel]
    assert rec["read"] + rec["write"] == rec["dram_bytes_per_launch"]
    path = os.path.join(PROFILES, rec["summary"])
    assert os.path.exists(path), rec["summary"]
    text = open(path).read()
    assert f"source_hash {rec['source_hash']}" in text
    assert "ncu " in text and "--clock-control none" in text
    # the summary states the read bytes the record carries, exactly or in MB to two decimals
    assert f"{rec['read']:,}" in text or f"{rec['read'] / 1e6:.2f} MB" in text


def test_profiles_hold_text_only():
    for name in os.listdir(PROFILES):
        assert name.endswith((".md", ".txt", ".json")), name
