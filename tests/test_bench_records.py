"""The measurement records the benchmark reads (CPU): the ncu traffic records
under profiles/ and the rule that a record is used only while the kernel's
source file is the one it was captured on."""
import json
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def test_traffic_records_name_existing_summaries():
    recs = json.load(open(bench.TRAFFIC_FILE))
    assert recs
    for key, rec in recs.items():
        workload, kernel = key.split(":")
        assert kernel in ("attend", "index_score"), key
        assert isinstance(rec["bytes_per_launch"], int) and rec["bytes_per_launch"] > 0, key
        assert re.fullmatch(r"[0-9a-f]{16}", rec["source_sha"]), key
        assert os.path.exists(os.path.join(ROOT, rec["from"])), (key, rec["from"])


def test_traffic_record_needs_the_captured_source(tmp_path):
    attend = bench.source_hash("long_context_sparse_21_b300/csrc/attend.cu")
    index = bench.source_hash("long_context_sparse_21_b300/csrc/index.cu")
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps({
        "w:attend": {"bytes_per_launch": 123, "source_sha": attend, "from": "x"},
        "w:index_score": {"bytes_per_launch": 456, "source_sha": "0" * 16 if index != "0" * 16 else "1" * 16,
                          "from": "x"},
    }))
    assert bench.traffic_record("w", "attend", str(f)) == 123
    assert bench.traffic_record("w", "L3.attend", str(f)) == 123      # per-layer stage names
    assert bench.traffic_record("w", "index_score", str(f)) is None   # the source changed since the capture
    assert bench.traffic_record("other", "attend", str(f)) is None    # no capture of that workload
    assert bench.traffic_record("w", "attend", str(tmp_path / "missing.json")) is None


def test_profiles_hold_short_text_summaries_only():
    for name in os.listdir(PROFILES):
        path = os.path.join(PROFILES, name)
        assert name.endswith(".md") or name == "traffic.json", name
        assert os.path.getsize(path) < 16 * 1024, name
