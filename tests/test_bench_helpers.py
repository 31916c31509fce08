"""bench.py's host-side helpers on CPU: the kernel-source fingerprint that keys
the committed DRAM-traffic record, and the record lookup.  No GPU needed."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_and_layout():
    a = "int x = 1;  // one\n/* block\n comment */ float y = 2.0f;\n"
    b = "int x = 1;\nfloat   y = 2.0f; // changed comment\n"
    assert bench._code_only(a) == bench._code_only(b)


def test_code_only_keeps_literals_and_code():
    src = 'asm("mov.u32 %0, 1; // not a comment");\nconst char *s = "/* kept */";\nchar c = \'"\';'
    out = bench._code_only(src)
    assert "// not a comment" in out and "/* kept */" in out and "'\"'" in out
    assert bench._code_only("int x = 1;") != bench._code_only("int x = 2;")


def test_csrc_hash_is_stable_and_hex():
    h1, h2 = bench.csrc_hash(), bench.csrc_hash()
    assert h1 == h2 and len(h1) == 16
    int(h1, 16)


def test_recorded_traffic_needs_matching_kernel_and_sources(monkeypatch, tmp_path):
    prof = tmp_path / "profiles"
    prof.mkdir()
    rec = {"w": {"kernel": "k", "csrc_hash": "a" * 16, "dram_bytes_per_launch": 123}}
    (prof / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "csrc_hash", lambda: "a" * 16)
    assert bench.recorded_traffic("w", "k") == 123
    assert bench.recorded_traffic("w", "other_kernel") is None
    assert bench.recorded_traffic("other_workload", "k") is None
    monkeypatch.setattr(bench, "csrc_hash", lambda: "0" * 16)
    assert bench.recorded_traffic("w", "k") is None      # sources changed since the capture
