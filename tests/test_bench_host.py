"""Host-side pieces of bench.py that need no GPU."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _digest_of(tmp_path, text):
    p = tmp_path / "k.cu"
    p.write_text(text)
    rel = os.path.relpath(p, bench.ROOT)
    return bench.sources_digest([rel])


def test_sources_digest_ignores_comments_but_not_code(tmp_path):
    base = _digest_of(tmp_path, "int f(int x) {  // add one\n  return x + 1;\n}\n")
    assert _digest_of(tmp_path, "/* a block\n comment */ int f(int x) {\n  return x + 1;  // other words\n}\n") == base
    assert _digest_of(tmp_path, "int f(int x) {\n  return x + 2;\n}\n") != base


def test_traffic_record_names_existing_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for kernel, e in rec.items():
        assert e["dram_bytes_per_launch"] > 0
        for rel in e["sources"]:
            assert os.path.exists(os.path.join(ROOT, rel)), rel
        assert os.path.exists(os.path.join(ROOT, e["summary"]))
