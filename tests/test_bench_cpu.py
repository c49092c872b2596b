"""Host logic of the benchmark that needs no GPU: the kernel-source fingerprint
that keys the committed ncu traffic records."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_fingerprint_ignores_comments_and_whitespace_only(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("int f(int x) { return x + 1; } // one\n/* block\n comment */\n")
    b = tmp_path / "b.cu"
    b.write_text("int f(int x)\n{\n    return x + 1;   // another comment\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) { return x + 2; }\n")
    assert bench.source_fingerprint(str(a)) == bench.source_fingerprint(str(b))
    assert bench.source_fingerprint(str(a)) != bench.source_fingerprint(str(c))


def test_committed_traffic_records_match_the_kernel_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    for kernel, rec in d.items():
        assert bench.source_fingerprint(os.path.join(ROOT, rec["source"])) == rec["source_fingerprint"], kernel
