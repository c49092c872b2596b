"""Host logic of the benchmark that needs no GPU: the kernel-source fingerprint
that keys the committed ncu traffic records."""
import bench


def test_fingerprint_ignores_comments_and_whitespace_only(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("int f(int x) { return x + 1; } // one\n/* block\n comment */\n")
    b = tmp_path / "b.cu"
    b.write_text("int f(int x)\n{\n    return x + 1;   // another comment\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) { return x + 2; }\n")
    assert bench.source_fingerprint(str(a)) == bench.source_fingerprint(str(b))
    assert bench.source_fingerprint(str(a)) != bench.source_fingerprint(str(c))
