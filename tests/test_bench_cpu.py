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


def test_fingerprint_follows_in_tree_includes(tmp_path):
    """A change in a header the kernel source includes (a shared device
    function) changes the fingerprint; system headers are not followed."""
    h = tmp_path / "common.cuh"
    h.write_text("inline int g(int x) { return x * 2; }\n")
    a = tmp_path / "a.cu"
    a.write_text('#include <stdint.h>\n#include "common.cuh"\nint f(int x) { return g(x); }\n')
    before = bench.source_fingerprint(str(a))
    h.write_text("inline int g(int x) { return x * 2; }  // a comment only\n")
    assert bench.source_fingerprint(str(a)) == before
    h.write_text("inline int g(int x) { return x * 3; }\n")
    assert bench.source_fingerprint(str(a)) != before
