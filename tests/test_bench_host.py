"""Host-side pieces of bench.py, without a GPU: the kernel-source hash that
ties a committed ncu summary to the code it was captured on."""
import bench


def test_source_hash_ignores_comments_and_whitespace(tmp_path):
    a = tmp_path / "a.cuh"
    a.write_text("int f(int x) {\n  return x + 1;  // add one\n}\n/* note */\n")
    b = tmp_path / "b.cuh"
    b.write_text("int f(int x){ return x+1; }\n// another comment\n")
    c = tmp_path / "c.cuh"
    c.write_text("int f(int x){ return x+2; }\n")
    ha = bench.kernel_source_hash([str(a)])
    assert ha == bench.kernel_source_hash([str(b)])
    assert ha != bench.kernel_source_hash([str(c)])

