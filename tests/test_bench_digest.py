"""bench.py reports the committed DRAM-traffic capture only while the kernel
sources match the digest recorded with it; comments do not count as a change,
code does."""
import bench


def test_comments_and_blank_lines_do_not_change_the_code():
    a = "int f(int x) {\n  return x + 1;  // add one\n}\n"
    b = "/* header\n   comment */\nint f(int x) {\n\n  return x + 1;\n}   \n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(a.replace("x + 1", "x + 2"))


def test_committed_capture_matches_the_sources():
    # the traffic summary under profiles/ is for the kernels in this tree
    assert bench.load_traffic("qwen2_7b", "backward") is not None
    assert bench.load_traffic("qwen2_7b", "forward") is not None
    assert bench.load_traffic("qwen3_8b", "backward") is None
