"""Host-side helpers of bench.py on the CPU: the code digest that ties the committed attention
capture to the kernel source, and the traffic lookup built on it."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _write(tmp_path, name, text):
    p = tmp_path / name
    p.write_text(text)
    return str(p)


def test_code_digest_ignores_comments_and_whitespace(tmp_path):
    a = _write(tmp_path, "a.cu", "int f(int x) {\n  return x + 1;  // one more\n}\n/* block\n comment */\n")
    b = _write(tmp_path, "b.cu", "// a header comment\nint  f(int x)\n{\n\treturn x + 1;\n}\n")
    c = _write(tmp_path, "c.cu", "int f(int x) {\n  return x + 2;\n}\n")
    assert bench.code_digest([a]) == bench.code_digest([b])
    assert bench.code_digest([a]) != bench.code_digest([c])
    assert len(bench.code_digest([a])) == 16


def test_traffic_lookup_follows_the_committed_capture():
    """The committed capture's digest matches the committed attention source, so the 128K bf16
    workload gets its traffic; other workloads and precisions get none."""

    class W:
        name, Hq, Hkv = "llama128k", 32, 8

    t = bench.profile_traffic(W, "bf16")
    assert isinstance(t, int) and t > 0, (
        "the attention kernel's code changed since profiles/bsattn_llama128k_h4.md was captured: "
        "recapture it (the command is in the file) and update its digest and traffic lines")
    assert bench.profile_traffic(W, "q8") is None

    class V:
        name, Hq, Hkv = "cogvideox", 30, 30

    assert bench.profile_traffic(V, "bf16") is None
