"""bench.py's host-side bookkeeping (no GPU): the FLOP counts behind every
TFLOP/s figure, and the rule that a DRAM-traffic figure from an ncu capture is
reported only while the kernel's sources are the ones that were captured."""

import os

import bench
from exact_attention_fattn_gb300 import workloads as W


def test_flop_counts():
    w = W.Workload("x", 2, 3, 256, 64, False)
    fwd, bwd = bench.flop_counts(w)
    # two GEMMs of 2 N^2 d FLOPs each per head; the backward does five
    assert fwd == 4.0 * 2 * 3 * 256 * 256 * 64
    assert bwd == 2.5 * fwd
    wc = W.Workload("x", 2, 3, 256, 64, True)
    assert bench.flop_counts(wc)[0] == fwd / 2


def _write(path, text):
    os.makedirs(os.path.dirname(path), exist_ok=True)
    with open(path, "w", encoding="utf-8") as f:
        f.write(text)


def test_source_hash_ignores_comments_and_layout(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _write(str(tmp_path / "a.cu"), "int f(int x) { return x + 1; }  // add one\n")
    _write(str(tmp_path / "b.cu"), "/* add one */\nint f(int x)\n{\n  return x + 1;\n}\n")
    _write(str(tmp_path / "c.cu"), "int f(int x) { return x + 2; }\n")
    _write(str(tmp_path / "d.cu"), "int g();\n")
    assert bench.source_hash(("a.cu",)) == bench.source_hash(("b.cu",))
    assert bench.source_hash(("a.cu",)) != bench.source_hash(("c.cu",))
    # several files: their concatenation, in order
    assert bench.source_hash(("a.cu", "d.cu")) != bench.source_hash(("a.cu",))
    assert bench.source_hash(("a.cu", "d.cu")) != bench.source_hash(("d.cu", "a.cu"))


def test_traffic_reported_only_for_the_captured_sources(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", {"fwd": ("k.cu", "s.h")})
    _write(str(tmp_path / "k.cu"), "__global__ void k() {}\n")
    _write(str(tmp_path / "s.h"), "int s();\n")
    h = bench.source_hash(("k.cu", "s.h"))
    _write(str(tmp_path / "profiles" / "dram_traffic.txt"),
           f"# kernel workload bytes hash\nfwd wl 123456 {h}\n")
    assert bench.load_traffic("fwd", "wl") == 123456.0
    assert bench.load_traffic("fwd", "other") is None
    # a comment-only edit keeps the figure; a code change in any source drops it
    _write(str(tmp_path / "k.cu"), "// the kernel\n__global__ void k() {}\n")
    assert bench.load_traffic("fwd", "wl") == 123456.0
    _write(str(tmp_path / "s.h"), "int s(int);\n")
    assert bench.load_traffic("fwd", "wl") is None
