"""bench.py's link between the committed ncu summaries and the kernel source
(CPU): the summaries' recorded hash is of the code, without comments, of every
source the product kernel and its launch plan depend on, so a comment edit
keeps the recorded DRAM traffic and a code edit in any of them drops it."""
from __future__ import annotations

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_hash_ignores_comments_and_blank_lines(tmp_path):
    a = tmp_path / "a.cuh"
    b = tmp_path / "b.cuh"
    a.write_text('int f(int x) {\n    return x + 1;  // add one\n}\n')
    b.write_text('// a new header comment\n\nint f(int x) {\n    return x + 1;\n}\n\n')
    assert bench.code_sha256(str(a)) == bench.code_sha256(str(b))


def test_code_hash_sees_code_and_keeps_string_contents(tmp_path):
    a = tmp_path / "a.cuh"
    b = tmp_path / "b.cuh"
    c = tmp_path / "c.cuh"
    a.write_text('int f(int x) { return x + 1; }\n')
    b.write_text('int f(int x) { return x + 2; }\n')
    c.write_text('const char *s = "a // b";\n')
    assert bench.code_sha256(str(a)) != bench.code_sha256(str(b))
    d = tmp_path / "d.cuh"
    d.write_text('const char *s = "a ";\n')
    assert bench.code_sha256(str(c)) != bench.code_sha256(str(d))


def test_kernel_hash_covers_every_kernel_source(tmp_path, monkeypatch):
    srcs = []
    for i, name in enumerate(("k.cuh", "dev.cuh", "plan.cu")):
        p = tmp_path / name
        p.write_text(f"int f{i}() {{ return {i}; }}\n")
        srcs.append(str(p))
    monkeypatch.setattr(bench, "ROOT", "/")
    base = bench.kernel_code_sha256(srcs)
    for i, p in enumerate(srcs):
        orig = open(p).read()
        open(p, "w").write(orig + "// a comment\n")
        assert bench.kernel_code_sha256(srcs) == base
        open(p, "w").write(orig.replace(f"return {i}", f"return {i + 10}"))
        assert bench.kernel_code_sha256(srcs) != base, p
        open(p, "w").write(orig)
    assert bench.kernel_code_sha256(srcs) == base


def test_bench_lists_the_kernel_sources():
    for rel in bench.KERNEL_SOURCES:
        assert os.path.exists(os.path.join(ROOT, rel)), rel
    names = {os.path.basename(r) for r in bench.KERNEL_SOURCES}
    assert {"q4mv_kernel.cuh", "abg_dev.cuh", "q4mv.cu", "q4mv_fixed.cu"} <= names
