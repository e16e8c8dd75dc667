"""bench.py's link between the committed ncu summaries and the kernel source
(CPU): the summaries' recorded hash is of the kernel's code without comments,
so a comment edit keeps the recorded DRAM traffic and a code edit drops it."""
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
