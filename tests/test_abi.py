"""The C ABI without a GPU: the library loads, exports every declared entry
point, mirrors struct abg_node exactly, and rejects bad arguments with the
documented status before touching the device."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "abg.h")

import affine_bit_group_gb300 as abg  # noqa: E402

OK, EINVAL, EALIGN, ESHAPE, EALIAS = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def lib():
    return abg.library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(abg_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    nm = subprocess.run(["nm", "-D", "--defined-only", os.path.join(ROOT, "affine_bit_group_gb300", "libabg.so")],
                        capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (abg_\w+)", nm))
    assert set(names) <= exported


@pytest.mark.parametrize("ctype,cname", [(abg._Node, "abg_node"), (abg._GdnArgs, "abg_gdn_args"),
                                         (abg._AtqArgs, "abg_atq_args")])
def test_struct_layout_matches_c(tmp_path, ctype, cname):
    """sizeof and field offsets of the node and mixer-argument structs as gcc
    sees the header."""
    fields = [f for f, _ in ctype._fields_]
    prog = tmp_path / "layout.c"
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "abg.h"', "int main(void){",
             f'printf("%zu\\n", sizeof({cname}));']
    lines += [f'printf("%zu\\n", offsetof({cname}, {f}));' for f in fields]
    lines += ["return 0;}"]
    prog.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)], check=True)
    out = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert out[0] == ctypes.sizeof(ctype)
    assert len(out) == len(fields) + 1
    for f, off in zip(fields, out[1:]):
        assert getattr(ctype, f).offset == off, f


def test_constants_match_c(tmp_path):
    """The binding's mode, node-kind, prologue and scale/bias-type constants
    equal the header's enumerators, as gcc sees them."""
    names = ["TREE", "FAST", "NODE_Q4MV", "NODE_RMSQ", "NODE_SWQ", "NODE_GSUM", "NODE_GDN", "NODE_ATQ", "NODE_COPY",
             "PRO_NONE", "PRO_GSUM", "PRO_RMSQ", "PRO_SWQ", "SB_F32", "SB_BF16", "SB_F16"]
    prog = tmp_path / "consts.c"
    lines = ["#include <stdio.h>", '#include "abg.h"', "int main(void){"]
    lines += [f'printf("%d\\n", (int)ABG_{n});' for n in names]
    lines += ["return 0;}"]
    prog.write_text("\n".join(lines))
    exe = tmp_path / "consts"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)], check=True)
    out = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert out == [getattr(abg, n) for n in names]


def test_status_strings(lib):
    assert lib.abg_status_str(0) == b"ok"
    assert lib.abg_status_str(4) == b"output overlaps an input"
    assert lib.abg_status_str(99) == b"unknown status"


A = 0x7F0000000000  # fake, 256-byte aligned device addresses: only validation runs


def q4(lib, w=A, s=A + 0x100000, b=A + 0x200000, x=A + 0x300000, xs=A + 0x310000, y=A + 0x400000, rows=8, cols=128,
       row0=0, n=8, mode=0, rpw=0):
    return lib.abg_q4mv(w, s, b, x, xs, y, rows, cols, row0, n, mode, rpw, None)


def test_q4mv_validation(lib):
    assert q4(lib, w=0) == EINVAL
    assert q4(lib, mode=2) == EINVAL
    assert q4(lib, rpw=3) == EINVAL
    assert q4(lib, cols=100) == ESHAPE
    assert q4(lib, cols=0) == ESHAPE
    assert q4(lib, cols=16384 + 64) == ESHAPE
    assert q4(lib, row0=4, n=5) == ESHAPE
    assert q4(lib, n=-1) == ESHAPE
    assert q4(lib, w=A + 4) == EALIGN
    assert q4(lib, x=A + 0x300008) == EALIGN
    assert q4(lib, y=A + 0x400002) == EALIGN
    assert q4(lib, y=A + 0x300010) == EALIAS          # y overlaps x
    assert q4(lib, y=A + 8) == EALIAS                 # y overlaps the packed weights
    assert q4(lib, n=0, row0=8) == OK                 # empty: nothing enqueued, no device use


def q4x(lib, sb=0, group=64, w=A, s=A + 0x100000, b=A + 0x200000, x=A + 0x300000, xs=A + 0x310000, y=A + 0x400000,
        rows=8, cols=256, row0=0, n=8, mode=0, rpw=0):
    return lib.abg_q4mv_ex(w, s, b, sb, group, x, xs, y, rows, cols, row0, n, mode, rpw, None)


def test_q4mv_ex_validation(lib):
    assert q4x(lib, group=16) == EINVAL
    assert q4x(lib, group=0) == EINVAL
    assert q4x(lib, sb=3) == EINVAL
    assert q4x(lib, sb=-1) == EINVAL
    assert q4x(lib, group=128, cols=192) == ESHAPE     # not whole 128-column groups
    assert q4x(lib, group=32, cols=96) == ESHAPE       # whole groups but not a multiple of 64
    assert q4x(lib, sb=1, s=A + 0x100001) == EALIGN    # 16-bit scale must be 2-byte aligned
    assert q4x(lib, sb=0, s=A + 0x100002) == EALIGN    # f32 scale must be 4-byte aligned
    assert q4x(lib, sb=1, s=A + 0x100002, y=0) == EINVAL  # 2-byte aligned 16-bit scale passes the alignment check
    # y overlapping the bias: bias spans rows*cols/group elements of the stored type
    assert q4x(lib, sb=0, group=32, y=A + 0x200000 + 4 * (8 * 8 - 1)) == EALIAS
    assert q4x(lib, sb=2, group=32, y=A + 0x200000 + 2 * (8 * 8 - 2)) == EALIAS   # last 4 bytes of the bias
    assert q4x(lib, n=0, row0=8, group=128, sb=1) == OK


def test_q4mm_validation(lib):
    w, s, b, x, xs, y = A, A + 0x100000, A + 0x200000, A + 0x300000, A + 0x310000, A + 0x400000
    assert lib.abg_q4mm(w, s, b, x, xs, y, 8, 128, 0, 8, 0, 0, 0, None) == EINVAL   # T = 0
    assert lib.abg_q4mm(w, s, b, x, xs, y, 8, 128, 0, 8, 9, 0, 0, None) == EINVAL   # T > 8
    assert lib.abg_q4mm(w, s, b, x, xs, y, 8, 100, 0, 8, 2, 0, 0, None) == ESHAPE
    # y [T][n] reaching into token 3's activation row x[3]
    assert lib.abg_q4mm(w, s, b, x, xs, x + 4 * 128 * 3 - 4 * 8, 8, 128, 0, 8, 4, 0, 0, None) == EALIAS
    # y overlapping the last token's group sums
    assert lib.abg_q4mm(w, s, b, x, xs, xs + 4 * 2 * 3, 8, 128, 0, 8, 4, 0, 0, None) == EALIAS
    assert lib.abg_q4mm(w, s, b, x, xs, y, 8, 128, 8, 0, 4, 0, 0, None) == OK      # empty


def test_vector_ex_validation(lib):
    assert lib.abg_gsum_ex(A, A + 0x1000, 128, 16, 0, None) == EINVAL
    assert lib.abg_gsum_ex(A, A + 0x1000, 192, 128, 0, None) == ESHAPE
    assert lib.abg_gsum_ex(A, A + 4 * 127, 128, 32, 0, None) == EALIAS
    assert lib.abg_rmsq_ex(A, A + 0x1000, ctypes.c_float(1e-6), A + 0x2000, A + 0x3000, 64, 128, 0, None) == ESHAPE
    assert lib.abg_rmsq_ex(A, A + 0x1000, ctypes.c_float(1e-6), A + 0x2000, A + 0x2000 + 4 * 127, 128, 32, 0,
                           None) == EALIAS
    assert lib.abg_swq_ex(A, A + 0x2000, A + 0x3000, 128, 48, 0, None) == EINVAL
    assert lib.abg_swq_ex(A, A + 0x2000, A + 0x3000, 320, 128, 0, None) == ESHAPE


def test_vector_validation(lib):
    assert lib.abg_gsum(A, A + 0x1000, 100, 0, None) == ESHAPE
    assert lib.abg_gsum(A + 4, A + 0x1000, 128, 0, None) == EALIGN
    assert lib.abg_gsum(A, A + 4, 128, 0, None) == EALIAS
    assert lib.abg_rmsq(A, A + 0x1000, ctypes.c_float(1e-6), A + 0x2000, A + 0x3000, (1 << 20) + 64, 0, None) == ESHAPE
    assert lib.abg_rmsq(A, A + 0x1000, ctypes.c_float(1e-6), A, A + 0x3000, 128, 0, None) == EALIAS
    assert lib.abg_rmsq(A, A + 0x1000, ctypes.c_float(1e-6), A + 0x2000, A + 0x2000, 128, 0, None) == EALIAS
    assert lib.abg_swq(A, A + 0x100, A + 0x3000, 128, 0, None) == EALIAS   # o inside a = [gate | up]
    assert lib.abg_swq(A, A + 0x2000, A + 0x3000, 96, 0, None) == ESHAPE
    assert lib.abg_swq(None, A + 0x2000, A + 0x3000, 128, 0, None) == EINVAL
    assert lib.abg_swq(A, A + 0x2000, A + 0x3000, 128, 7, None) == EINVAL


def node(**kw):
    return abg._Node(**kw)


def create(lib, nodes, mode=0, rpw=0):
    arr = (abg._Node * len(nodes))(*nodes)
    h = ctypes.c_void_p()
    st = lib.abg_stage_graph_create(arr, len(nodes), mode, rpw, ctypes.byref(h))
    assert not h.value
    return st


def test_stage_graph_validation(lib):
    h = ctypes.c_void_p()
    assert lib.abg_stage_graph_create(None, 0, 0, 0, ctypes.byref(h)) == EINVAL
    assert lib.abg_stage_graph_create(None, 1, 0, 0, None) == EINVAL
    prod = dict(kind=0, stage=1, w=A, scale=A + 0x100000, bias=A + 0x200000, rows=8, cols=128, row0=0, n=8,
                y=A + 0x400000, x=A + 0x300000, xsum=A + 0x310000)
    assert create(lib, [node(**{**prod, "kind": 9})]) == EINVAL
    assert create(lib, [node(**{**prod, "cols": 96})]) == ESHAPE
    assert create(lib, [node(**{**prod, "prologue": 7})]) == EINVAL
    # the producer of x in the same stage as the product reading it
    rms = dict(kind=1, stage=1, x=A + 0x500000, wt=A + 0x510000, out=A + 0x300000, out_sum=A + 0x310000, len=128)
    assert create(lib, [node(**rms), node(**prod)]) == EALIAS
    # a node that writes a product's scale
    gs = dict(kind=3, stage=0, x=A + 0x500000, out_sum=A + 0x100000, len=128)
    assert create(lib, [node(**gs), node(**prod)]) == EALIAS
    # two products of one stage writing the same y
    assert create(lib, [node(**prod), node(**{**prod, "w": A + 0x600000})]) == EALIAS
    assert lib.abg_stage_graph_launch(None, None) == EINVAL
    assert lib.abg_stage_graph_destroy(None) == EINVAL


def _gdn_args(H=4, D=128, K=4, **over):
    """gdn arguments at fake, well-separated addresses (16 MiB apart)."""
    names = ["x", "conv", "state", "a", "b", "z", "A_log", "dt_bias", "nw", "S", "y", "ysum"]
    kw = {n: 0x7F0000100000 + (1 << 24) * i for i, n in enumerate(names)}
    kw.update(H=H, D=D, K=K, eps=1e-6, eps_n=1e-6)
    kw.update(over)
    return abg._GdnArgs(**kw)


def _atq_args(Hq=8, Hkv=2, D=128, P=4096, pos=100, **over):
    names = ["q", "gate", "k", "v", "qn_w", "kn_w", "cos", "sin", "Kc", "Vc", "y", "ysum"]
    kw = {n: 0x7E0000100000 + (1 << 26) * i for i, n in enumerate(names)}
    kw.update(Hq=Hq, Hkv=Hkv, D=D, P=P, pos=pos, eps=1e-6)
    kw.update(over)
    return abg._AtqArgs(**kw)


def test_stage_graph_mixer_node_validation(lib):
    """gdn and atq nodes: null or invalid argument structs are refused as the
    direct calls refuse them, and their outputs (including the state and the
    caches they update in place) take part in the stage hazard checks."""
    assert create(lib, [node(kind=abg.NODE_GDN, stage=0)]) == EINVAL           # no args
    assert create(lib, [node(kind=abg.NODE_ATQ, stage=0)]) == EINVAL
    g = _gdn_args(D=96)
    assert create(lib, [node(kind=abg.NODE_GDN, stage=0, args=ctypes.addressof(g))]) == ESHAPE
    g = _gdn_args(S=0x7F0000100000 + 9 * (1 << 24) + 4)                         # S not 16-byte aligned
    assert create(lib, [node(kind=abg.NODE_GDN, stage=0, args=ctypes.addressof(g))]) == EALIGN
    g = _gdn_args(y=0x7F0000100000)                                             # y == x
    assert create(lib, [node(kind=abg.NODE_GDN, stage=0, args=ctypes.addressof(g))]) == EALIAS
    t = _atq_args(pos=4096)                                                     # pos >= P
    assert create(lib, [node(kind=abg.NODE_ATQ, stage=0, args=ctypes.addressof(t))]) == ESHAPE
    t = _atq_args(Hq=6, Hkv=4)
    assert create(lib, [node(kind=abg.NODE_ATQ, stage=0, args=ctypes.addressof(t))]) == ESHAPE
    # a product in the gdn node's stage reading its y
    g = _gdn_args()
    prod = dict(kind=0, stage=0, w=A, scale=A + 0x100000, bias=A + 0x200000, rows=8, cols=128, row0=0, n=8,
                y=A + 0x400000, x=g.y, xsum=A + 0x310000)
    gn = node(kind=abg.NODE_GDN, stage=0, args=ctypes.addressof(g))
    assert create(lib, [gn, node(**prod)]) == EALIAS
    # a product of the same stage reading the recurrent state S the node updates
    assert create(lib, [gn, node(**{**prod, "x": g.S})]) == EALIAS
    # an atq node writing a product's weights (its value cache over w)
    t = _atq_args(Vc=A)
    tn = node(kind=abg.NODE_ATQ, stage=0, args=ctypes.addressof(t))
    assert create(lib, [tn, node(**{**prod, "stage": 1, "x": A + 0x300000})]) == EALIAS
    # two mixers of one stage that share an output
    t2 = _atq_args(y=g.y)
    assert create(lib, [gn, node(kind=abg.NODE_ATQ, stage=0, args=ctypes.addressof(t2))]) == EALIAS
    # a node of an earlier stage writing an atq node's key cache
    t3 = _atq_args()
    gs = dict(kind=3, stage=0, x=A + 0x500000, out_sum=t3.Kc + 4096, len=128)
    assert create(lib, [node(**gs), node(kind=abg.NODE_ATQ, stage=1, args=ctypes.addressof(t3))]) == EALIAS


def test_stage_graph_copy_node_validation(lib):
    """Copy nodes: null pointers, an empty or misaligned copy and overlapping
    ranges are refused before any device call."""
    cp = dict(kind=abg.NODE_COPY, stage=0, x=A, out=A + 0x100000, len=64)
    assert create(lib, [node(**{**cp, "x": 0})]) == EINVAL
    assert create(lib, [node(**{**cp, "out": 0})]) == EINVAL
    assert create(lib, [node(**{**cp, "len": 0})]) == ESHAPE
    assert create(lib, [node(**{**cp, "x": A + 2})]) == EALIGN
    assert create(lib, [node(**{**cp, "out": A + 128})]) == EALIAS


def test_stage_graph_copy_node_validation(lib):
    """Copy nodes: null pointers, an empty or misaligned copy and overlapping
    ranges are refused before any device call."""
    cp = dict(kind=abg.NODE_COPY, stage=0, x=A, out=A + 0x100000, len=64)
    assert create(lib, [node(**{**cp, "x": 0})]) == EINVAL
    assert create(lib, [node(**{**cp, "out": 0})]) == EINVAL
    assert create(lib, [node(**{**cp, "len": 0})]) == ESHAPE
    assert create(lib, [node(**{**cp, "x": A + 2})]) == EALIGN
    assert create(lib, [node(**{**cp, "out": A + 128})]) == EALIAS


def test_tuning_validation(lib):
    assert lib.abg_set_q4mv_tuning(300, 0, 0, 0) == EINVAL
    assert lib.abg_set_q4mv_tuning(0, 17, 0, 0) == EINVAL
    assert lib.abg_set_q4mv_tuning(0, 0, 0, 300) == EINVAL
    assert lib.abg_set_q4mv_tuning(0, 0, 0, 0) == OK


def test_product_path_has_no_cpu_fallback():
    """The package never imports the oracle: its modules name no oracle import."""
    pkg = os.path.join(ROOT, "affine_bit_group_gb300")
    for f in os.listdir(pkg):
        if f.endswith(".py"):
            src = open(os.path.join(pkg, f)).read()
            assert "import oracle" not in src and "from oracle" not in src, f


def test_unknown_graph_handles_are_refused(lib):
    fake = 0x7F0000001000
    assert lib.abg_stage_graph_launch(fake, None) == EINVAL
    assert lib.abg_stage_graph_destroy(fake) == EINVAL
    n = ctypes.c_int64()
    assert lib.abg_stage_graph_launches(fake, ctypes.byref(n)) == EINVAL
    assert lib.abg_stage_graph_swiglu_pairs(fake, ctypes.byref(n)) == EINVAL


def test_static_mlp_rejects_before_device_work(lib):
    """abg_swiglu_mlp_static checks sizes against its static scratch (n <= 16384)
    and its arguments before touching the device."""
    f = lib.abg_swiglu_mlp_static
    p = [0x7F0000100000 + 4096 * i for i in range(12)]
    assert f(*p, 16384 + 64, 2048, 10, 0, None) == ESHAPE   # more than the static scratch holds
    assert f(*p, 100, 2048, 10, 0, None) == ESHAPE          # n not a multiple of 64
    assert f(*p, 1024, 2000, 10, 0, None) == ESHAPE         # cols not a multiple of 64
    assert f(*p, 1024, 2048, 10, 7, None) == EINVAL         # bad mode
    q = list(p)
    q[11] = p[9]                                           # y == x
    assert f(*q, 1024, 2048, 10, 0, None) == EALIAS
    q = list(p)
    q[0] += 4                                              # gate words not 16-byte aligned
    assert f(*q, 1024, 2048, 10, 0, None) == EALIGN
    assert f(*([None] + p[1:]), 1024, 2048, 10, 0, None) == EINVAL


def test_gdn_rejects_before_device_work(lib):
    """abg_gdn checks its shape, mode, alignment and output overlaps before any
    device work (fake, well-separated addresses; none is dereferenced)."""
    f = lib.abg_gdn
    p = [0x7F0000100000 + (1 << 24) * i for i in range(12)]
    F = ctypes.c_float
    ok = dict(H=4, D=128, K=4)

    def call(ptrs, H=4, D=128, K=4, mode=0):
        return f(*ptrs, H, D, K, F(1e-6), F(1e-6), mode, None)

    assert call(p, D=96) == ESHAPE                # head dimension not 64, 128 or 256
    assert call(p, K=1) == ESHAPE and call(p, K=9) == ESHAPE
    assert call(p, H=0) == ESHAPE
    assert call(p, mode=3) == EINVAL
    assert call([None] + p[1:]) == EINVAL
    q = list(p)
    q[9] = p[0]                                   # S over x
    assert call(q, **ok) == EALIAS
    q = list(p)
    q[10] = p[11]                                 # y over ysum
    assert call(q, **ok) == EALIAS
    q = list(p)
    q[2] += 2                                     # state not 4-byte aligned
    assert call(q, **ok) == EALIGN
    q = list(p)
    q[9] += 4                                     # S not 16-byte aligned (one bulk copy per head)
    assert call(q, **ok) == EALIGN


def test_atq_rejects_before_device_work(lib):
    """abg_atq checks its shape (including the 8192-position limit), mode,
    alignment and output overlaps before any device work."""
    f = lib.abg_atq
    p = [0x7F0000100000 + (1 << 28) * i for i in range(12)]
    F = ctypes.c_float

    def call(ptrs, Hq=8, Hkv=2, D=256, P=4096, pos=100, mode=0):
        return f(*ptrs, Hq, Hkv, D, P, pos, F(1e-6), mode, None)

    assert call(p, Hq=6, Hkv=4) == ESHAPE        # query heads not a multiple of the kv heads
    assert call(p, D=96) == ESHAPE
    assert call(p, pos=4096) == ESHAPE           # pos past the cache
    assert call(p, P=10000, pos=8192) == ESHAPE  # past the position limit
    assert call(p, pos=-1) == ESHAPE
    assert call(p, mode=5) == EINVAL
    assert call([None] + p[1:]) == EINVAL
    q = list(p)
    q[10] = p[0]                                 # y over q
    assert call(q) == EALIAS
    q = list(p)
    q[9] = p[8]                                  # V cache over K cache
    assert call(q) == EALIAS
    q = list(p)
    q[8] += 2
    assert call(q) == EALIGN
    for i in (8, 9):                             # a cache 4- but not 16-byte aligned
        q = list(p)
        q[i] += 4
        assert call(q) == EALIGN
