"""GPU parity of the other weight formats against the CPU oracle.

Group sizes 32, 64 and 128 columns, scale and bias stored as f32, bf16 or f16
(the MLX 4-bit variants of "Metal: queued rmsq, swq, gdn and atq kernels and a
4-row q4mv ..." (bendlang/bend #1440), Why).  Tree mode is bit-for-bit the
oracle's; fast mode within 1e-5 * max(|y|, sum_g |scale*d| + |bias*xsum|).
Shapes span several tiles and 1024-column chunks with ragged tails, every
rows-per-warp setting, the largest width, both ways of reading scale and bias,
activations that take the plain product path, the producers' group sums, the
fused prologues in a stage graph, and the 4096x2048 product in full.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from affine_bit_group_gb300 import synth
from helpers import assert_bits_equal, assert_fast_close, dev, dev_words, empty, host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
abg = pytest.importorskip("affine_bit_group_gb300")

FORMATS = [(g, sb) for g in synth.GROUPS for sb in synth.SB_TYPES]


def dev_sb(a):
    """Scale or bias on the device: f32 values or 16-bit patterns (as int16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).cuda()
    return dev(a)


def run(m, x, xs=None, mode=abg.TREE, rpw=0, row0=0, n=None, scale=None, bias=None):
    n = m.rows - row0 if n is None else n
    xs = oracle.gsum_ex(x, m.group) if xs is None else xs
    y = empty(max(n, 1))
    abg.q4mv_ex(dev_words(m.w), dev_sb(m.scale) if scale is None else scale,
                dev_sb(m.bias) if bias is None else bias, m.sb, m.group, dev(x), dev(xs), y, cols=m.cols,
                row0=row0, n=n, mode=mode, rows_per_warp=rpw)
    torch.cuda.synchronize()
    return host(y)[:n]


def expect(m, x, xs=None, row0=0, n=None):
    xs = oracle.gsum_ex(x, m.group) if xs is None else xs
    return oracle.q4mv_ex(*m.arrays(), m.sb, m.group, x, xs, m.cols, row0=row0, n=n)


def widened(m):
    G = m.cols // m.group
    if m.sb == "f32":
        return m.scale.astype(np.float64), m.bias.astype(np.float64)
    return (oracle.half_to_f32(m.scale, m.sb).reshape(m.rows, G).astype(np.float64),
            oracle.half_to_f32(m.bias, m.sb).reshape(m.rows, G).astype(np.float64))


def magnitude(m, x):
    """A_r = sum_g |scale*d| + |bias*xsum| in float64 (scales the fast-mode bound)."""
    s, b = widened(m)
    q = np.zeros((m.rows, m.cols), np.float64)
    for j in range(8):
        q[:, j::8] = (m.w >> np.uint32(4 * j)) & 0xF
    G, gs = m.cols // m.group, m.group
    d = (q * x.astype(np.float64)).reshape(m.rows, G, gs).sum(axis=2)
    xs = x.astype(np.float64).reshape(G, gs).sum(axis=1)
    return (np.abs(s * d) + np.abs(b * xs)).sum(axis=1)


SHAPES = [(1, 128), (37, 384), (129, 1152), (65, 2048), (31, 3200), (300, 1024), (77, 6144), (9, 16384)]


@pytest.mark.parametrize("group,sb", FORMATS)
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_formats_tree_bit_exact(group, sb, rows, cols):
    m, x = synth.fmt_case(group, sb, rows, cols)
    exp = expect(m, x)
    for rpw in (1, 2, 4, 8):
        assert_bits_equal(run(m, x, rpw=rpw), exp, f"g{group} {sb} {rows}x{cols} R={rpw}")


@pytest.mark.parametrize("group", [32, 64])
def test_group_counts_not_multiple_of_four(group):
    """cols = 192: 6 or 3 groups per row, so a row of f32 scales is not 16 bytes; plain loads."""
    for sb in synth.SB_TYPES:
        m, x = synth.fmt_case(group, sb, 45, 192)
        assert_bits_equal(run(m, x), expect(m, x), f"g{group} {sb} 45x192")


@pytest.mark.parametrize("group,sb", FORMATS)
def test_formats_fast_within_bound(group, sb):
    m, x = synth.fmt_case(group, sb, 129, 3072)
    tree = expect(m, x)
    mag = magnitude(m, x)
    for rpw in (1, 8):
        assert_fast_close(run(m, x, mode=abg.FAST, rpw=rpw), tree, mag, what=f"fast g{group} {sb}")


@pytest.mark.parametrize("group,sb", FORMATS)
def test_formats_full_4096x2048(group, sb):
    """The 4096x2048 product of every format, all outputs, and its hash."""
    m, x = synth.fmt_case(group, sb, 4096, 2048)
    exp = expect(m, x)
    got = run(m, x)
    assert_bits_equal(got, exp, f"4096x2048 g{group} {sb}")
    assert oracle.hash32(got) == oracle.hash32(exp)


@pytest.mark.parametrize("group,sb", [(32, "bf16"), (128, "f16"), (128, "f32"), (64, "bf16")])
def test_row_range_and_unaligned_scale_bias(group, sb):
    m, x = synth.fmt_case(group, sb, 300, 2048)
    assert_bits_equal(run(m, x, row0=37, n=200), expect(m, x, row0=37, n=200), "row range")
    # scale and bias one element past a 16-byte boundary: read with ordinary loads
    pad = np.zeros(1, m.scale.dtype)
    sbuf = dev_sb(np.concatenate([pad, m.scale.ravel()]))
    bbuf = dev_sb(np.concatenate([pad, m.bias.ravel()]))
    assert sbuf[1:].data_ptr() % 16 != 0
    assert_bits_equal(run(m, x, scale=sbuf[1:], bias=bbuf[1:]), expect(m, x), "unaligned scale/bias")


@pytest.mark.parametrize("group", synth.GROUPS)
@pytest.mark.parametrize("case", ["neg_zero", "inf", "nan", "all_negative", "mixed_negative_groups"])
def test_formats_special_activations(group, case):
    """Values outside the fused-multiply-add identity take the plain path; groups
    of all-negative values (spanning 1, 2 or 4 lanes) are marked for the sign
    of a zero group sum, and the mark must cover exactly the group's lanes."""
    m, x = synth.fmt_case(group, "bf16", 70, 2048)
    x = x.copy()
    if case == "neg_zero":
        x[::5] = -0.0
    elif case == "inf":
        x[17] = np.inf
    elif case == "nan":
        x[1000] = np.nan
    elif case == "all_negative":
        x = -np.abs(x)
    else:
        x = np.abs(x)
        for g in range(0, 2048 // group, 3):
            x[group * g:group * g + group] *= -1
        x[32:64] *= -1  # a negative half of a 64-column span
    xs = oracle.gsum_ex(x, group)
    assert_bits_equal(run(m, x, xs=xs), expect(m, x, xs=xs), f"g{group} {case}")
    assert abg.device_status(clear=True) == 0


def test_all_q_zero_with_negative_group_keeps_signed_zero():
    """q = 0 and a group of negative x: RN(0*x) = -0, d = -0; with bias 0 the
    group term is -0 + (+-0).  Bits must match the oracle, signs included."""
    for group in synth.GROUPS:
        m, x = synth.fmt_case(group, "f32", 8, 256)
        m.w[:] = 0
        m.bias[:] = 0.0
        x = -np.abs(x)
        assert_bits_equal(run(m, x), expect(m, x), f"signed zero g{group}")


@pytest.mark.parametrize("group", synth.GROUPS)
@pytest.mark.parametrize("sb", synth.SB_TYPES)
def test_formats_zero_groups_of_negative_activations(group, sb):
    """All-negative activations with planted zero groups (whole rows with zero
    bias, single groups, single groups with zero bias): the exact path with the
    sign fix for zero group sums must give the oracle's bits, -0 results included."""
    m, x = synth.fmt_case(group, sb, 150, 2048)
    x = -np.abs(x)
    G, wpg = 2048 // group, group // 8
    rng = np.random.default_rng(group)
    m.w[:6] = 0
    m.bias[:6] = 0
    for r in range(20, 60):
        g = int(rng.integers(G))
        m.w[r, wpg * g:wpg * (g + 1)] = 0
        if r >= 40:
            m.bias[r, g] = 0
    exp = expect(m, x)
    assert (exp[:6] == 0).all() and np.signbit(exp[:6]).all()
    assert_bits_equal(run(m, x), exp, f"zero groups g{group} {sb}")
    assert abg.device_status(clear=True) == 0


@pytest.mark.parametrize("group", synth.GROUPS)
def test_producers_group_sums(group):
    rng = np.random.default_rng(group)
    n = 3072
    v = synth.activations(rng, n)
    wt = synth.rms_weights(rng, n)
    a = synth.activations(rng, 2 * n)
    s = empty(n // group)
    abg.gsum(dev(v), s, group=group)
    xn, xs = empty(n), empty(n // group)
    abg.rmsq(dev(v), dev(wt), xn, xs, eps=1e-6, group=group)
    o, os_ = empty(n), empty(n // group)
    abg.swq(dev(a), o, os_, group=group)
    torch.cuda.synchronize()
    assert_bits_equal(host(s), oracle.gsum_ex(v, group), "gsum")
    xn_o, _ = oracle.rmsq(v, wt, 1e-6)
    assert_bits_equal(host(xn), xn_o, "rmsq")
    assert_bits_equal(host(xs), oracle.gsum_ex(xn_o, group), "rmsq sums")
    o_o, _ = oracle.swq(a)
    assert_bits_equal(host(o), o_o, "swq")
    assert_bits_equal(host(os_), oracle.gsum_ex(o_o, group), "swq sums")


@pytest.mark.parametrize("group,sb", [(64, "bf16"), (64, "f16"), (32, "f32"), (32, "bf16"), (128, "f32"),
                                      (128, "f16")])
@pytest.mark.parametrize("rows,cols", [(20480, 2048), (9000, 4096), (15360, 6144), (2048, 2048), (700, 6144)])
def test_fixed_shapes_every_format(group, sb, rows, cols):
    """Every format runs the fixed-shape instantiations at 2048, 4096 and 6144
    columns (many tiles: 8 rows per item, two blocks per SM or, for 6144
    columns, 18 warps in one; few tiles: 4 rows per item, 16 warps): every row
    bit-exact in tree mode; fast mode within its bound (the smaller shapes)."""
    m, x = synth.fmt_case(group, sb, rows, cols)
    exp = expect(m, x)
    assert_bits_equal(run(m, x), exp, f"g{group} {sb} {rows}x{cols}")
    if rows * cols <= 8 << 20:
        assert_fast_close(run(m, x, mode=abg.FAST), exp, magnitude(m, x), what=f"fast g{group} {sb} {rows}x{cols}")
    assert abg.device_status(clear=True) == 0


@pytest.mark.parametrize("group,sb", [(32, "bf16"), (128, "f16"), (32, "f32"), (128, "f32"), (64, "bf16"),
                                      (64, "f16")])
def test_graph_prologues_and_grouping(group, sb):
    """Stage graph with the node's group and sb_type: an rmsq node feeding a
    product, and products with each fused prologue; siblings grouped."""
    rng = np.random.default_rng([group, len(sb)])
    C = 2048
    h = synth.activations(rng, C)
    wt = synth.rms_weights(rng, C)
    a = synth.activations(rng, 2 * C)
    mats = [synth.fmt_case(group, sb, r, C)[0] for r in (1024, 256, 256)]
    hd, wtd, ad = dev(h), dev(wt), dev(a)
    xn, xs = empty(C), empty(C // group)
    dms = [(dev_words(m.w), dev_sb(m.scale), dev_sb(m.bias)) for m in mats]
    ys = {k: [empty(m.rows) for m in mats] for k in ("none", "gsum", "rmsq", "swq")}
    nodes = [abg.Node.rmsq(0, hd, wtd, xn, xs, eps=1e-6, group=group)]
    for (w, s, b), y in zip(dms, ys["none"]):
        nodes.append(abg.Node.q4mv(1, w, s, b, y, C, x=xn, xsum=xs, group=group, sb_type=sb))
    for (w, s, b), y in zip(dms, ys["gsum"]):
        nodes.append(abg.Node.q4mv(2, w, s, b, y, C, x=hd, prologue=abg.PRO_GSUM, group=group, sb_type=sb))
    for (w, s, b), y in zip(dms, ys["rmsq"]):
        nodes.append(abg.Node.q4mv(3, w, s, b, y, C, x=hd, wt=wtd, eps=1e-6, prologue=abg.PRO_RMSQ, group=group,
                                   sb_type=sb))
    for (w, s, b), y in zip(dms, ys["swq"]):
        nodes.append(abg.Node.q4mv(4, w, s, b, y, C, x=ad, prologue=abg.PRO_SWQ, group=group, sb_type=sb))
    keep = [hd, wtd, ad, xn, xs] + [t for d in dms for t in d] + [y for v in ys.values() for y in v]
    g = abg.StageGraph(nodes, keep=keep)
    assert g.launches == 5  # the rmsq node, then one grouped launch per stage
    g.launch()
    torch.cuda.synchronize()
    xn_o, _ = oracle.rmsq(h, wt, 1e-6)
    o_o, _ = oracle.swq(a)
    acts = {"none": xn_o, "gsum": h, "rmsq": xn_o, "swq": o_o}
    assert_bits_equal(host(xs), oracle.gsum_ex(xn_o, group), "rmsq node sums")
    for k, act in acts.items():
        axs = oracle.gsum_ex(act, group)
        for m, y in zip(mats, ys[k]):
            exp = oracle.q4mv_ex(*m.arrays(), sb, group, act, axs, C)
            assert_bits_equal(host(y), exp, f"{k} g{group} {sb} {m.rows}")
    g.close()
    assert abg.device_status(clear=True) == 0


def test_mixed_formats_in_one_stage_are_separate_launches():
    C = 1024
    x = synth.activations(np.random.default_rng(3), C)
    xd = dev(x)
    mats = [synth.fmt_case(32, "bf16", 300, C)[0], synth.fmt_case(128, "f32", 200, C)[0],
            synth.fmt_case(32, "bf16", 100, C)[0]]
    dms = [(dev_words(m.w), dev_sb(m.scale), dev_sb(m.bias)) for m in mats]
    ys = [empty(m.rows) for m in mats]
    nodes = [abg.Node.q4mv(0, w, s, b, y, C, x=xd, prologue=abg.PRO_GSUM, group=m.group, sb_type=m.sb)
             for m, (w, s, b), y in zip(mats, dms, ys)]
    g = abg.StageGraph(nodes, keep=[xd] + ys + [t for d in dms for t in d])
    assert g.launches == 2
    g.launch()
    torch.cuda.synchronize()
    for m, y in zip(mats, ys):
        assert_bits_equal(host(y), expect(m, x), f"mixed g{m.group} {m.sb}")
    g.close()
