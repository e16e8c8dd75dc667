"""GPU parity of the product kernel against the CPU oracle (through the C ABI).

Tree mode must be bit-for-bit equal to the oracle; fast mode within
1e-5 * max(|y|, sum_g |scale*d| + |bias*xsum|) per output.  Shapes span
several row tiles and 1024-column chunks with ragged tails (rows not a
multiple of the tile, cols not a multiple of 1024, group counts that are not
powers of two), every rows-per-warp setting, row sub-ranges, both ways of
reading scale and bias, and activations with special values.
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


def run(m, x, xs=None, mode=abg.TREE, rpw=0, row0=0, n=None, scale=None, bias=None):
    n = m.rows - row0 if n is None else n
    xs = oracle.gsum(x) if xs is None else xs
    y = empty(max(n, 1))
    abg.q4mv(dev_words(m.w), dev(m.scale) if scale is None else scale, dev(m.bias) if bias is None else bias,
             dev(x), dev(xs), y, cols=m.cols, row0=row0, n=n, mode=mode, rows_per_warp=rpw)
    torch.cuda.synchronize()
    return host(y)[:n]


def expect(m, x, row0=0, n=None):
    xs = oracle.gsum(x)
    return oracle.q4mv(*m.arrays(), x, xs, m.cols, row0=row0, n=n)


@pytest.mark.parametrize("rpw", [0, 1, 2, 4, 8])
def test_tiny_tree_bit_exact(rpw):
    m, x = synth.tiny()
    assert_bits_equal(run(m, x, rpw=rpw), expect(m, x), "tiny")


SHAPES = [(1, 64), (5, 128), (13, 192), (33, 960), (257, 1024), (100, 1088), (65, 2048), (31, 3008),
          (129, 4096), (77, 6144), (9, 16384), (600, 2048), (1000, 320)]


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("rpw", [1, 4, 8])
def test_shapes_tree_bit_exact(rows, cols, rpw):
    m, x = synth.random_case(1000 + rows + cols, rows, cols)
    assert_bits_equal(run(m, x, rpw=rpw), expect(m, x), f"{rows}x{cols} R={rpw}")


@pytest.mark.parametrize("rows,cols", [(77, 6144), (129, 4096), (33, 960), (600, 2048)])
def test_fast_mode_within_bound(rows, cols):
    m, x = synth.random_case(2000 + rows, rows, cols)
    xs = oracle.gsum(x)
    tree = expect(m, x)
    mag = oracle.q4mv_absmag(*m.arrays(), x, xs, cols)
    for rpw in (1, 2, 4, 8):
        assert_fast_close(run(m, x, mode=abg.FAST, rpw=rpw), tree, mag, what=f"fast {rows}x{cols}")


@pytest.mark.parametrize("row0,n", [(0, 1), (1, 7), (37, 200), (299, 1), (150, 150)])
def test_row_range(row0, n):
    m, x = synth.random_case(3, 300, 2048)
    assert_bits_equal(run(m, x, row0=row0, n=n), expect(m, x, row0, n), f"rows {row0}+{n}")


def test_scale_bias_unaligned_take_plain_loads():
    """scale/bias offset by 4 bytes: rows are read with ordinary loads, same bits."""
    m, x = synth.random_case(4, 150, 2048)
    G = m.cols // 64
    sbuf = dev(np.concatenate([[0.0], m.scale.ravel()]).astype(np.float32))
    bbuf = dev(np.concatenate([[0.0], m.bias.ravel()]).astype(np.float32))
    got = run(m, x, scale=sbuf[1:], bias=bbuf[1:])
    assert sbuf[1:].data_ptr() % 16 == 4 and G % 4 == 0
    assert_bits_equal(got, expect(m, x), "unaligned scale/bias")


@pytest.mark.parametrize("case", ["neg_zero", "inf", "nan", "huge", "subnormal", "zeros"])
def test_special_activations(case):
    """Values outside the fused-multiply-add identity take the plain path; bits still match."""
    m, x = synth.random_case(5, 40, 2048)
    x = x.copy()
    if case == "neg_zero":
        x[::3] = -0.0
    elif case == "inf":
        x[5], x[700] = np.inf, -np.inf
    elif case == "nan":
        x[9] = np.nan
    elif case == "huge":
        x[100] = np.float32(3e30)
    elif case == "subnormal":
        x[::2] = np.float32(1e-42)
    elif case == "zeros":
        x[:] = 0.0
    xs = oracle.gsum(x)
    got = run(m, x, xs=xs)
    exp = oracle.q4mv(*m.arrays(), x, xs, m.cols)
    assert_bits_equal(got, exp, case)


def test_empty_product_enqueues_nothing():
    m, x = synth.random_case(6, 10, 128)
    y = torch.full((1,), 7.0, device="cuda")
    abg.q4mv(dev_words(m.w), dev(m.scale), dev(m.bias), dev(x), dev(oracle.gsum(x)), y, cols=128, row0=10, n=0)
    torch.cuda.synchronize()
    assert float(y[0]) == 7.0


def test_mid_400_calls_hash():
    """4096x2048, 400 calls back to back: identical bits every call, hash equal to the oracle's."""
    m, x = synth.mid()
    xs = oracle.gsum(x)
    exp = oracle.q4mv(*m.arrays(), x, xs, m.cols)
    w, s, b, xd, xsd = dev_words(m.w), dev(m.scale), dev(m.bias), dev(x), dev(xs)
    ys = [empty(m.rows) for _ in range(2)]
    for i in range(400):
        abg.q4mv(w, s, b, xd, xsd, ys[i % 2], cols=m.cols)
        if i == 0:
            torch.cuda.synchronize()
            first = host(ys[0]).copy()
    torch.cuda.synchronize()
    assert_bits_equal(first, exp, "mid call 1")
    assert_bits_equal(host(ys[1]), exp, "mid call 400")
    assert oracle.hash32(host(ys[1])) == oracle.hash32(exp)
    for rpw in (1, 2, 8):
        y = empty(m.rows)
        abg.q4mv(w, s, b, xd, xsd, y, cols=m.cols, rows_per_warp=rpw)
        torch.cuda.synchronize()
        assert oracle.hash32(host(y)) == oracle.hash32(exp)


def test_head_all_rows():
    """248320x2048 output head with x = rmsq(hidden): every row equals the oracle's."""
    m, hidden, wt = synth.head()
    xn_o, xs_o = oracle.rmsq(hidden, wt, 1e-6)
    xn, xsd = empty(2048), empty(32)
    abg.rmsq(dev(hidden), dev(wt), xn, xsd, eps=1e-6)
    torch.cuda.synchronize()
    assert_bits_equal(host(xn), xn_o, "head rmsq")
    assert_bits_equal(host(xsd), xs_o, "head rmsq sums")
    y = empty(m.rows)
    abg.q4mv(dev_words(m.w), dev(m.scale), dev(m.bias), xn, xsd, y, cols=m.cols)
    torch.cuda.synchronize()
    got = host(y)
    assert_bits_equal(got, oracle.q4mv(*m.arrays(), xn_o, xs_o, m.cols), "head, all rows")
    assert np.all(np.isfinite(got))


@pytest.mark.parametrize("rows,cols", [(16384, 6144), (65536, 2048), (6144, 4096)])
def test_sweep_points_whole_output(rows, cols):
    m, x = synth.sweep_point(rows, cols)
    xs = oracle.gsum(x)
    assert_bits_equal(run(m, x, xs=xs), oracle.q4mv(*m.arrays(), x, xs, cols), f"{rows}x{cols}")


def test_grouped_launch_matches_single_calls():
    """Products sharing x in one stage run as one grouped launch; same bits as single calls."""
    mats = [synth.random_case(70 + i, r, 2048)[0] for i, r in enumerate([4096, 512, 512])]
    x = synth.activations(np.random.default_rng(9), 2048)
    xs = oracle.gsum(x)
    xd, xsd = dev(x), dev(xs)
    ys = [empty(m.rows) for m in mats]
    dms = [(dev_words(m.w), dev(m.scale), dev(m.bias)) for m in mats]
    nodes = [abg.Node.q4mv(0, w, s, b, y, 2048, x=xd, xsum=xsd) for (w, s, b), y in zip(dms, ys)]
    g = abg.StageGraph(nodes, keep=[xd, xsd] + ys + [t for d in dms for t in d])
    assert g.launches == 1
    g.launch()
    torch.cuda.synchronize()
    for m, y in zip(mats, ys):
        assert_bits_equal(host(y), oracle.q4mv(*m.arrays(), x, xs, 2048), "grouped")
    g.close()


def test_grouped_launch_negative_activation():
    """A grouped launch over all-negative activations: the exact path with the
    sign fix for zero group sums, one product holding rows whose every term is zero."""
    mats = [synth.random_case(80 + i, r, 1024)[0] for i, r in enumerate([2048, 256, 256])]
    mats[1].w[:3] = 0
    mats[1].bias[:3] = 0.0
    x = -np.abs(synth.activations(np.random.default_rng(10), 1024))
    xs = oracle.gsum(x)
    xd, xsd = dev(x), dev(xs)
    ys = [empty(m.rows) for m in mats]
    dms = [(dev_words(m.w), dev(m.scale), dev(m.bias)) for m in mats]
    nodes = [abg.Node.q4mv(0, w, s, b, y, 1024, x=xd, xsum=xsd) for (w, s, b), y in zip(dms, ys)]
    g = abg.StageGraph(nodes, keep=[xd, xsd] + ys + [t for d in dms for t in d])
    g.launch()
    torch.cuda.synchronize()
    for m, y in zip(mats, ys):
        assert_bits_equal(host(y), oracle.q4mv(*m.arrays(), x, xs, 1024), "grouped negative")
    g.close()
    assert abg.device_status(clear=True) == 0


@pytest.mark.parametrize("cols", [1024, 2048, 6144])
def test_mixed_negative_groups(cols):
    """Some 64-value groups all negative, others not: lanes of one warp disagree about
    their own group, the warp must still agree on its path (and not stall)."""
    m, x = synth.random_case(90, 300, cols)
    x = np.abs(x)
    for g in range(0, cols // 64, 3):
        x[64 * g:64 * g + 64] *= -1
    x[64:128] *= -1  # a lone positive-negative mix
    xs = oracle.gsum(x)
    assert_bits_equal(run(m, x, xs=xs), oracle.q4mv(*m.arrays(), x, xs, cols), f"mixed {cols}")
    assert abg.device_status(clear=True) == 0


def zero_group_case(seed, rows, cols, group=64):
    """All-negative activations with zero groups planted in the weights: rows
    0..9 all nibbles and bias zero (the oracle's y is -0), rows 40..79 one zero
    group each, rows 100..109 one zero group whose bias is also zero."""
    m, x = synth.random_case(seed, rows, cols)
    x = -np.abs(x)
    G, wpg = cols // group, group // 8
    rng = np.random.default_rng(seed)
    m.w[:10] = 0
    m.bias[:10] = 0.0
    for r in range(40, min(rows, 110)):
        if 80 <= r < 100:
            continue
        g = int(rng.integers(G))
        m.w[r, wpg * g:wpg * (g + 1)] = 0
        if r >= 100:
            m.bias[r, g] = 0.0
    return m, x


@pytest.mark.parametrize("rpw", [1, 2, 4, 8])
@pytest.mark.parametrize("cols", [256, 1088, 2048, 6144])
def test_zero_groups_of_negative_activations(rpw, cols):
    """All-negative groups take the exact product path, whose zero sums are +0;
    there a zero group sum means every q is 0, and RN's sum is -0 (RN(0*x) = -0),
    so rows whose every term is zero come out -0 like the oracle's, and rows
    with a single zero group match bit for bit."""
    m, x = zero_group_case(400 + cols, 300, cols)
    exp = expect(m, x)
    assert (exp[:10] == 0).all() and np.signbit(exp[:10]).all()
    assert_bits_equal(run(m, x, rpw=rpw), exp, f"zero groups {cols} R={rpw}")
    assert abg.device_status(clear=True) == 0


def test_zero_groups_fast_mode():
    """Fast mode does not fix the sign of zero group sums; zeros of either sign are within the bound."""
    m, x = zero_group_case(401, 300, 2048)
    xs = oracle.gsum(x)
    y = run(m, x, mode=abg.FAST)
    assert_fast_close(y, oracle.q4mv(*m.arrays(), x, xs, 2048), oracle.q4mv_absmag(*m.arrays(), x, xs, 2048), what="zero groups fast")


def test_no_device_timeouts():
    assert abg.device_status(clear=True) == 0


@pytest.mark.parametrize("tuning", [(0, 0, 1, 1), (0, 4, 1, 2), (0, 0, 0, 0), (220, 16, 0, 64)])
def test_many_tiles_per_block(tuning):
    """Stage rings and partial buffers that wrap many times per block: small
    stages (up to 8 of them), one block per SM, 500000 short rows; every
    output bit-exact (a phase or buffer-rotation error shows up here)."""
    m, x = synth.random_case(95, 500_000, 128)
    abg.set_q4mv_tuning(*tuning)
    try:
        got = run(m, x)
    finally:
        abg.set_q4mv_tuning(0, 0, 0, 0)
    assert_bits_equal(got, expect(m, x), f"tuning {tuning}")
    assert abg.device_status(clear=True) == 0
