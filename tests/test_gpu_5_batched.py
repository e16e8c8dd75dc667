"""GPU parity of the batched product (abg_q4mm) against the oracle.

A batch of T tokens shares one pass over the weights; every token's output must
be bit-for-bit its own single-token product (tree mode), or within the
fast-mode bound.  Covers T = 1..8 (four tokens share a launch on rows of 2048
columns, otherwise pairs; an odd last token runs alone), shapes with ragged
row tiles and
column counts that are not a multiple of a warp's chunk, up to 16384 columns;
tokens whose slices take different product paths; row ranges; unaligned
scale/bias; the 4096x2048 product and the 248320x2048 head in full.
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


def tokens(seed, T, cols):
    rng = np.random.default_rng([seed, T, cols])
    return np.stack([synth.activations(rng, cols) for _ in range(T)])


def run(m, X, XS=None, mode=abg.TREE, row0=0, n=None, scale=None, bias=None):
    T = X.shape[0]
    n = m.rows - row0 if n is None else n
    XS = np.stack([oracle.gsum(x) for x in X]) if XS is None else XS
    Y = empty(max(T * n, 1))
    abg.q4mm(dev_words(m.w), dev(m.scale) if scale is None else scale, dev(m.bias) if bias is None else bias,
             dev(X), dev(XS), Y, cols=m.cols, row0=row0, n=n, mode=mode)
    torch.cuda.synchronize()
    return host(Y)[:T * n].reshape(T, n)


def expect(m, X, row0=0, n=None):
    XS = np.stack([oracle.gsum(x) for x in X])
    return oracle.q4mm(*m.arrays(), X, XS, m.cols, row0=row0, n=n)


SHAPES = [(1, 64), (7, 128), (37, 320), (129, 1024), (65, 2048), (31, 3008), (100, 4096), (77, 6144), (9, 16384)]


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_batched_tree_bit_exact(T, rows, cols):
    m, _ = synth.random_case(3000 + rows + cols, rows, cols)
    X = tokens(1, T, cols)
    assert_bits_equal(run(m, X), expect(m, X), f"T={T} {rows}x{cols}")


@pytest.mark.parametrize("T", [2, 4])
@pytest.mark.parametrize("cols", [2048, 3072, 4096])
def test_batched_fast_within_bound(T, cols):
    m, _ = synth.random_case(3100 + cols, 300, cols)
    X = tokens(2, T, cols)
    tree = expect(m, X)
    got = run(m, X, mode=abg.FAST)
    for t in range(T):
        mag = oracle.q4mv_absmag(*m.arrays(), X[t], oracle.gsum(X[t]), cols)
        assert_fast_close(got[t], tree[t], mag, what=f"fast T={T} token {t}")


@pytest.mark.parametrize("T", [2, 3, 4])
def test_batched_special_and_negative_tokens(T):
    """One token with -0, inf and NaN (the plain path for the whole batch), one
    with all-negative groups: every token still exact."""
    m, _ = synth.random_case(3200, 200, 2048)
    X = tokens(3, T, 2048)
    X[0, ::7] = -0.0
    X[0, 5] = np.inf
    X[0, 900] = np.nan
    X[1] = -np.abs(X[1])
    if T > 2:
        X[2, 64:128] = -np.abs(X[2, 64:128])
    assert_bits_equal(run(m, X), expect(m, X), f"special T={T}")
    assert abg.device_status(clear=True) == 0


@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_batched_zero_groups_of_negative_tokens(T):
    """Tokens of all-negative values (token 1 of a pair mixed) with planted zero
    groups: whole rows with zero bias (-0 results for the negative tokens) and
    single zero groups; the sign of each token's zero group sums as RN's."""
    m, _ = synth.random_case(3250, 200, 2048)
    X = -np.abs(tokens(6, T, 2048))
    if T > 1:
        X[1] = np.abs(X[1])
        X[1, ::2] *= -1
    rng = np.random.default_rng(T)
    m.w[:5] = 0
    m.bias[:5] = 0.0
    for r in range(30, 70):
        g = int(rng.integers(32))
        m.w[r, 8 * g:8 * g + 8] = 0
        if r >= 50:
            m.bias[r, g] = 0.0
    exp = expect(m, X)
    assert (exp[0, :5] == 0).all() and np.signbit(exp[0, :5]).all()
    assert_bits_equal(run(m, X), exp, f"zero groups T={T}")
    assert abg.device_status(clear=True) == 0


@pytest.mark.parametrize("T", [2, 4, 6])
def test_batched_row_range_and_unaligned_scale_bias(T):
    m, _ = synth.random_case(3300, 300, 2048)
    X = tokens(4, T, 2048)
    assert_bits_equal(run(m, X, row0=37, n=200), expect(m, X, row0=37, n=200), "row range")
    sbuf = dev(np.concatenate([[0.0], m.scale.ravel()]).astype(np.float32))
    bbuf = dev(np.concatenate([[0.0], m.bias.ravel()]).astype(np.float32))
    assert_bits_equal(run(m, X, scale=sbuf[1:], bias=bbuf[1:]), expect(m, X), "unaligned scale/bias")


@pytest.mark.parametrize("T", [2, 4, 8])
def test_batched_full_4096x2048(T):
    m, _ = synth.mid()
    X = tokens(5, T, 2048)
    got = run(m, X)
    exp = expect(m, X)
    assert_bits_equal(got, exp, f"4096x2048 T={T}")
    for t in range(T):
        assert oracle.hash32(got[t]) == oracle.hash32(exp[t])


def test_batched_head_all_rows():
    m, _, _ = synth.head()
    X = tokens(6, 4, 2048)
    got = run(m, X)
    XS = np.stack([oracle.gsum(x) for x in X])
    assert_bits_equal(got, oracle.q4mm(*m.arrays(), X, XS, m.cols), "head, every row of every token")


def test_batched_empty_and_no_timeouts():
    m, _ = synth.random_case(3400, 10, 128)
    X = tokens(7, 4, 128)
    y = torch.full((4,), 7.0, device="cuda")
    abg.q4mm(dev_words(m.w), dev(m.scale), dev(m.bias), dev(X), dev(np.stack([oracle.gsum(x) for x in X])), y,
             cols=128, row0=10, n=0)
    torch.cuda.synchronize()
    assert float(y[0]) == 7.0
    assert abg.device_status(clear=True) == 0
