"""Pins for the CPU oracle: each check ties it to something other than itself.

The oracle is the definition the CUDA library is compared against, so it is
checked here against what the pages and the mathematics fix:

* hand-derived tree sums and the affine-term rounding (tests/golden/);
* exact rational arithmetic (fractions.Fraction) of the dequantize-then-dot
  definition on inputs where every float operation is exact, and within the
  textbook forward-error bound where it is not;
* closed forms (RMS norm of a constant vector, SwiGLU limits), libm's double
  exp, the published FNV-1a test vectors.

Pages: "Array.q4mv on Metal: one kernel thread per row ..." (bendlang/bend
#1435), "Array.q4go/Array.q4wait queue Metal Q4 products ..." (#1437) and
"Metal: queued rmsq, swq, gdn and atq kernels and a 4-row q4mv ..." (#1440).
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from affine_bit_group_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32_EPS = 2.0 ** -24  # unit roundoff of binary32


def gamma(k: int) -> float:
    """Higham's gamma_k = k u / (1 - k u): the forward-error factor of k roundings."""
    return k * F32_EPS / (1 - k * F32_EPS)


def tree_depth(m: int) -> int:
    return max(0, math.ceil(math.log2(m))) if m > 1 else 0


def pack_nibbles(q: np.ndarray) -> np.ndarray:
    """Pack q[rows, cols] (0..15) into u32 words, column 8k+j in bits 4j..4j+3 of word k.

    Written here from the format statement, independently of the generators,
    so the pins below do not depend on how synth draws words.
    """
    rows, cols = q.shape
    q = q.astype(np.uint32).reshape(rows, cols // 8, 8)
    w = np.zeros((rows, cols // 8), np.uint32)
    for j in range(8):
        w |= q[:, :, j] << np.uint32(4 * j)
    return w


def unpack_nibbles(w: np.ndarray, cols: int) -> np.ndarray:
    rows = w.shape[0]
    out = np.zeros((rows, cols), np.int64)
    for c in range(cols):
        out[:, c] = (w[:, c // 8] >> np.uint32(4 * (c % 8))) & 0xF
    return out


def exact_q4mv(q, scale, bias, x):
    """Dequantize-then-dot in exact rationals: y[r] = sum_c (scale*q + bias) * x."""
    rows, cols = q.shape
    y = []
    for r in range(rows):
        acc = Fraction(0)
        for c in range(cols):
            g = c // 64
            wq = Fraction(float(scale[r, g])) * int(q[r, c]) + Fraction(float(bias[r, g]))
            acc += wq * Fraction(float(x[c]))
        y.append(acc)
    return y


def abs_terms(q, scale, bias, x):
    """sum_g |scale*d| + |bias*xsum| in exact rationals (the magnitude the bound scales)."""
    rows, cols = q.shape
    out = []
    for r in range(rows):
        acc = Fraction(0)
        for g in range(cols // 64):
            d = sum(int(q[r, c]) * Fraction(float(x[c])) for c in range(64 * g, 64 * g + 64))
            xs = sum(Fraction(float(x[c])) for c in range(64 * g, 64 * g + 64))
            acc += abs(Fraction(float(scale[r, g])) * d) + abs(Fraction(float(bias[r, g])) * xs)
        out.append(acc)
    return out


# ---------------------------------------------------------------- TREE ----

def _golden_tree():
    cases = []
    with open(os.path.join(GOLDEN, "tree_order.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            leaves, expected = line.split("|")
            cases.append(([float(v) for v in leaves.split()], float(expected)))
    return cases


@pytest.mark.parametrize("leaves,expected", _golden_tree())
def test_tree_golden(leaves, expected):
    assert float(oracle.tree(np.array(leaves, np.float32))) == expected


@pytest.mark.parametrize("m", [1, 2, 3, 5, 7, 13, 64, 96, 100, 257])
def test_tree_exact_on_integers(m):
    rng = np.random.default_rng(m)
    v = rng.integers(-1000, 1000, m).astype(np.float32)
    assert float(oracle.tree(v)) == float(sum(int(a) for a in v))


@pytest.mark.parametrize("m", [2, 3, 31, 64, 96, 1000])
def test_tree_forward_error_bound(m):
    rng = np.random.default_rng(100 + m)
    v = rng.normal(0, 1, m).astype(np.float32)
    exact = sum(Fraction(float(a)) for a in v)
    bound = gamma(tree_depth(m)) * sum(abs(Fraction(float(a))) for a in v)
    assert abs(Fraction(float(oracle.tree(v))) - exact) <= bound


def test_tree_single_element_and_signed_zero():
    assert float(oracle.tree(np.array([3.5], np.float32))) == 3.5
    z = oracle.tree(np.array([-0.0, -0.0, -0.0], np.float32))
    assert z == 0 and math.copysign(1, float(z)) == -1


def test_gsum_is_tree_of_each_group():
    rng = np.random.default_rng(5)
    v = rng.integers(-50, 50, 64 * 7).astype(np.float32)
    s = oracle.gsum(v)
    assert s.shape == (7,)
    for g in range(7):
        assert float(s[g]) == float(sum(int(a) for a in v[64 * g:64 * g + 64]))
    v2 = np.zeros(128, np.float32)
    v2[64:] = [16777216.0] + [1.0] * 63
    assert float(oracle.gsum(v2)[1]) == 16777278.0  # the 64-leaf golden case


# ---------------------------------------------------------------- q4mv ----

def test_packing_one_hot():
    """scale=1, bias=0, x = e_c gives y[r] = q[r][c]: fixes nibble order and column index."""
    rng = np.random.default_rng(11)
    rows, cols = 5, 128
    q = rng.integers(0, 16, (rows, cols))
    w = pack_nibbles(q)
    scale = np.ones((rows, cols // 64), np.float32)
    bias = np.zeros((rows, cols // 64), np.float32)
    for c in [0, 1, 7, 8, 9, 63, 64, 65, 127]:
        x = np.zeros(cols, np.float32)
        x[c] = 1.0
        y = oracle.q4mv(w, scale, bias, x, oracle.gsum(x), cols)
        assert np.array_equal(y, q[:, c].astype(np.float32)), c


def test_packing_matches_generator_words():
    """The generator's raw words decode as low-nibble-first columns."""
    m, _ = synth.tiny()
    q = unpack_nibbles(m.w, m.cols)
    assert np.array_equal(pack_nibbles(q), m.w)
    scale = np.ones_like(m.scale)
    bias = np.zeros_like(m.bias)
    x = np.zeros(m.cols, np.float32)
    x[13] = 1.0
    y = oracle.q4mv(m.w, scale, bias, x, oracle.gsum(x), m.cols)
    assert np.array_equal(y, ((m.w[:, 1] >> 20) & 0xF).astype(np.float32))


@pytest.mark.parametrize("rows,cols,seed", [(3, 64, 0), (4, 128, 1), (2, 192, 2), (3, 320, 3)])
def test_q4mv_exact_when_every_op_is_exact(rows, cols, seed):
    """Small integers and power-of-two scales: every rounding is exact, so y is the exact value."""
    rng = np.random.default_rng(seed)
    G = cols // 64
    q = rng.integers(0, 16, (rows, cols))
    scale = (2.0 ** rng.integers(-3, 2, (rows, G))).astype(np.float32)
    bias = (rng.integers(-16, 16, (rows, G)) * 0.25).astype(np.float32)
    x = rng.integers(-4, 5, cols).astype(np.float32)
    y = oracle.q4mv(pack_nibbles(q), scale, bias, x, oracle.gsum(x), cols)
    exact = exact_q4mv(q, scale, bias, x)
    assert [Fraction(float(v)) for v in y] == exact


@pytest.mark.parametrize("rows,cols,seed", [(13, 128, 0), (6, 384, 7), (4, 6144 // 8, 8)])
def test_q4mv_within_forward_error_bound(rows, cols, seed):
    """Random f32 data: |y - exact| <= gamma_(6 + depth(G) + 2) * sum_g(|s d| + |b xsum|)."""
    m, x = synth.random_case(seed, rows, cols)
    G = cols // 64
    q = unpack_nibbles(m.w, cols)
    xs = oracle.gsum(x)
    y = oracle.q4mv(m.w, m.scale, m.bias, x, xs, cols)
    exact = exact_q4mv(q, m.scale, m.bias, x)
    mag = abs_terms(q, m.scale, m.bias, x)
    k = 6 + tree_depth(G) + 2 + 1  # products + 64-tree, affine term, row tree; +1 for xsum
    for r in range(rows):
        assert abs(Fraction(float(y[r])) - exact[r]) <= gamma(k) * mag[r] * 2, r


def test_q4mv_against_float64_dequantized_matvec():
    m, x = synth.random_case(21, 40, 1024)
    q = unpack_nibbles(m.w, 1024).astype(np.float64)
    wdq = np.repeat(m.scale.astype(np.float64), 64, axis=1) * q + np.repeat(m.bias.astype(np.float64), 64, axis=1)
    ref = wdq @ x.astype(np.float64)
    y = oracle.q4mv(m.w, m.scale, m.bias, x, oracle.gsum(x), 1024)
    mag = oracle.q4mv_absmag(m.w, m.scale, m.bias, x, oracle.gsum(x), 1024)
    assert np.all(np.abs(y - ref) <= 1e-5 * mag)


def test_affine_term_golden():
    vals = {}
    with open(os.path.join(GOLDEN, "affine_term.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split("=")
                vals[k.strip()] = float(v)
    q = np.zeros((1, 64), np.int64)
    q[0, 0] = int(vals["q0"])
    x = np.zeros(64, np.float32)
    x[0], x[1] = vals["x0"], vals["x1"]
    scale = np.array([[vals["scale"]]], np.float32)
    bias = np.array([[vals["bias"]]], np.float32)
    xs = oracle.gsum(x)
    assert float(xs[0]) == 1.0
    y = oracle.q4mv(pack_nibbles(q), scale, bias, x, xs, 64)
    assert float(y[0]) == vals["expected_y"]
    assert float(y[0]) != vals["fma_would_give"]


def test_q4mv_zero_weights_reduce_to_bias_term():
    """q = 0: y = TREE_g(RN(scale*(+0)) + RN(bias*xsum)) = TREE_g(bias*xsum) exactly for these values."""
    rows, cols = 3, 256
    q = np.zeros((rows, cols), np.int64)
    scale = np.full((rows, 4), 0.5, np.float32)
    bias = np.array([[1, -2, 0.5, 4]] * rows, np.float32)
    x = np.arange(cols, dtype=np.float32) / 8.0
    xs = oracle.gsum(x)
    y = oracle.q4mv(pack_nibbles(q), scale, bias, x, xs, cols)
    expected = sum(float(bias[0, g]) * float(xs[g]) for g in range(4))
    assert np.all(y == np.float32(expected))


def test_zero_group_sum_of_negative_activations_is_minus_zero():
    """The fact the GPU kernels' sign rule rests on, checked on the plain
    definition: with every x of a 64-value group negative, products RN(q*x)
    are all <= 0, so the group sum d is zero exactly when every q of the group
    is 0, and then d = -0 (the sum of -0 products); otherwise d < 0.  With
    scale 1 and bias 0 the output is d itself (RN(1*d) + RN(0*xsum) = d + -0),
    so each row's y shows its group sum, sign of zero included."""
    rng = np.random.default_rng(11)
    rows, cols = 400, 64
    x = -np.abs(synth.activations(rng, cols)).astype(np.float32)
    x[:8] = -np.float32(1e-40)  # subnormal magnitudes: q*x still never rounds to zero
    q = rng.integers(0, 16, size=(rows, cols))
    q[::3] = 0                                      # whole groups of zeros
    q[1::3] = np.maximum(q[1::3], 1)                # no zero ...
    for r in range(1, rows, 3):
        q[r, rng.integers(0, cols)] = 0             # ... but one
    scale = np.ones((rows, 1), np.float32)
    bias = np.zeros((rows, 1), np.float32)
    xs = oracle.gsum(x)
    y = oracle.q4mv(pack_nibbles(q), scale, bias, x, xs, cols)
    allzero = (q == 0).all(axis=1)
    assert allzero.sum() == len(range(0, rows, 3))
    assert np.all((y == 0) == allzero)
    assert np.all(np.signbit(y[allzero]))
    assert np.all(y[~allzero] < 0)


def test_q4mv_row_range():
    """Array.q4go(w, x, y, r, n, cols, rows): rows r..r+n-1 of the matrix land in y[0..n)."""
    m, x = synth.random_case(9, 37, 256)
    xs = oracle.gsum(x)
    full = oracle.q4mv(*m.arrays(), x, xs, 256)
    part = oracle.q4mv(*m.arrays(), x, xs, 256, row0=11, n=17)
    assert np.array_equal(part, full[11:28])
    assert oracle.q4mv(*m.arrays(), x, xs, 256, row0=37, n=0).size == 0
    with pytest.raises(ValueError):
        oracle.q4mv(*m.arrays(), x, xs, 256, row0=30, n=8)


def test_absmag_bounds_the_output():
    m, x = synth.random_case(12, 9, 256)
    q = unpack_nibbles(m.w, 256)
    a = oracle.q4mv_absmag(*m.arrays(), x, oracle.gsum(x), 256)
    exact = exact_q4mv(q, m.scale, m.bias, x)
    mag = abs_terms(q, m.scale, m.bias, x)
    for r in range(9):
        assert abs(float(exact[r])) <= a[r] * (1 + 1e-12)
        assert abs(a[r] - float(mag[r])) <= 1e-6 * a[r]  # xsum is the rounded f32 tree sum


# ---------------------------------------------------------------- rmsq ----

def _ulp(v: np.ndarray) -> np.ndarray:
    return np.spacing(np.abs(v).astype(np.float32)).astype(np.float64)


@pytest.mark.parametrize("c", [1.0, 0.37, -2.5, 1e-3, 30.0])
def test_rmsq_constant_vector_closed_form(c):
    n = 256
    x = np.full(n, c, np.float32)
    w = np.random.default_rng(1).uniform(0.5, 1.5, n).astype(np.float32)
    xn, xs = oracle.rmsq(x, w, 1e-6)
    c64 = float(np.float32(c))
    ref = c64 * w.astype(np.float64) / math.sqrt(c64 * c64 + float(np.float32(1e-6)))
    assert np.all(np.abs(xn - ref) <= 3 * _ulp(ref))


def test_rmsq_against_float64():
    rng = np.random.default_rng(2)
    n = 2048
    x = rng.normal(0, 1, n).astype(np.float32)
    w = rng.uniform(0.5, 1.5, n).astype(np.float32)
    xn, xs = oracle.rmsq(x, w, 1e-6)
    x64 = x.astype(np.float64)
    r = 1.0 / math.sqrt(np.mean(x64 * x64) + float(np.float32(1e-6)))
    ref = x64 * r * w.astype(np.float64)
    assert np.all(np.abs(xn - ref) <= 4 * _ulp(ref) + 1e-30)
    ref_sums = ref.reshape(-1, 64).sum(axis=1)
    assert np.all(np.abs(xs - ref_sums) <= 1e-5 * np.abs(ref).reshape(-1, 64).sum(axis=1))
    assert np.array_equal(xs, oracle.gsum(xn))


def test_rmsq_one_hot_and_scale():
    n = 128
    x = np.zeros(n, np.float32)
    x[70] = 4.0
    w = np.full(n, 0.5, np.float32)
    xn, xs = oracle.rmsq(x, w, 1e-6)
    ref = 4.0 / math.sqrt(16.0 / n + float(np.float32(1e-6))) * 0.5
    assert abs(float(xn[70]) - ref) <= 3 * np.spacing(np.float32(ref))
    assert np.all(xn[np.arange(n) != 70] == 0)
    assert float(xs[0]) == 0 and float(xs[1]) == float(xn[70])
    # scaling x by a power of two leaves the output nearly unchanged (eps breaks exactness)
    rng = np.random.default_rng(3)
    x = rng.normal(0, 1, n).astype(np.float32)
    a, _ = oracle.rmsq(x, w, 1e-6)
    b, _ = oracle.rmsq(x * np.float32(8), w, 1e-6)
    assert np.all(np.abs(a - b) <= 1e-6 * np.abs(a) + 1e-7)


def test_rmsq_rejects_ragged_n():
    with pytest.raises(ValueError):
        oracle.rmsq(np.ones(100, np.float32), np.ones(100, np.float32))


# ---------------------------------------------------------------- EXP -----

def test_exp_constants_are_rounded_reciprocal_factorials():
    """The polynomial's coefficients are RN(1/i!) and ln 2 is split as the header states."""
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    for i, bits in enumerate(["0x3F800000u", "0x3F800000u", "0x3F000000u", "0x3E2AAAABu", "0x3D2AAAABu",
                              "0x3C088889u", "0x3AB60B61u", "0x39500D01u"]):
        assert np.float32(1.0 / math.factorial(i)).view(np.uint32) == int(bits[:-1], 16)
        assert bits in src
    ln2 = np.float32(math.log(2)).view(np.uint32)
    hi = np.uint32(ln2 & np.uint32(0xFFFFF000))
    assert hi == 0x3F317000
    lo = np.float32(math.log(2) - float(hi.view(np.float32)))
    assert lo.view(np.uint32) == 0x3805FDF4
    assert np.float32(1 / math.log(2)).view(np.uint32) == 0x3FB8AA3B


def _exp_ulp_error(v: np.ndarray) -> np.ndarray:
    got = oracle.exp(v).astype(np.float64)
    ref = np.exp(v.astype(np.float64))
    ulp = np.spacing(np.minimum(ref, np.finfo(np.float32).max).astype(np.float32)).astype(np.float64)
    ulp = np.maximum(ulp, 2.0 ** -149)
    return np.abs(got - ref) / ulp


def test_exp_against_libm_sampled():
    """Every 37th float in [-104, 89] (about 60M values): within 2 ulp of double exp."""
    worst = 0.0
    lo_neg, hi_neg = np.float32(-0.0).view(np.uint32), np.float32(-104.0).view(np.uint32)
    lo_pos, hi_pos = np.uint32(0), np.float32(88.72).view(np.uint32)
    for lo, hi in [(lo_neg, hi_neg), (lo_pos, hi_pos)]:
        for start in range(int(lo), int(hi), 37 * 2_000_000):
            bits = np.arange(start, min(int(hi), start + 37 * 2_000_000), 37, dtype=np.uint64).astype(np.uint32)
            worst = max(worst, float(_exp_ulp_error(bits.view(np.float32)).max()))
    assert worst <= 2.0, worst


def test_exp_dense_window_and_specials():
    bits = np.arange(np.float32(-1.0).view(np.uint32) - 400_000, np.float32(-1.0).view(np.uint32) + 400_000,
                     dtype=np.uint32)
    assert _exp_ulp_error(bits.view(np.float32)).max() <= 2.0
    v = np.array([0.0, -0.0, 1.0, 89.5, 1000.0, -104.5, -1000.0, np.inf, -np.inf, np.nan], np.float32)
    e = oracle.exp(v)
    assert e[0] == 1.0 and e[1] == 1.0
    assert e[2] == np.float32(math.e)
    assert np.isinf(e[3]) and np.isinf(e[4]) and np.isinf(e[7])
    assert e[5] == 0 and e[6] == 0 and e[8] == 0
    assert np.isnan(e[9])


# ---------------------------------------------------------------- swq -----

def test_swq_against_float64():
    rng = np.random.default_rng(4)
    n = 6144
    a = (rng.normal(0, 3, 2 * n)).astype(np.float32)
    o, os_ = oracle.swq(a)
    g = a[:n].astype(np.float64)
    u = a[n:].astype(np.float64)
    ref = g / (1.0 + np.exp(-g)) * u
    assert np.all(np.abs(o - ref) <= 8 * _ulp(ref) + 1e-38)
    assert np.array_equal(os_, oracle.gsum(o))


def test_swq_limits():
    n = 64
    g = np.zeros(n, np.float32)
    g[1], g[2], g[3], g[4] = 200.0, -200.0, 30.0, -0.0
    u = np.full(n, 3.0, np.float32)
    o, _ = oracle.swq(np.concatenate([g, u]))
    assert o[0] == 0.0
    assert o[1] == np.float32(600.0)  # silu(g) = g once exp(-g) underflows
    assert o[2] == 0.0 and math.copysign(1, float(o[2])) == -1  # g / inf = -0
    assert o[3] == np.float32(np.float32(30.0 / (1 + math.exp(-30.0))) * 3.0)
    assert math.copysign(1, float(o[4])) == -1


def test_swq_rejects_ragged_n():
    with pytest.raises(ValueError):
        oracle.swq(np.ones(2 * 32, np.float32))


# ---------------------------------------------------------------- hash ----

def test_fnv1a_published_vectors():
    assert oracle.fnv1a(b"") == 0x811C9DC5
    assert oracle.fnv1a(b"a") == 0xE40C292C
    assert oracle.fnv1a(b"foobar") == 0xBF9CF968


def test_hash32_is_fnv1a_of_little_endian_bytes():
    y = np.array([1.0, -2.5, 3.25e-7, 0.0], np.float32)
    assert oracle.hash32(y) == oracle.fnv1a(y.astype("<f4").tobytes())


# --------------------------------------------------------- decode token ---

def test_decode_token_wiring_small():
    """A two-layer model of the decode-token stage list, checked stage by stage.

    Each stage's input is what the stage list says it is: rmsq of the hidden
    vector feeds q/k/v; the o product reads q with its group sums; rmsq of o
    feeds gate and up; swq of [gate | up] feeds down, whose output is the next
    layer's hidden vector; the head reads rmsq of the last hidden vector.
    Checked in float64 (dequantize-then-dot) within a relative 1e-4.
    """
    model, h = synth.decode_model(seed=7, n_layers=2, hidden=128, mlp=192, head_rows=96, q_rows=256, kv_rows=64)
    logits, trace, (xf, xfs) = oracle.decode_token(model, h, keep=True)

    def dq(m, v):
        q = unpack_nibbles(m.w, m.cols).astype(np.float64)
        w = np.repeat(m.scale.astype(np.float64), 64, 1) * q + np.repeat(m.bias.astype(np.float64), 64, 1)
        return w @ v.astype(np.float64)

    def rms(v, wt):
        v = v.astype(np.float64)
        return v / math.sqrt(np.mean(v * v) + float(np.float32(1e-6))) * wt

    def close(a, b, tol=1e-4):
        return np.all(np.abs(a - b) <= tol * (np.abs(b).max() + 1e-30))

    hid = h
    for L, t in zip(model.layers, trace):
        assert close(t["xn"], rms(hid, L.rms1))
        assert close(t["q"], dq(L.q, t["xn"])) and close(t["k"], dq(L.k, t["xn"])) and close(t["v"], dq(L.v, t["xn"]))
        assert t["q"].size == 256 and t["k"].size == 64
        assert close(t["o"], dq(L.o, t["q"]))
        assert close(t["xn2"], rms(t["o"], L.rms2))
        assert close(t["gate"], dq(L.gate, t["xn2"])) and close(t["up"], dq(L.up, t["xn2"]))
        g = t["gate"].astype(np.float64)
        assert close(t["s"], g / (1 + np.exp(-g)) * t["up"])
        assert close(t["h"], dq(L.down, t["s"]))
        hid = t["h"]
    assert close(xf, rms(hid, model.rms_final))
    assert close(logits, dq(model.head, xf))


# ------------------------------------------------------------- batched ----

def test_q4mm_is_the_product_per_token_exactly():
    """Batched tokens: with small integers and power-of-two scales every row of Y is
    the exact dequantize-then-dot value for its own token (tokens never mix)."""
    rng = np.random.default_rng(77)
    rows, cols, T = 5, 192, 3
    G = cols // 64
    q = rng.integers(0, 16, (rows, cols))
    scale = (2.0 ** rng.integers(-3, 2, (rows, G))).astype(np.float32)
    bias = (rng.integers(-16, 16, (rows, G)) * 0.25).astype(np.float32)
    X = rng.integers(-4, 5, (T, cols)).astype(np.float32)
    XS = np.stack([oracle.gsum(x) for x in X])
    Y = oracle.q4mm(pack_nibbles(q), scale, bias, X, XS, cols)
    assert Y.shape == (T, rows)
    for t in range(T):
        assert [Fraction(float(v)) for v in Y[t]] == exact_q4mv(q, scale, bias, X[t])


def test_q4mm_token_order_and_single_token():
    m, x = synth.random_case(78, 19, 256)
    rng = np.random.default_rng(79)
    X = np.stack([x, synth.activations(rng, 256), synth.activations(rng, 256)])
    XS = np.stack([oracle.gsum(v) for v in X])
    Y = oracle.q4mm(*m.arrays(), X, XS, 256)
    assert np.array_equal(Y[0], oracle.q4mv(*m.arrays(), x, oracle.gsum(x), 256))
    P = oracle.q4mm(*m.arrays(), X[::-1], XS[::-1], 256)
    assert np.array_equal(P, Y[::-1])
    with pytest.raises(ValueError):
        oracle.q4mm(*m.arrays(), X, XS[:2], 256)
