"""Pins for the oracle's other formats: group sizes 32 and 128 besides 64, and
scale/bias stored as bf16 or f16 besides f32 (the MLX 4-bit variants named in
"Metal: queued rmsq, swq, gdn and atq kernels and a 4-row q4mv ..." (bendlang/
bend #1440), Why).

Each check ties the oracle to something outside it: numpy's and torch's own
half-precision conversions, exact rational arithmetic on inputs where every
float operation is exact, properties of the pairwise tree, and the pinned
64-column f32 oracle on the case it covers.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest

import oracle
from affine_bit_group_gb300 import synth

from test_oracle import pack_nibbles, unpack_nibbles

ALL_BITS = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def _same_floats(a: np.ndarray, b: np.ndarray) -> bool:
    """Bitwise equal, except that any NaN matches any NaN."""
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    nan = np.isnan(a) & np.isnan(b)
    return bool(np.all(nan | (a.view(np.uint32) == b.view(np.uint32))))


def test_f16_widening_matches_numpy_for_every_pattern():
    got = oracle.half_to_f32(ALL_BITS, "f16")
    want = ALL_BITS.view(np.float16).astype(np.float32)
    assert _same_floats(got, want)


def test_bf16_widening_matches_torch_for_every_pattern():
    torch = pytest.importorskip("torch")
    got = oracle.half_to_f32(ALL_BITS, "bf16")
    want = torch.from_numpy(ALL_BITS.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    assert _same_floats(got, want)


def test_f16_subnormals_and_signed_zero():
    v = oracle.half_to_f32(np.array([0x0001, 0x8001, 0x0200, 0x8000, 0x0000], np.uint16), "f16")
    assert v[0] == 2.0 ** -24 and v[1] == -(2.0 ** -24) and v[2] == 2.0 ** -15
    assert np.signbit(v[3]) and v[3] == 0 and not np.signbit(v[4])


@pytest.mark.parametrize("gs", synth.GROUPS)
def test_gsum_ex_exact_on_integers(gs):
    rng = np.random.default_rng(gs)
    v = rng.integers(-100, 100, 384).astype(np.float32)
    s = oracle.gsum_ex(v, gs)
    assert s.shape == (384 // gs,)
    for g in range(384 // gs):
        assert float(s[g]) == float(sum(int(a) for a in v[gs * g:gs * g + gs]))


def test_gsum_ex_halves_add_to_the_double_group():
    """The pairwise tree over a power-of-two block is RN(tree(first half) + tree(second half))."""
    rng = np.random.default_rng(7)
    v = rng.normal(0, 1, 1024).astype(np.float32)
    s32, s64, s128 = (oracle.gsum_ex(v, g) for g in (32, 64, 128))
    assert np.array_equal(s64, s32[0::2] + s32[1::2])
    assert np.array_equal(s128, s64[0::2] + s64[1::2])
    assert np.array_equal(s64, oracle.gsum(v))


def test_gsum_ex_rejects_bad_group():
    with pytest.raises(ValueError):
        oracle.gsum_ex(np.zeros(96, np.float32), 64)
    with pytest.raises(ValueError):
        oracle.gsum_ex(np.zeros(128, np.float32), 16)


def exact_q4mv_fmt(q, scale, bias, x, gs):
    """Dequantize-then-dot in exact rationals with per-gs-column scale and bias (as f32 values)."""
    rows, cols = q.shape
    out = []
    for r in range(rows):
        acc = Fraction(0)
        for c in range(cols):
            g = c // gs
            acc += (Fraction(float(scale[r, g])) * int(q[r, c]) + Fraction(float(bias[r, g]))) * Fraction(float(x[c]))
        out.append(acc)
    return out


@pytest.mark.parametrize("gs", synth.GROUPS)
@pytest.mark.parametrize("sb", synth.SB_TYPES)
def test_q4mv_ex_exact_when_every_op_is_exact(gs, sb):
    """Power-of-two scales, quarter-integer biases, small integer activations:
    every rounding is exact, so y is the exact value of the definition.  A wrong
    group index for scale, bias or xsum, or a wrong nibble, changes it."""
    rng = np.random.default_rng([gs, len(sb)])
    rows, cols = 4, 256
    G = cols // gs
    q = rng.integers(0, 16, (rows, cols))
    scale = (2.0 ** rng.integers(-3, 2, (rows, G))).astype(np.float32)
    bias = (rng.integers(-16, 16, (rows, G)) * 0.25).astype(np.float32)
    x = rng.integers(-4, 5, cols).astype(np.float32)
    if sb == "f32":
        s_in, b_in = scale, bias
    else:
        s_in, b_in = synth.store16(scale, sb), synth.store16(bias, sb)
        # these values are exact in both 16-bit types
        assert np.array_equal(oracle.half_to_f32(s_in, sb).reshape(rows, G), scale)
    y = oracle.q4mv_ex(pack_nibbles(q), s_in, b_in, sb, gs, x, oracle.gsum_ex(x, gs), cols)
    assert [Fraction(float(v)) for v in y] == exact_q4mv_fmt(q, scale, bias, x, gs)


@pytest.mark.parametrize("gs", synth.GROUPS)
def test_q4mv_ex_unit_scale_is_one_tree_over_the_row(gs):
    """scale = 1, bias = 0: every group term is d itself, and a tree over groups
    of power-of-two trees is the tree over the whole row, whatever the group size."""
    rng = np.random.default_rng(30 + gs)
    rows, cols = 3, 640 if gs != 128 else 768
    q = rng.integers(0, 16, (rows, cols))
    x = rng.normal(0, 1, cols).astype(np.float32)
    G = cols // gs
    y = oracle.q4mv_ex(pack_nibbles(q), np.ones((rows, G), np.float32), np.zeros((rows, G), np.float32), "f32", gs,
                       x, oracle.gsum_ex(x, gs), cols)
    for r in range(rows):
        prods = q[r].astype(np.float32) * x  # numpy float32 multiply: RN(q*x)
        assert y[r] == oracle.tree(prods)


def test_q4mv_ex_group64_f32_is_the_pinned_product():
    m, x = synth.random_case(41, 33, 1024)
    xs = oracle.gsum(x)
    a = oracle.q4mv(*m.arrays(), x, xs, 1024)
    b = oracle.q4mv_ex(m.w, m.scale, m.bias, "f32", 64, x, oracle.gsum_ex(x, 64), 1024)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("gs", synth.GROUPS)
@pytest.mark.parametrize("sb", ["bf16", "f16"])
def test_q4mv_ex_16bit_reads_the_widened_values(gs, sb):
    m, x = synth.fmt_case(gs, sb, 9, 512)
    xs = oracle.gsum_ex(x, gs)
    y16 = oracle.q4mv_ex(m.w, m.scale, m.bias, sb, gs, x, xs, 512)
    G = 512 // gs
    s32 = oracle.half_to_f32(m.scale, sb).reshape(9, G)
    b32 = oracle.half_to_f32(m.bias, sb).reshape(9, G)
    y32 = oracle.q4mv_ex(m.w, s32, b32, "f32", gs, x, xs, 512)
    assert np.array_equal(y16.view(np.uint32), y32.view(np.uint32))


@pytest.mark.parametrize("gs", synth.GROUPS)
def test_q4mv_ex_against_float64_dequantized_matvec(gs):
    m, x = synth.fmt_case(gs, "f16", 24, 1024)
    G = 1024 // gs
    q = unpack_nibbles(m.w, 1024).astype(np.float64)
    s = oracle.half_to_f32(m.scale, "f16").reshape(24, G).astype(np.float64)
    b = oracle.half_to_f32(m.bias, "f16").reshape(24, G).astype(np.float64)
    ref = (np.repeat(s, gs, axis=1) * q + np.repeat(b, gs, axis=1)) @ x.astype(np.float64)
    y = oracle.q4mv_ex(m.w, m.scale, m.bias, "f16", gs, x, oracle.gsum_ex(x, gs), 1024)
    mag = (np.abs(np.repeat(s, gs, axis=1) * q) + np.abs(np.repeat(b, gs, axis=1))) @ np.abs(x.astype(np.float64))
    assert np.all(np.abs(y - ref) <= 1e-5 * mag)


def test_q4mv_ex_row_range_and_checks():
    m, x = synth.fmt_case(128, "bf16", 21, 256)
    xs = oracle.gsum_ex(x, 128)
    full = oracle.q4mv_ex(*m.arrays(), "bf16", 128, x, xs, 256)
    part = oracle.q4mv_ex(*m.arrays(), "bf16", 128, x, xs, 256, row0=5, n=9)
    assert np.array_equal(part, full[5:14])
    with pytest.raises(ValueError):
        oracle.q4mv_ex(*m.arrays(), "bf16", 64, x, xs, 256)  # scale has 2 groups per row, not 4
    with pytest.raises(ValueError):
        oracle.q4mv_ex(*m.arrays(), "bf16", 128, x, xs, 256, row0=20, n=2)
