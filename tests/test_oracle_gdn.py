"""CPU pins of the oracle's LOG and gdn mixer (oracle.c or_log, or_gdn).

gdn follows the published gated DeltaNet recurrence with the library's own
binary32 steps (see the oracle's header for the reading); these tests pin it
to properties the mathematics fixes, not to a retyping of its formula:
  - LOG within 3 ulp of the correctly rounded logarithm, exact specials;
  - the conv window: one-hot taps select state entries oldest first, then x;
    the state shifts by one;
  - decay alone (beta = 0): S' = alpha S with alpha = exp(-exp(A_log) *
    softplus(a + dt_bias)) evaluated in float64;
  - the delta rule (alpha = beta = 1): after the update S'^T k^ = v, since k^
    is a unit vector -- this fails for a wrong sign, a transposed state or an
    unnormalized key;
  - zero state: o = beta (k^ . q^) v with q^ scaled by 1/sqrt(D), read back
    through a gated norm whose eps dominates (the norm is then a known scale),
    and with the default eps, y = o / sqrt(mean(o^2) + eps) * nw * silu(z);
  - ysum is the group sums of y.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle


def ulps(a, b):
    ai = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    bi = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    ai = np.where(ai < 0, -(ai & 0x7FFFFFFF), ai)
    bi = np.where(bi < 0, -(bi & 0x7FFFFFFF), bi)
    return np.abs(ai - bi)


def test_log_specials_and_exact_points():
    v = np.array([1.0, 0.0, -0.0, -1.0, np.inf, np.nan, -np.inf], np.float32)
    got = oracle.log(v)
    assert got[0] == 0.0 and not np.signbit(got[0])
    assert got[1] == -np.inf and got[2] == -np.inf
    assert np.isnan(got[3]) and got[4] == np.inf and np.isnan(got[5]) and np.isnan(got[6])


def test_log_within_3_ulp():
    rng = np.random.default_rng(11)
    bits = rng.integers(1, 0x7F800000, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    v = np.concatenate([bits.view(np.float32), np.linspace(0.5, 2.0, 100_001, dtype=np.float32),
                        np.float32(2.0) ** np.arange(-149, 128, dtype=np.float32)])
    ref = np.log(v.astype(np.float64)).astype(np.float32)
    assert ulps(oracle.log(v), ref).max() <= 3


def silu64(u):
    u = np.asarray(u, np.float64)
    return u / (1.0 + np.exp(-u))


def case(H=2, D=64, K=4, seed=0):
    rng = np.random.default_rng(seed)
    C = 3 * H * D
    return dict(x=rng.standard_normal(C).astype(np.float32),
                conv=rng.standard_normal((C, K)).astype(np.float32) * 0.5,
                state=rng.standard_normal((C, K - 1)).astype(np.float32),
                a=rng.standard_normal(H).astype(np.float32), b=rng.standard_normal(H).astype(np.float32),
                z=rng.standard_normal(H * D).astype(np.float32),
                A_log=(rng.standard_normal(H) * 0.5).astype(np.float32),
                dt_bias=(rng.standard_normal(H) * 0.5).astype(np.float32),
                nw=(1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32),
                S=(rng.standard_normal((H, D, D)) * 0.1).astype(np.float32))


def one_hot_conv(C, K, tap):
    conv = np.zeros((C, K), np.float32)
    conv[:, tap] = 1.0
    return conv


def acts(c, tap):
    """The activations a one-hot tap selects: silu of that window entry."""
    K = c["conv"].shape[1]
    win = np.concatenate([c["state"], c["x"][:, None]], axis=1)
    return silu64(win[:, tap]), K


def test_state_shift_is_exact():
    c = case()
    _, _, _, st = oracle.gdn(**c)
    exp = np.concatenate([c["state"][:, 1:], c["x"][:, None]], axis=1)
    assert np.array_equal(st, exp)


@pytest.mark.parametrize("tap", [0, 1, 2, 3])
def test_conv_window_order(tap):
    """alpha = beta = 1 on a zero state: S' = k^ (x) v, so v is read back from S';
    a one-hot tap at `tap` must select window entry `tap` (state oldest first,
    then x)."""
    H, D, K = 2, 64, 4
    c = case(H, D, K, seed=tap)
    c["conv"] = one_hot_conv(3 * H * D, K, tap)
    c["S"] = np.zeros((H, D, D), np.float32)
    c["A_log"] = np.full(H, -np.inf, np.float32)  # decay exp(-0) = 1
    c["b"] = np.full(H, 100.0, np.float32)  # beta = 1
    _, _, S1, _ = oracle.gdn(**c)
    act, _ = acts(c, tap)
    for h in range(H):
        k = act[H * D + h * D:H * D + (h + 1) * D]
        v = act[2 * H * D + h * D:2 * H * D + (h + 1) * D]
        kh = k / np.sqrt(np.sum(k * k) + 1e-6)
        i = int(np.argmax(np.abs(kh)))
        np.testing.assert_allclose(S1[h][i] / kh[i], v, rtol=2e-5, atol=1e-6)


def test_decay_alone():
    """beta = 0: the update adds nothing, S' = alpha S."""
    H, D = 3, 64
    c = case(H, D, seed=5)
    c["b"] = np.full(H, -200.0, np.float32)
    _, _, S1, _ = oracle.gdn(**c)
    u = c["a"].astype(np.float64) + c["dt_bias"]
    alpha = np.exp(-np.exp(c["A_log"].astype(np.float64)) * np.log1p(np.exp(u)))
    for h in range(H):
        mask = np.abs(c["S"][h]) > 1e-3
        np.testing.assert_allclose(S1[h][mask] / c["S"][h][mask], alpha[h], rtol=5e-6)


def test_delta_rule_writes_v_at_k():
    """alpha = beta = 1: S'^T k^ = S^T k^ + (k^.k^)(v - S^T k^) = v."""
    H, D = 2, 128
    c = case(H, D, seed=7)
    c["A_log"] = np.full(H, -np.inf, np.float32)
    c["b"] = np.full(H, 100.0, np.float32)
    c["conv"] = one_hot_conv(3 * H * D, 4, 3)
    _, _, S1, _ = oracle.gdn(**c)
    act, _ = acts(c, 3)
    for h in range(H):
        k = act[H * D + h * D:H * D + (h + 1) * D]
        v = act[2 * H * D + h * D:2 * H * D + (h + 1) * D]
        kh = k / np.sqrt(np.sum(k * k) + 1e-6)
        got = S1[h].astype(np.float64).T @ kh
        np.testing.assert_allclose(got, v, rtol=0, atol=2e-5 * np.abs(v).max() + 1e-6)
    # a transposed state would not satisfy it
    assert not np.allclose(S1[0].astype(np.float64) @ kh, v, atol=1e-3)


def test_zero_state_output():
    """S = 0, any alpha: S' = beta k^ (x) v and o = beta (k^ . q^) v, q^ = q/|q|/sqrt(D).
    With eps_n = 1e30 the gated norm is the known scale 1e-15; with the default
    eps_n, y = o / sqrt(mean(o^2) + eps_n) * nw * silu(z)."""
    H, D = 2, 128
    c = case(H, D, seed=9)
    c["S"] = np.zeros((H, D, D), np.float32)
    c["conv"] = one_hot_conv(3 * H * D, 4, 3)
    act, _ = acts(c, 3)
    beta = 1.0 / (1.0 + np.exp(-c["b"].astype(np.float64)))
    big = dict(c, eps_n=1e30)
    y, ys, _, _ = oracle.gdn(**big)
    y2, _, _, _ = oracle.gdn(**c)
    for h in range(H):
        q = act[h * D:(h + 1) * D]
        k = act[H * D + h * D:H * D + (h + 1) * D]
        v = act[2 * H * D + h * D:2 * H * D + (h + 1) * D]
        qh = q / np.sqrt(np.sum(q * q) + 1e-6) / np.sqrt(D)
        kh = k / np.sqrt(np.sum(k * k) + 1e-6)
        o = beta[h] * np.dot(kh, qh) * v
        gate = c["nw"] * silu64(c["z"][h * D:(h + 1) * D])
        np.testing.assert_allclose(y[h * D:(h + 1) * D], o * 1e-15 * gate, rtol=3e-5, atol=1e-22)
        np.testing.assert_allclose(y2[h * D:(h + 1) * D], o / np.sqrt(np.mean(o * o) + 1e-6) * gate, rtol=3e-5,
                                   atol=1e-6)
    np.testing.assert_array_equal(ys, oracle.gsum(y))
