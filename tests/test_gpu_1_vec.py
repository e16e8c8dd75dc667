"""GPU parity of the activation producers (gsum, rmsq, swq) against the oracle.

Tree mode is bit-for-bit equal to the oracle, including the library's own
exponential inside swq; fast mode is checked against float64 closed forms.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
from helpers import assert_bits_equal, dev, empty, host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
abg = pytest.importorskip("affine_bit_group_gb300")


@pytest.mark.parametrize("n", [64, 128, 192, 2048, 6144, 64 * 1000, 64 * 4096])
def test_gsum_tree(n):
    v = np.random.default_rng(n).normal(0, 2, n).astype(np.float32)
    s = empty(n // 64)
    abg.gsum(dev(v), s)
    torch.cuda.synchronize()
    assert_bits_equal(host(s), oracle.gsum(v), f"gsum {n}")


@pytest.mark.parametrize("n", [64, 128, 192, 2048, 6144, 64 * 1000, 1 << 20])
def test_rmsq_tree(n):
    rng = np.random.default_rng(n + 1)
    x = rng.normal(0, 1, n).astype(np.float32)
    wt = rng.uniform(0.5, 1.5, n).astype(np.float32)
    xn, xs = empty(n), empty(n // 64)
    abg.rmsq(dev(x), dev(wt), xn, xs, eps=1e-6)
    torch.cuda.synchronize()
    exn, exs = oracle.rmsq(x, wt, 1e-6)
    assert_bits_equal(host(xn), exn, f"rmsq xn {n}")
    assert_bits_equal(host(xs), exs, f"rmsq xsum {n}")


def test_rmsq_fast_close():
    rng = np.random.default_rng(7)
    n = 2048
    x = rng.normal(0, 1, n).astype(np.float32)
    wt = rng.uniform(0.5, 1.5, n).astype(np.float32)
    xn, xs = empty(n), empty(n // 64)
    abg.rmsq(dev(x), dev(wt), xn, xs, eps=1e-6, mode=abg.FAST)
    torch.cuda.synchronize()
    x64 = x.astype(np.float64)
    ref = x64 / math.sqrt(np.mean(x64 * x64) + 1e-6) * wt
    assert np.all(np.abs(host(xn) - ref) <= 1e-5 * np.abs(ref) + 1e-30)


@pytest.mark.parametrize("n", [64, 6144, 64 * 777])
def test_swq_tree(n):
    rng = np.random.default_rng(n + 2)
    a = rng.normal(0, 3, 2 * n).astype(np.float32)
    o, os_ = empty(n), empty(n // 64)
    abg.swq(dev(a), o, os_)
    torch.cuda.synchronize()
    eo, eos = oracle.swq(a)
    assert_bits_equal(host(o), eo, f"swq o {n}")
    assert_bits_equal(host(os_), eos, f"swq osum {n}")


def test_swq_exp_over_wide_range():
    """silu(g) * 1 for 4M values of g spread over every exponent the exponential sees."""
    rng = np.random.default_rng(11)
    n = 1 << 22
    bits = rng.integers(0, 2 ** 32, n, dtype=np.uint64).astype(np.uint32)
    g = bits.view(np.float32).copy()
    g[np.abs(g) > 120] = np.float32(rng.uniform(-120, 120))  # keep most values where exp is non-trivial
    g[:8] = [0.0, -0.0, 88.7, -88.7, 103.9, -103.9, np.inf, np.nan]
    a = np.concatenate([g, np.ones(n, np.float32)])
    o, os_ = empty(n), empty(n // 64)
    abg.swq(dev(a), o, os_)
    torch.cuda.synchronize()
    eo, _ = oracle.swq(a)
    assert_bits_equal(host(o), eo, "silu")


def test_swq_fast_close():
    rng = np.random.default_rng(12)
    n = 6144
    a = rng.normal(0, 3, 2 * n).astype(np.float32)
    o, os_ = empty(n), empty(n // 64)
    abg.swq(dev(a), o, os_, mode=abg.FAST)
    torch.cuda.synchronize()
    g, u = a[:n].astype(np.float64), a[n:].astype(np.float64)
    ref = g / (1 + np.exp(-g)) * u
    assert np.all(np.abs(host(o) - ref) <= 1e-5 * np.abs(ref) + 1e-30)


def test_argument_errors_raise():
    x = torch.zeros(100, device="cuda")
    with pytest.raises(abg.AbgError) as e:
        abg.rmsq(x, x.clone(), torch.zeros(100, device="cuda"), torch.zeros(2, device="cuda"))
    assert e.value.status == 3
    x = torch.zeros(128, device="cuda")
    with pytest.raises(abg.AbgError) as e:
        abg.swq(x, x[:64], torch.zeros(1, device="cuda"))
    assert e.value.status == 4
