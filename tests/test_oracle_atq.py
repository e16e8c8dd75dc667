"""CPU pins of the oracle's gated attention token (oracle.c or_atq).

The reading is grouped-query attention at position pos with q/k RMS norms,
a rotation of column pairs (i, i + D/2) by this position's cos/sin, the new
key/value appended to the caches, softmax attention and a sigmoid output gate
(see the oracle's header).  Pinned against properties the mathematics fixes:
  - at position 0 the softmax is exactly 1: y = v * sigmoid(gate);
  - keys all equal: every probability is 1/(pos+1), y = mean(V) * sigmoid(gate);
  - one-hot values expose the probabilities, which must be softmax(q^.K^T/sqrt D)
    with the rotation computed independently as a complex multiplication, the
    query head h reading key/value head h / (Hq/Hkv);
  - the cache rows: row pos of K is the rotated, normed key (again as a complex
    product), row pos of V is v, every other row untouched;
  - ysum is the group sums of y.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle


def sigmoid64(u):
    return 1.0 / (1.0 + np.exp(-np.asarray(u, np.float64)))


def rms_rot64(u, w, cs, sn, eps=1e-6):
    u = np.asarray(u, np.float64)
    D = u.size
    un = u / np.sqrt(np.mean(u * u) + eps) * w
    z = (un[:D // 2] + 1j * un[D // 2:]) * (np.asarray(cs, np.float64) + 1j * np.asarray(sn, np.float64))
    return np.concatenate([z.real, z.imag])


def case(Hq=4, Hkv=2, D=64, P=96, pos=40, seed=0):
    rng = np.random.default_rng(seed)
    ang = rng.uniform(0, 2 * np.pi, D // 2)
    c = dict(q=rng.standard_normal(Hq * D).astype(np.float32), gate=rng.standard_normal(Hq * D).astype(np.float32),
             k=rng.standard_normal(Hkv * D).astype(np.float32), v=rng.standard_normal(Hkv * D).astype(np.float32),
             qn_w=(1 + 0.1 * rng.standard_normal(D)).astype(np.float32),
             kn_w=(1 + 0.1 * rng.standard_normal(D)).astype(np.float32),
             cos=np.cos(ang).astype(np.float32), sin=np.sin(ang).astype(np.float32),
             Kc=rng.standard_normal((Hkv, P, D)).astype(np.float32),
             Vc=rng.standard_normal((Hkv, P, D)).astype(np.float32), pos=pos)
    return c


def test_position_zero_is_the_value():
    c = case(pos=0)
    y, ys, Kc, Vc = oracle.atq(**c)
    D, per = 64, 2
    for h in range(4):
        g = h // per
        np.testing.assert_allclose(y[h * D:(h + 1) * D], c["v"][g * D:(g + 1) * D] *
                                   sigmoid64(c["gate"][h * D:(h + 1) * D]), rtol=1e-6, atol=1e-7)
    np.testing.assert_array_equal(ys, oracle.gsum(y))


def test_equal_keys_average_the_values():
    c = case(pos=37, seed=1)
    D, P, pos = 64, 96, 37
    # every cached key equal to the new one, as the oracle will store it
    _, _, Kc0, _ = oracle.atq(**dict(c, pos=0))
    for g in range(2):
        c["Kc"][g, :pos] = Kc0[g, 0]
    y, _, _, _ = oracle.atq(**c)
    for h in range(4):
        g = h // 2
        V = np.concatenate([c["Vc"][g, :pos], c["v"][None, g * D:(g + 1) * D]]).astype(np.float64)
        np.testing.assert_allclose(y[h * D:(h + 1) * D], V.mean(0) * sigmoid64(c["gate"][h * D:(h + 1) * D]),
                                   rtol=2e-5, atol=1e-6)


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (4, 1), (2, 2)])
def test_one_hot_values_reveal_softmax(Hq, Hkv):
    D, P, pos = 64, 80, 50
    c = case(Hq, Hkv, D, P, pos, seed=Hq * 10 + Hkv)
    c["Vc"][:] = 0.0
    for g in range(Hkv):
        for t in range(pos):
            c["Vc"][g, t, t] = 1.0
    c["v"][:] = 0.0
    for g in range(Hkv):
        c["v"][g * D + pos] = 1.0
    y, _, Kc, Vc = oracle.atq(**c)
    per = Hq // Hkv
    for h in range(Hq):
        g = h // per
        qr = rms_rot64(c["q"][h * D:(h + 1) * D], c["qn_w"], c["cos"], c["sin"])
        kr_new = rms_rot64(c["k"][g * D:(g + 1) * D], c["kn_w"], c["cos"], c["sin"])
        K = np.concatenate([c["Kc"][g, :pos].astype(np.float64), kr_new[None]])
        s = K @ qr / np.sqrt(D)
        p = np.exp(s - s.max())
        p /= p.sum()
        got = y[h * D:h * D + pos + 1] / sigmoid64(c["gate"][h * D:h * D + pos + 1])
        np.testing.assert_allclose(got, p, rtol=2e-4, atol=1e-7)
        assert np.all(y[h * D + pos + 1:(h + 1) * D] == 0)


def test_cache_rows():
    c = case(pos=23, seed=3)
    D = 64
    _, _, Kc, Vc = oracle.atq(**c)
    rows = np.arange(96) != 23
    assert np.array_equal(Kc[:, rows], c["Kc"][:, rows]) and np.array_equal(Vc[:, rows], c["Vc"][:, rows])
    for g in range(2):
        np.testing.assert_allclose(Kc[g, 23], rms_rot64(c["k"][g * D:(g + 1) * D], c["kn_w"], c["cos"], c["sin"]),
                                   rtol=2e-6, atol=2e-6)
        assert np.array_equal(Vc[g, 23], c["v"][g * D:(g + 1) * D])
