"""GPU parity of the gated DeltaNet mixer (abg_gdn) against the oracle.

Every output -- y, its group sums, the updated state S and the conv state --
must be bit-for-bit the oracle's, for head dimensions 64, 128 and 256, 2 to 8
conv taps, one to 16 heads, several tokens in a row (the state carried from
token to token), and the edge cases of the decay and gate: beta 0 and 1,
alpha 1, softplus past its threshold, an all-zero query.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from affine_bit_group_gb300 import synth
from helpers import assert_bits_equal, dev, empty, host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
abg = pytest.importorskip("affine_bit_group_gb300")


def run_gdn(c, tokens=1, xs=None):
    """Runs `tokens` tokens on the device and in the oracle, comparing after each."""
    H, D = c["S"].shape[0], c["S"].shape[1]
    d = {k: dev(v) for k, v in c.items()}
    S_ref, st_ref = c["S"], c["state"]
    for t in range(tokens):
        x = c["x"] if xs is None else xs[t]
        d["x"] = dev(x)
        y, ys = empty(H * D), empty(H * D // 64)
        abg.gdn(d["x"], d["conv"], d["state"], d["a"], d["b"], d["z"], d["A_log"], d["dt_bias"], d["nw"], d["S"], y,
                ys)
        torch.cuda.synchronize()
        ref = dict(c, x=x, S=S_ref, state=st_ref)
        ey, eys, S_ref, st_ref = oracle.gdn(**ref)
        assert_bits_equal(host(y), ey, f"y, token {t}")
        assert_bits_equal(host(ys), eys, f"ysum, token {t}")
        assert_bits_equal(host(d["S"]).reshape(S_ref.shape), S_ref, f"S, token {t}")
        assert_bits_equal(host(d["state"]).reshape(st_ref.shape), st_ref, f"conv state, token {t}")
    assert abg.device_status(clear=True) == 0


@pytest.mark.parametrize("H,D,K", [(16, 128, 4), (1, 64, 2), (3, 256, 8), (5, 128, 3), (2, 64, 7)])
def test_gdn_bit_exact(H, D, K):
    run_gdn(synth.gdn_case(np.random.default_rng([H, D, K]), H, D, K))


def test_gdn_tokens_carry_state():
    rng = np.random.default_rng(42)
    c = synth.gdn_case(rng)
    xs = [rng.standard_normal(c["x"].size).astype(np.float32) for _ in range(4)]
    run_gdn(c, tokens=4, xs=xs)


def test_gdn_gate_and_decay_edges():
    """beta = 0 and 1 (b = -200, 100), alpha = 1 (A_log = -inf), softplus past
    20 (a = 30), and a head whose query is zero (x = 0 with zero state and taps
    on the current input: SILU(0) = 0)."""
    H, D, K = 6, 128, 4
    c = synth.gdn_case(np.random.default_rng(7), H, D, K)
    c["b"][:] = [-200.0, 100.0, 0.0, 0.0, 1.0, -1.0]
    c["A_log"][2] = -np.inf
    c["a"][3] = 30.0
    c["dt_bias"][3] = 1.0
    c["x"][5 * D:6 * D] = 0.0                    # head 5's query channels
    c["state"][5 * D:6 * D] = 0.0
    c["conv"][5 * D:6 * D] = 0.0
    c["conv"][5 * D:6 * D, K - 1] = 1.0
    run_gdn(c)


def run_atq(c, tokens=1):
    """Runs tokens at positions pos, pos+1, ... (same q, k, v) on the device and
    in the oracle, comparing y, ysum and both caches after each."""
    d = {k: dev(v) for k, v in c.items() if k != "pos"}
    Hkv, P, D = c["Kc"].shape
    Hq = c["q"].size // D
    Kr, Vr = c["Kc"], c["Vc"]
    for t in range(tokens):
        pos = c["pos"] + t
        y, ys = empty(Hq * D), empty(Hq * D // 64)
        abg.atq(d["q"], d["gate"], d["k"], d["v"], d["qn_w"], d["kn_w"], d["cos"], d["sin"], d["Kc"], d["Vc"], y, ys,
                pos=pos)
        torch.cuda.synchronize()
        ey, eys, Kr, Vr = oracle.atq(**dict(c, Kc=Kr, Vc=Vr, pos=pos))
        assert_bits_equal(host(y), ey, f"y at {pos}")
        assert_bits_equal(host(ys), eys, f"ysum at {pos}")
        assert_bits_equal(host(d["Kc"]).reshape(Kr.shape), Kr, f"K cache at {pos}")
        assert_bits_equal(host(d["Vc"]).reshape(Vr.shape), Vr, f"V cache at {pos}")
    assert abg.device_status(clear=True) == 0


@pytest.mark.parametrize("Hq,Hkv,D,P,pos", [(8, 2, 256, 4096, 2047), (4, 4, 64, 64, 0), (4, 2, 128, 300, 31),
                                            (4, 2, 128, 300, 32), (6, 3, 64, 200, 33), (2, 1, 256, 8192, 8191),
                                            (8, 1, 128, 5000, 1000)])
def test_atq_bit_exact(Hq, Hkv, D, P, pos):
    run_atq(synth.atq_case(np.random.default_rng([Hq, Hkv, D, P, pos]), Hq, Hkv, D, P, pos))


def test_atq_tokens_append_rows():
    run_atq(synth.atq_case(np.random.default_rng(5), 4, 2, 128, 256, 60), tokens=5)
