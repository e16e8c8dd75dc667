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
from helpers import assert_bits_equal, dev, dev_words, empty, host

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
                                            (8, 1, 128, 5000, 1000), (6, 2, 64, 130, 127), (8, 2, 64, 700, 64),
                                            (16, 4, 128, 1000, 511), (3, 1, 256, 100, 95)])
def test_atq_bit_exact(Hq, Hkv, D, P, pos):
    run_atq(synth.atq_case(np.random.default_rng([Hq, Hkv, D, P, pos]), Hq, Hkv, D, P, pos))


def test_atq_tokens_append_rows():
    run_atq(synth.atq_case(np.random.default_rng(5), 4, 2, 128, 256, 60), tokens=5)


def test_mixers_as_stage_graph_nodes():
    """gdn and atq as nodes of one stage of a stage graph, each followed in the
    next stage by a product reading its y and group sums.  Every replay is the
    oracle's next token, bit for bit (the gdn state carried, the atq cache row
    rewritten), also with a direct atq call at a later position (which grows
    the calls' shared buffer) between replays: the graph's atq has its own."""
    rng = np.random.default_rng(11)
    cg = synth.gdn_case(rng)                              # y: 16 x 128
    ca = synth.atq_case(rng, 4, 2, 128, 600, 300)        # y: 4 x 128
    Hg, Dg = cg["S"].shape[0], cg["S"].shape[1]
    Dq = ca["Kc"].shape[2]
    Hq = ca["q"].size // Dq
    mg, ma = synth.q4_matrix(rng, 1000, Hg * Dg), synth.q4_matrix(rng, 700, Hq * Dq)
    g_ = {k: dev(v) for k, v in cg.items()}
    a_ = {k: dev(v) for k, v in ca.items() if k != "pos"}
    wg, wa = [dev_words(mg.w), dev(mg.scale), dev(mg.bias)], [dev_words(ma.w), dev(ma.scale), dev(ma.bias)]
    yg, ysg, ya, ysa = empty(Hg * Dg), empty(Hg * Dg // 64), empty(Hq * Dq), empty(Hq * Dq // 64)
    og, oa = empty(mg.rows), empty(ma.rows)
    N = abg.Node
    nodes = [N.gdn(0, g_["x"], g_["conv"], g_["state"], g_["a"], g_["b"], g_["z"], g_["A_log"], g_["dt_bias"],
                   g_["nw"], g_["S"], yg, ysg),
             N.atq(0, a_["q"], a_["gate"], a_["k"], a_["v"], a_["qn_w"], a_["kn_w"], a_["cos"], a_["sin"], a_["Kc"],
                   a_["Vc"], ya, ysa, pos=ca["pos"]),
             N.q4mv(1, *wg, og, Hg * Dg, yg, ysg),
             N.q4mv(1, *wa, oa, Hq * Dq, ya, ysa)]
    keep = list(g_.values()) + list(a_.values()) + wg + wa + [yg, ysg, ya, ysa, og, oa]
    graph = abg.StageGraph(nodes, keep=keep)
    assert graph.launches == 7  # gdn, the four atq launches, two products
    other = synth.atq_case(np.random.default_rng(12), 8, 2, 256, 4096, 4000)
    o_ = {k: dev(v) for k, v in other.items() if k != "pos"}
    S_ref, st_ref, Kr, Vr = cg["S"], cg["state"], ca["Kc"], ca["Vc"]
    for t in range(3):
        graph.launch()
        if t == 1:
            abg.atq(o_["q"], o_["gate"], o_["k"], o_["v"], o_["qn_w"], o_["kn_w"], o_["cos"], o_["sin"], o_["Kc"],
                    o_["Vc"], empty(8 * 256), empty(32), pos=other["pos"])
        torch.cuda.synchronize()
        ey, eys, S_ref, st_ref = oracle.gdn(**dict(cg, S=S_ref, state=st_ref))
        ay, ays, Kr, Vr = oracle.atq(**dict(ca, Kc=Kr, Vc=Vr))
        assert_bits_equal(host(yg), ey, f"gdn y, replay {t}")
        assert_bits_equal(host(ysg), eys, f"gdn ysum, replay {t}")
        assert_bits_equal(host(g_["S"]).reshape(S_ref.shape), S_ref, f"gdn S, replay {t}")
        assert_bits_equal(host(g_["state"]).reshape(st_ref.shape), st_ref, f"gdn conv state, replay {t}")
        assert_bits_equal(host(ya), ay, f"atq y, replay {t}")
        assert_bits_equal(host(ysa), ays, f"atq ysum, replay {t}")
        assert_bits_equal(host(a_["Kc"]).reshape(Kr.shape), Kr, f"K cache, replay {t}")
        assert_bits_equal(host(a_["Vc"]).reshape(Vr.shape), Vr, f"V cache, replay {t}")
        assert_bits_equal(host(og), oracle.q4mv(mg.w, mg.scale, mg.bias, ey, eys, Hg * Dg), f"gdn product {t}")
        assert_bits_equal(host(oa), oracle.q4mv(ma.w, ma.scale, ma.bias, ay, ays, Hq * Dq), f"atq product {t}")
    graph.close()
    assert abg.device_status(clear=True) == 0


def test_atq_tokens_back_to_back():
    """Four tokens at positions 127..130 (across a chunk boundary) queued back
    to back on one stream, with no sync between them: each token's first launch
    reads the cache rows below its position before waiting for the launch
    before it, so the row the previous token wrote must already be there.
    Every output and both caches bit-exact to the oracle."""
    c = synth.atq_case(np.random.default_rng(9), 8, 2, 128, 300, 127)
    d = {k: dev(v) for k, v in c.items() if k != "pos"}
    Hkv, P, D = c["Kc"].shape
    Hq = c["q"].size // D
    rng = np.random.default_rng(10)
    ins = [{k: rng.standard_normal(c[k].size).astype(np.float32) for k in ("q", "gate", "k", "v")} for _ in range(4)]
    dins = [{k: dev(v) for k, v in t.items()} for t in ins]
    ys = [(empty(Hq * D), empty(Hq * D // 64)) for _ in ins]
    for t in range(4):
        abg.atq(dins[t]["q"], dins[t]["gate"], dins[t]["k"], dins[t]["v"], d["qn_w"], d["kn_w"], d["cos"], d["sin"],
                d["Kc"], d["Vc"], ys[t][0], ys[t][1], pos=127 + t)
    torch.cuda.synchronize()
    Kr, Vr = c["Kc"], c["Vc"]
    for t in range(4):
        ey, eys, Kr, Vr = oracle.atq(**dict(c, **ins[t], Kc=Kr, Vc=Vr, pos=127 + t))
        assert_bits_equal(host(ys[t][0]), ey, f"y at {127 + t}")
        assert_bits_equal(host(ys[t][1]), eys, f"ysum at {127 + t}")
    assert_bits_equal(host(d["Kc"]).reshape(Kr.shape), Kr, "K cache")
    assert_bits_equal(host(d["Vc"]).reshape(Vr.shape), Vr, "V cache")
    assert abg.device_status(clear=True) == 0


def test_mixers_after_copy_nodes():
    """gdn and atq nodes right after copy nodes (their first launches start
    only after the copies), taking x and q from pinned host memory and handing
    y back there: bit-exact to the oracle over two replays."""
    rng = np.random.default_rng(94)
    cg = synth.gdn_case(rng, 4, 128, 4)
    ca = synth.atq_case(rng, 4, 2, 128, 400, 200)
    g_ = {k: dev(v) for k, v in cg.items()}
    a_ = {k: dev(v) for k, v in ca.items() if k != "pos"}
    Hg, Dg = cg["S"].shape[0], cg["S"].shape[1]
    Dq = ca["Kc"].shape[2]
    Hq = ca["q"].size // Dq
    xh = torch.from_numpy(cg["x"]).pin_memory()
    qh = torch.from_numpy(ca["q"].ravel()).pin_memory()
    yg, ysg, ya, ysa = empty(Hg * Dg), empty(Hg * Dg // 64), empty(Hq * Dq), empty(Hq * Dq // 64)
    ygh = torch.empty(Hg * Dg, dtype=torch.float32).pin_memory()
    yah = torch.empty(Hq * Dq, dtype=torch.float32).pin_memory()
    N = abg.Node
    nodes = [N.copy(0, xh, g_["x"]), N.copy(0, qh, a_["q"]),
             N.gdn(1, g_["x"], g_["conv"], g_["state"], g_["a"], g_["b"], g_["z"], g_["A_log"], g_["dt_bias"],
                   g_["nw"], g_["S"], yg, ysg),
             N.copy(2, yg, ygh),
             N.atq(3, a_["q"], a_["gate"], a_["k"], a_["v"], a_["qn_w"], a_["kn_w"], a_["cos"], a_["sin"], a_["Kc"],
                   a_["Vc"], ya, ysa, pos=ca["pos"]),
             N.copy(4, ya, yah)]
    keep = list(g_.values()) + list(a_.values()) + [xh, qh, yg, ysg, ya, ysa, ygh, yah]
    graph = abg.StageGraph(nodes, keep=keep)
    assert graph.launches == 5
    S_ref, st_ref, Kr, Vr = cg["S"], cg["state"], ca["Kc"], ca["Vc"]
    for t in range(2):
        graph.launch()
        torch.cuda.synchronize()
        ey, eys, S_ref, st_ref = oracle.gdn(**dict(cg, S=S_ref, state=st_ref))
        ay, ays, Kr, Vr = oracle.atq(**dict(ca, Kc=Kr, Vc=Vr))
        assert_bits_equal(ygh.numpy(), ey, f"gdn y, replay {t}")
        assert_bits_equal(host(ysg), eys, f"gdn ysum, replay {t}")
        assert_bits_equal(yah.numpy(), ay, f"atq y, replay {t}")
        assert_bits_equal(host(ysa), ays, f"atq ysum, replay {t}")
        assert_bits_equal(host(a_["Kc"]).reshape(Kr.shape), Kr, f"K cache, replay {t}")
    graph.close()
    assert abg.device_status(clear=True) == 0
