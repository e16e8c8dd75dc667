"""The decode-token stage graph on the GPU against the oracle's decode token.

Tree mode: the head's output (and every intermediate) is bit-for-bit the
oracle's, for the unfused graph (one launch per step) and the fused one
(producers recomputed inside the products).  Replays are deterministic and
two graphs replayed in turn match their solo runs.
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
from affine_bit_group_gb300 import decode  # noqa: E402

SMALL = dict(seed=7, n_layers=3, hidden=1024, mlp=3072, head_rows=5000, q_rows=2048, kv_rows=256)


@pytest.fixture(scope="module")
def small():
    model, h = synth.decode_model(**SMALL)
    logits, trace, (xf, xfs) = oracle.decode_token(model, h, keep=True)
    return model, h, logits, trace, decode.DeviceModel.upload(model)


@pytest.mark.parametrize("fused", [False, True])
def test_small_decode_token_bit_exact(small, fused):
    model, h, logits, trace, dm = small
    h0 = dev(h)
    g, out = decode.decode_token_graph(dm, h0, fused=fused)
    g.launch()
    torch.cuda.synchronize()
    for i, (o, t) in enumerate(zip(out["layers"], trace)):
        for key in ("q", "k", "v", "o", "h"):
            assert_bits_equal(host(o[key]), t[key], f"layer {i} {key}")
        assert_bits_equal(host(o["gu"]), np.concatenate([t["gate"], t["up"]]), f"layer {i} gate|up")
        if not fused:
            assert_bits_equal(host(o["xn"]), t["xn"], f"layer {i} xn")
            assert_bits_equal(host(o["qs"]), t["qs"], f"layer {i} qs")
            assert_bits_equal(host(o["s"]), t["s"], f"layer {i} s")
    assert_bits_equal(host(out["logits"]), logits, "logits")
    expected_launches = (4 if fused else 8) * SMALL["n_layers"] + (1 if fused else 2)
    assert g.launches == expected_launches
    g.close()


def test_replay_and_interleaving(small):
    model, h, logits, trace, dm = small
    h0 = dev(h)
    g1, out1 = decode.decode_token_graph(dm, h0, fused=True)
    h2 = synth.activations(np.random.default_rng(99), SMALL["hidden"])
    h0b = dev(h2)
    g2, out2 = decode.decode_token_graph(dm, h0b, fused=False)
    exp2 = oracle.decode_token(model, h2)
    for _ in range(3):
        g1.launch()
        g2.launch()
    torch.cuda.synchronize()
    assert_bits_equal(host(out1["logits"]), logits, "graph 1 after interleaving")
    assert_bits_equal(host(out2["logits"]), exp2, "graph 2 after interleaving")
    # replacing the input between replays changes only what it should
    h0.copy_(h0b)
    g1.launch()
    torch.cuda.synchronize()
    assert_bits_equal(host(out1["logits"]), exp2, "graph 1 with the second input")
    g1.close()
    g2.close()


def test_fast_graph_equals_fast_calls(small):
    """Fast mode is deterministic: the graph gives the same bits as the same kernels called one by one."""
    model, h, logits, trace, dm = small
    h0 = dev(h)
    g, out = decode.decode_token_graph(dm, h0, fused=False, mode=abg.FAST)
    g.launch()
    torch.cuda.synchronize()
    L = dm.layers[0]
    xn, xs = empty(dm.hidden), empty(dm.hidden // 64)
    abg.rmsq(h0, L["rms1"], xn, xs, mode=abg.FAST)
    q = empty(L["q"].rows)
    abg.q4mv(L["q"].w, L["q"].scale, L["q"].bias, xn, xs, q, cols=L["q"].cols, mode=abg.FAST)
    torch.cuda.synchronize()
    assert_bits_equal(host(q), host(out["layers"][0]["q"]), "fast q")
    # and stays close to the tree result: errors of 1e-6 relative per step, renormalized every layer
    rel = np.max(np.abs(host(out["logits"]) - logits)) / np.max(np.abs(logits))
    assert rel < 1e-3, rel
    g.close()


def test_graph_rejects_same_stage_hazards(small):
    model, h, logits, trace, dm = small
    L = dm.layers[0]
    x, xs = empty(dm.hidden), empty(dm.hidden // 64)
    y = empty(L["q"].rows)
    q = L["q"]
    # a product and the producer of its input in the same stage
    nodes = [abg.Node.rmsq(0, dev(h), L["rms1"], x, xs), abg.Node.q4mv(0, q.w, q.scale, q.bias, y, q.cols, x=x, xsum=xs)]
    with pytest.raises(abg.AbgError) as e:
        abg.StageGraph(nodes)
    assert e.value.status == 4
    # a node that writes a product's weights
    wview = q.scale.view(-1)[: dm.hidden // 64]
    nodes = [abg.Node.gsum(0, x, wview), abg.Node.q4mv(1, q.w, q.scale, q.bias, y, q.cols, x=x, xsum=xs)]
    with pytest.raises(abg.AbgError) as e:
        abg.StageGraph(nodes)
    assert e.value.status == 4
    # a node that writes the norm weights of a later product's RMS-norm prologue
    # (they are read before the wait for the previous stage)
    wt = empty(dm.hidden)
    wt.copy_(L["rms1"])
    nodes = [abg.Node.gsum(0, x, wt[: dm.hidden // 64]),
             abg.Node.q4mv(1, q.w, q.scale, q.bias, y, q.cols, x=dev(h), prologue=abg.PRO_RMSQ, wt=wt)]
    with pytest.raises(abg.AbgError) as e:
        abg.StageGraph(nodes)
    assert e.value.status == 4


@pytest.mark.parametrize("cols", [128, 1088, 2048, 6144, 16384])
@pytest.mark.parametrize("rows", [40, 700, 9000])
def test_rmsq_prologue_shapes(rows, cols):
    """The RMS-norm prologue inside a product, over column counts with a ragged
    last chunk (1088), up to 8 chunks (one pass over x, warps keeping one chunk)
    and 16 chunks (two passes, warps walking chunks), and launches of few and of
    many tiles: bit-exact in tree mode (the norm's tree and rounding are the
    oracle's), within the bound in fast mode."""
    rng = np.random.default_rng([rows, cols])
    m = synth.q4_matrix(rng, rows, cols)
    h = synth.activations(rng, cols)
    wt = synth.rms_weights(rng, cols)
    hd, wtd = dev(h), dev(wt)
    w, sc, bi = dev_words(m.w), dev(m.scale), dev(m.bias)
    xn, xs = oracle.rmsq(h, wt, 1e-6)
    tree = oracle.q4mv(*m.arrays(), xn, xs, cols)
    for mode in (abg.TREE, abg.FAST):
        y = empty(rows)
        g = abg.StageGraph([abg.Node.q4mv(0, w, sc, bi, y, cols, x=hd, wt=wtd, eps=1e-6, prologue=abg.PRO_RMSQ)],
                           keep=[hd, wtd, w, sc, bi, y], mode=mode)
        g.launch()
        torch.cuda.synchronize()
        if mode == abg.TREE:
            assert_bits_equal(host(y), tree, f"rmsq prologue {rows}x{cols}")
        else:
            assert_fast_close(host(y), tree, oracle.q4mv_absmag(*m.arrays(), xn, xs, cols),
                              what=f"fast rmsq prologue {rows}x{cols}")
        g.close()
    assert abg.device_status(clear=True) == 0


@pytest.mark.slow
def test_full_decode_token_bit_exact():
    """24 layers, hidden 2048, MLP 6144, the 248320-row head: fused graph == oracle, bit for bit."""
    model, h = synth.decode_model()
    exp = oracle.decode_token(model, h)
    dm = decode.DeviceModel.upload(model)
    h0 = dev(h)
    g, out = decode.decode_token_graph(dm, h0, fused=True)
    assert g.swiglu_pairs == len(dm.layers)  # every layer's gate/up launch writes the SwiGLU vector
    g.launch()
    torch.cuda.synchronize()
    assert_bits_equal(host(out["logits"]), exp, "full decode logits")
    g2, out2 = decode.decode_token_graph(dm, h0, fused=False)
    g2.launch()
    torch.cuda.synchronize()
    assert_bits_equal(host(out2["logits"]), exp, "full decode logits, unfused")
    assert abg.device_status(clear=True) == 0
    g.close()
    g2.close()


@pytest.mark.parametrize("cols", [2048, 4096, 6144])
@pytest.mark.parametrize("adjacent", [True, False])
def test_swiglu_pair(cols, adjacent):
    """gate/up products into a = [gate | up], then a product with the SwiGLU
    prologue on a: with the reader in the next stage the gate/up launch writes
    the SwiGLU vector (one pair formed), otherwise not; either way every output
    equals the oracle's (gate, up, the SwiGLU of them, the product)."""
    n = 1088  # rows of gate and up, the reader's columns (not a whole tile count)
    mg, x = synth.random_case(8100 + cols, n, cols)
    mu, _ = synth.random_case(8200 + cols, n, cols)
    md, _ = synth.random_case(8300 + cols, 700, n)
    xd, xsd = dev(x), dev(oracle.gsum(x))
    a = empty(2 * n)
    yd = empty(700)
    G, U, D = [(dev_words(m.w), dev(m.scale), dev(m.bias)) for m in (mg, mu, md)]
    nodes = [abg.Node.q4mv(0, *G, a[:n], cols, x=xd, xsum=xsd), abg.Node.q4mv(0, *U, a[n:], cols, x=xd, xsum=xsd)]
    if not adjacent:
        spare = empty(64)
        nodes.append(abg.Node.gsum(1, xd[:64], spare[:1]))
    nodes.append(abg.Node.q4mv(1 if adjacent else 2, *D, yd, n, x=a, prologue=abg.PRO_SWQ))
    g = abg.StageGraph(nodes, keep=[xd, xsd, a, yd] + list(G) + list(U) + list(D))
    assert g.swiglu_pairs == (1 if adjacent else 0)
    g.launch()
    torch.cuda.synchronize()
    xs = oracle.gsum(x)
    gy = oracle.q4mv(*mg.arrays(), x, xs, cols)
    uy = oracle.q4mv(*mu.arrays(), x, xs, cols)
    assert_bits_equal(host(a)[:n], gy, "gate")
    assert_bits_equal(host(a)[n:], uy, "up")
    o, osum = oracle.swq(np.concatenate([gy, uy]))
    assert_bits_equal(host(yd), oracle.q4mv(*md.arrays(), o, osum, n), "reader of the SwiGLU")
    assert abg.device_status(clear=True) == 0
    g.close()


@pytest.mark.parametrize("cols,rows", [(2048, (4096, 512, 500)), (4096, (2048, 401, 299)), (3072, (1500, 300, 37))])
def test_grouped_products_with_quarter_tiles(cols, rows):
    """Three products of one stage sharing the RMS-norm prologue (one grouped
    launch), sized so that the whole tiles exceed the SMs by a little: the last
    products run as quarter tiles (ragged ends included).  Every output is the
    oracle's, bit for bit."""
    rng = np.random.default_rng([cols, *rows])
    ms = [synth.q4_matrix(rng, n, cols) for n in rows]
    h = synth.activations(rng, cols)
    wt = synth.rms_weights(rng, cols)
    hd, wtd = dev(h), dev(wt)
    mats = [(dev_words(m.w), dev(m.scale), dev(m.bias)) for m in ms]
    ys = [empty(n) for n in rows]
    nodes = [abg.Node.q4mv(0, *mat, y, cols, x=hd, wt=wtd, eps=1e-6, prologue=abg.PRO_RMSQ)
             for mat, y in zip(mats, ys)]
    g = abg.StageGraph(nodes, keep=[hd, wtd, *ys, *[t for mat in mats for t in mat]])
    assert g.launches == 1
    for _ in range(2):
        g.launch()
    torch.cuda.synchronize()
    xn, xs = oracle.rmsq(h, wt, 1e-6)
    for m, y, n in zip(ms, ys, rows):
        assert_bits_equal(host(y), oracle.q4mv(*m.arrays(), xn, xs, cols), f"{n}x{cols}")
    assert abg.device_status(clear=True) == 0
    g.close()


@pytest.mark.parametrize("prologue", ["rmsq", "swq", "gsum", "special"])
def test_prologues_many_tiles_6144(prologue):
    """Rows of 6144 columns in a launch of many tiles run 18 computing warps per
    block, whose cooperative prologue has a partial last round of units (1536
    units over 576 threads): each prologue, and an activation with special
    values and all-negative groups (the plain path in some warps), bit-exact
    in tree mode and within the bound in fast mode."""
    rows, cols = 20000, 6144
    rng = np.random.default_rng([rows, cols, len(prologue)])
    m = synth.q4_matrix(rng, rows, cols)
    w, sc, bi = dev_words(m.w), dev(m.scale), dev(m.bias)
    if prologue == "swq":
        a = np.concatenate([synth.activations(rng, cols), synth.activations(rng, cols)])
        x, xs = oracle.swq(a)
        xin, kw = dev(a), dict(prologue=abg.PRO_SWQ)
    elif prologue == "rmsq":
        h = synth.activations(rng, cols)
        wt = synth.rms_weights(rng, cols)
        x, xs = oracle.rmsq(h, wt, 1e-6)
        wtd = dev(wt)
        xin, kw = dev(h), dict(prologue=abg.PRO_RMSQ, wt=wtd, eps=1e-6)
    else:
        x = synth.activations(rng, cols)
        if prologue == "special":
            x[64:128] = -np.abs(x[64:128])
            x[5000] = np.inf
            x[5001] = -0.0
        xs = oracle.gsum(x)
        xin, kw = dev(x), dict(prologue=abg.PRO_GSUM)
    tree = oracle.q4mv(*m.arrays(), x, xs, cols)
    keep = [xin, w, sc, bi] + [v for v in kw.values() if hasattr(v, "data_ptr")]
    for mode in (abg.TREE, abg.FAST):
        y = empty(rows)
        g = abg.StageGraph([abg.Node.q4mv(0, w, sc, bi, y, cols, x=xin, **kw)], keep=keep + [y], mode=mode)
        g.launch()
        torch.cuda.synchronize()
        if mode == abg.TREE:
            assert_bits_equal(host(y), tree, f"{prologue} {rows}x{cols}")
        elif prologue != "special":
            assert_fast_close(host(y), tree, oracle.q4mv_absmag(*m.arrays(), x, xs, cols),
                              what=f"fast {prologue} {rows}x{cols}")
        g.close()
    assert abg.device_status(clear=True) == 0


@pytest.mark.parametrize("count,launches", [(256, 1), (257, 2), (300, 2)])
def test_many_products_of_one_stage(count, launches):
    """Products of one stage reading one x, of seven row counts: grouped
    launches of at most 256 products, each launch walking its problems tile
    by tile.  Every output bit-exact to the oracle."""
    rng = np.random.default_rng(77)
    cols = 512
    mats = [synth.q4_matrix(rng, 40 + 8 * (i % 7), cols) for i in range(count)]
    x = synth.activations(rng, cols)
    xs = oracle.gsum(x)
    dx, dxs = dev(x), dev(xs)
    dm = [(dev_words(m.w), dev(m.scale), dev(m.bias)) for m in mats]
    ys = [empty(m.rows) for m in mats]
    nodes = [abg.Node.q4mv(0, *dm[i], ys[i], cols, x=dx, xsum=dxs) for i in range(len(mats))]
    g = abg.StageGraph(nodes, keep=[dx, dxs] + ys + [t for d in dm for t in d])
    assert g.launches == launches
    for _ in range(2):
        g.launch()
    torch.cuda.synchronize()
    for i, m in enumerate(mats):
        assert_bits_equal(host(ys[i]), oracle.q4mv(m.w, m.scale, m.bias, x, xs, cols), f"product {i}")
    g.close()
    assert abg.device_status(clear=True) == 0


@pytest.mark.parametrize("count", [16, 17, 40, 256])
def test_few_tiles_table_capacity(count):
    """A stage of small products of 2048 columns reading one x (with the
    RMS-norm prologue): one grouped launch of few tiles.  Up to 16 products
    it runs the few-tiles instantiation, whose product table holds 16; more
    products run the 8-row instantiation with the full table.  Every output
    bit-exact to the oracle, in both cases."""
    rng = np.random.default_rng(500 + count)
    cols = 2048
    mats = [synth.q4_matrix(rng, 32 + 16 * (i % 3), cols) for i in range(count)]
    h = synth.activations(rng, cols)
    wt = synth.rms_weights(rng, cols)
    xn, xs = oracle.rmsq(h, wt, 1e-6)
    dh, dwt = dev(h), dev(wt)
    dm = [(dev_words(m.w), dev(m.scale), dev(m.bias)) for m in mats]
    ys = [empty(m.rows) for m in mats]
    nodes = [abg.Node.q4mv(0, *dm[i], ys[i], cols, x=dh, wt=dwt, eps=1e-6, prologue=abg.PRO_RMSQ)
             for i in range(count)]
    g = abg.StageGraph(nodes, keep=[dh, dwt] + ys + [t for d in dm for t in d])
    assert g.launches == 1
    for _ in range(2):
        g.launch()
    torch.cuda.synchronize()
    for i, m in enumerate(mats):
        assert_bits_equal(host(ys[i]), oracle.q4mv(m.w, m.scale, m.bias, xn, xs, cols), f"product {i}")
    g.close()
    assert abg.device_status(clear=True) == 0


def test_copy_nodes_host_in_host_out():
    """A replay that starts and ends in pinned host memory: copy x in, its
    group sums, three products of one stage (one grouped launch), copy the
    outputs out.  The launch count counts kernels only; every replay reads the
    host x as it is then (a new x gives the new results, bit-exact to the
    oracle)."""
    rng = np.random.default_rng(91)
    cols = 2048
    mats = [synth.q4_matrix(rng, r, cols) for r in (4096, 512, 512)]
    dm = [(dev_words(m.w), dev(m.scale), dev(m.bias)) for m in mats]
    xh = torch.empty(cols, dtype=torch.float32).pin_memory()
    yh = [torch.empty(m.rows, dtype=torch.float32).pin_memory() for m in mats]
    xd, xsd = empty(cols), empty(cols // 64)
    yd = [empty(m.rows) for m in mats]
    N = abg.Node
    nodes = ([N.copy(0, xh, xd), N.gsum(1, xd, xsd)] +
             [N.q4mv(2, *dm[i], yd[i], cols, x=xd, xsum=xsd) for i in range(3)] +
             [N.copy(3, yd[i], yh[i]) for i in range(3)])
    g = abg.StageGraph(nodes, keep=[xh, xd, xsd] + yh + yd + [t for d in dm for t in d])
    assert g.launches == 2
    for rep in range(3):
        x = synth.activations(rng, cols)
        xh.copy_(torch.from_numpy(x))
        g.launch()
        torch.cuda.synchronize()
        xs = oracle.gsum(x)
        for i, m in enumerate(mats):
            assert_bits_equal(yh[i].numpy(), oracle.q4mv(m.w, m.scale, m.bias, x, xs, cols), f"product {i}, {rep}")
    g.close()
    assert abg.device_status(clear=True) == 0


def test_copy_node_between_kernels():
    """A device-to-device copy between two dependent kernels (the RMS norm's
    output copied, then read by a product): the product starts only after
    the copy; bit-exact."""
    rng = np.random.default_rng(92)
    cols = 2048
    m = synth.q4_matrix(rng, 1000, cols)
    h = synth.activations(rng, cols)
    wt = synth.rms_weights(rng, cols)
    xn_ref, xs_ref = oracle.rmsq(h, wt, 1e-6)
    hd, wtd = dev(h), dev(wt)
    xn, xs, xn2, xs2 = empty(cols), empty(cols // 64), empty(cols), empty(cols // 64)
    y = empty(m.rows)
    w, sc, bi = dev_words(m.w), dev(m.scale), dev(m.bias)
    N = abg.Node
    nodes = [N.rmsq(0, hd, wtd, xn, xs), N.copy(1, xn, xn2), N.copy(1, xs, xs2),
             N.q4mv(2, w, sc, bi, y, cols, x=xn2, xsum=xs2)]
    g = abg.StageGraph(nodes, keep=[hd, wtd, xn, xs, xn2, xs2, y, w, sc, bi])
    assert g.launches == 2
    for _ in range(2):
        y.fill_(float("nan"))
        g.launch()
        torch.cuda.synchronize()
        assert_bits_equal(host(y), oracle.q4mv(m.w, m.scale, m.bias, xn_ref, xs_ref, cols), "product after copies")
    g.close()
    assert abg.device_status(clear=True) == 0


def test_copy_node_refusals():
    """Copy nodes in the stage hazard checks, and pageable host memory."""
    rng = np.random.default_rng(93)
    cols = 2048
    m = synth.q4_matrix(rng, 256, cols)
    w, sc, bi = dev_words(m.w), dev(m.scale), dev(m.bias)
    xh = torch.empty(cols, dtype=torch.float32).pin_memory()
    xd, xsd, y = empty(cols), empty(cols // 64), empty(m.rows)
    N = abg.Node
    # a product of the copy's own stage reading what it writes
    with pytest.raises(abg.AbgError) as e:
        abg.StageGraph([N.copy(0, xh, xd), N.q4mv(0, w, sc, bi, y, cols, x=xd, xsum=xsd)])
    assert e.value.status == 4
    # a copy over a product's weights
    sview = sc.view(-1)[: cols]
    with pytest.raises(abg.AbgError) as e:
        abg.StageGraph([N.copy(0, xh, sview), N.q4mv(1, w, sc, bi, y, cols, x=xd, xsum=xsd)])
    assert e.value.status == 4
    # pageable host memory: refused by the binding, and by the library
    pageable = torch.empty(cols, dtype=torch.float32)
    with pytest.raises(ValueError):
        N.copy(0, pageable, xd)
    raw = abg._Node(kind=abg.NODE_COPY, stage=0, x=pageable.data_ptr(), out=xd.data_ptr(), len=cols)
    with pytest.raises(abg.AbgError) as e:
        abg.StageGraph([raw])
    assert e.value.status == 1
    assert abg.device_status(clear=True) == 0


def test_decode_token_host_io(small):
    """The fused token reading its hidden vector from pinned host memory and
    writing its logits there (copy nodes of the same graph): the host logits
    bit-exact to the oracle, then again after a new hidden vector."""
    model, h, logits, _, dm = small
    h_host = torch.from_numpy(h).pin_memory()
    lh = torch.empty(logits.size, dtype=torch.float32).pin_memory()
    h_dev = empty(h.size)
    g, _ = decode.decode_token_graph(dm, h_dev, fused=True, host_io=(h_host, lh))
    g.launch()
    torch.cuda.synchronize()
    assert_bits_equal(lh.numpy(), logits, "logits")
    h2 = synth.activations(np.random.default_rng(5), h.size)
    h_host.copy_(torch.from_numpy(h2))
    g.launch()
    torch.cuda.synchronize()
    assert_bits_equal(lh.numpy(), oracle.decode_token(model, h2), "logits, new hidden vector")
    g.close()
    assert abg.device_status(clear=True) == 0
