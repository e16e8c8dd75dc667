"""Shared helpers for the GPU parity tests: upload, bit comparison, tolerances."""
from __future__ import annotations

import numpy as np


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_words(w):
    import torch
    return torch.from_numpy(np.ascontiguousarray(w).view(np.int32)).cuda()


def empty(n):
    import torch
    return torch.empty(n, dtype=torch.float32, device="cuda")


def host(t):
    return t.detach().cpu().numpy()


def assert_bits_equal(got, exp, what=""):
    """Bit-for-bit equality of float32 arrays; any NaN matches any NaN."""
    got = np.ascontiguousarray(got, np.float32)
    exp = np.ascontiguousarray(exp, np.float32)
    assert got.shape == exp.shape, (got.shape, exp.shape)
    gn, en = np.isnan(got), np.isnan(exp)
    assert np.array_equal(gn, en), f"{what}: NaN positions differ"
    g, e = got.view(np.uint32)[~gn], exp.view(np.uint32)[~en]
    bad = np.nonzero(g != e)[0]
    assert bad.size == 0, (f"{what}: {bad.size} of {g.size} differ; first at {bad[0]}: "
                           f"got {got[~gn][bad[0]]!r} expected {exp[~en][bad[0]]!r}")


def assert_fast_close(got, tree, mag, rel=1e-5, what=""):
    """Fast mode bound: |y_fast - y_tree| <= rel * max(|y_tree|, A_r) per output."""
    got = np.asarray(got, np.float64)
    tree = np.asarray(tree, np.float64)
    bound = rel * np.maximum(np.abs(tree), np.asarray(mag, np.float64))
    err = np.abs(got - tree)
    worst = np.argmax(err - bound)
    assert np.all(err <= bound), f"{what}: |diff| {err[worst]:.3e} > bound {bound[worst]:.3e} at {worst}"
