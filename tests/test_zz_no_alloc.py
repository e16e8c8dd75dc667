"""The allocation-free MLP call, abg_swiglu_mlp_static, on the GPU.

It serves callers that cannot allocate device memory themselves (their device
memory belongs to another allocator, or cudaMalloc/cudaFree would synchronize
the device on a latency path): the gate/up/SwiGLU/down block keeps its
intermediate vectors in a static array inside the library.  Its output must
equal, bit for bit in tree mode, what the allocating calls give (abg_q4mv for
gate and up, abg_swq, abg_q4mv for down), on two calls in a row, since every
call shares that array.  This file is collected last so that a run stopping at
the first failure has run every other test first; it passes alone as well.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import oracle
from affine_bit_group_gb300 import synth
from helpers import assert_bits_equal, dev, dev_words, empty, host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
abg = pytest.importorskip("affine_bit_group_gb300")


def allocating_reference(G, U, D, x, xs, n, cols, rows):
    """y through the existing entry points, with buffers allocated here."""
    a = empty(2 * n)
    abg.q4mv(*G, x, xs, a[:n], cols=cols)
    abg.q4mv(*U, x, xs, a[n:], cols=cols)
    o, osum = empty(n), empty(n // 64)
    abg.swq(a, o, osum)
    y = empty(rows)
    abg.q4mv(*D, o, osum, y, cols=n)
    torch.cuda.synchronize()
    return host(y)


def static_call(G, U, D, x, xs, y, n, cols, rows):
    """y through abg_swiglu_mlp_static, called through the C ABI."""
    lib = abg.library()
    ptrs = [t.data_ptr() for t in (*G, *U, *D, x, xs, y)]
    st = lib.abg_swiglu_mlp_static(*ptrs, n, cols, rows, abg.TREE, torch.cuda.current_stream().cuda_stream)
    assert st == 0, abg.AbgError(st, "abg_swiglu_mlp_static")


@pytest.mark.parametrize("n,cols,rows", [(1024, 2048, 700), (6144, 2048, 2048), (2048, 4096, 333), (16384, 2048, 64),
                                         (1088, 1024, 130)])
def test_static_mlp_equals_the_allocating_calls(n, cols, rows):
    mg, _ = synth.random_case(9100 + n, n, cols)
    mu, _ = synth.random_case(9200 + n, n, cols)
    md, _ = synth.random_case(9300 + n, rows, n)
    G, U, D = [(dev_words(m.w), dev(m.scale), dev(m.bias)) for m in (mg, mu, md)]
    for call in range(2):  # two calls in a row share the static scratch
        x_np = synth.activations(np.random.default_rng([9400, n, call]), cols)
        x, xs = dev(x_np), dev(oracle.gsum(x_np))
        y = empty(rows)
        static_call(G, U, D, x, xs, y, n, cols, rows)
        torch.cuda.synchronize()
        got = host(y)
        assert_bits_equal(got, allocating_reference(G, U, D, x, xs, n, cols, rows), f"{n}x{cols}->{rows} call {call}")
    assert abg.device_status(clear=True) == 0


def test_static_mlp_rejects_more_than_its_scratch():
    m, _ = synth.random_case(9500, 64, 2048)
    t = (dev_words(m.w), dev(m.scale), dev(m.bias))
    x = dev(synth.activations(np.random.default_rng(9501), 2048))
    xs = empty(32)
    y = empty(64)
    lib = abg.library()
    st = lib.abg_swiglu_mlp_static(*[p.data_ptr() for p in (*t, *t, *t, x, xs, y)], 16384 + 64, 2048, 64,
                                   abg.TREE, None)
    assert st == 3  # ABG_ESHAPE
