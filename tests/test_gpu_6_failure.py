"""Failure detection on the GPU, without faulting it.

A bounded device wait that runs out is reported through the status word and
leaves the context usable (the self-test's producer withholds its data, so the
computing warps' waits expire after the 0.5 s limit); a destroyed graph handle
is refused; a call that synchronizes the device during a stream capture
returns an error status and leaves the context usable.
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


def product_ok():
    m, x = synth.tiny()
    xs = oracle.gsum(x)
    y = empty(m.rows)
    abg.q4mv(dev_words(m.w), dev(m.scale), dev(m.bias), dev(x), dev(xs), y, cols=m.cols)
    torch.cuda.synchronize()
    assert_bits_equal(host(y), oracle.q4mv(*m.arrays(), x, xs, m.cols), "product after the failure")


def test_expired_wait_is_reported_and_context_survives():
    assert abg.device_status(clear=True) == 0
    abg.selftest_wait_timeout()
    torch.cuda.synchronize()
    bits = abg.device_status(clear=True)
    assert bits & 1, bits             # a bounded wait ran out
    assert bits & 32, bits            # the wait for a stage's arrival
    assert abg.device_status(clear=True) == 0
    product_ok()                      # the context is still usable
    assert abg.device_status(clear=True) == 0


def test_destroyed_graph_handle_is_refused():
    m, x = synth.tiny()
    xd, xsd, y = dev(x), dev(oracle.gsum(x)), empty(m.rows)
    w, s, b = dev_words(m.w), dev(m.scale), dev(m.bias)
    g = abg.StageGraph([abg.Node.q4mv(0, w, s, b, y, m.cols, x=xd, xsum=xsd)], keep=[w, s, b, xd, xsd, y])
    h = g._h.value
    g.close()
    lib = abg.library()
    assert lib.abg_stage_graph_launch(h, None) == 1          # ABG_EINVAL: replay after destroy
    assert lib.abg_stage_graph_destroy(h) == 1                # a second destroy
    assert lib.abg_stage_graph_launches(h, None) == 1


def test_device_sync_during_a_capture_returns_a_status():
    """abg_device_status synchronizes the device, which a stream capture forbids:
    called mid-capture it returns ABG_ECUDA with CUDA's message (the capture is
    invalidated, the context is not)."""
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    err = None
    with torch.cuda.stream(st):
        graph.capture_begin()
        try:
            try:
                abg.device_status(clear=False)
            except abg.AbgError as e:
                err = e
        finally:
            try:
                graph.capture_end()
            except Exception:
                pass
    torch.cuda.synchronize()
    assert err is not None and err.status == 5, err  # ABG_ECUDA
    assert "captur" in str(err).lower()
    product_ok()
    assert abg.device_status(clear=True) == 0
