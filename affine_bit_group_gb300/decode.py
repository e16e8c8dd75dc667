"""The synthetic decode token as a stage graph.

One token of a 2B-class decoder reduced to its quantized products and the
two producers between them ("Metal: queued rmsq, swq, gdn and atq kernels and
a 4-row q4mv, so a decode token is one command buffer with one wait",
bendlang/bend #1440, Why and Verification).  Per layer:

    rmsq(h) -> {q, k, v} products -> group sums of q -> o product (reads q)
    -> rmsq -> {gate, up} products -> swq -> down product (the next h)

then a final rmsq and the output head.  Attention and the recurrent mixers
are not part of it (they need trained weights); the o product reads the q
product's output directly, and the k and v outputs are computed but unused.

``fused=False`` records one node per step (the producers as their own
launches).  ``fused=True`` lets each product recompute its producer in every
thread block (abg_node prologues), which gives bit-identical results with
fewer launches.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import PRO_GSUM, PRO_RMSQ, PRO_SWQ, TREE, Node, StageGraph


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _words(w):
    import torch
    return torch.from_numpy(np.ascontiguousarray(w).view(np.int32)).cuda()


@dataclass
class DeviceMatrix:
    w: object
    scale: object
    bias: object
    rows: int
    cols: int

    @classmethod
    def upload(cls, m):
        return cls(_words(m.w), _dev(m.scale), _dev(m.bias), m.rows, m.cols)

    @property
    def nbytes(self) -> int:
        return self.rows * self.cols // 2 + 8 * self.rows * (self.cols // 64)


@dataclass
class DeviceModel:
    layers: list = field(default_factory=list)  # dicts of DeviceMatrix and rms weight tensors
    rms_final: object = None
    head: DeviceMatrix = None
    hidden: int = 0
    mlp: int = 0

    @classmethod
    def upload(cls, model):
        dm = cls(hidden=model.hidden, mlp=model.mlp)
        for L in model.layers:
            dm.layers.append(dict(rms1=_dev(L.rms1), q=DeviceMatrix.upload(L.q), k=DeviceMatrix.upload(L.k),
                                  v=DeviceMatrix.upload(L.v), o=DeviceMatrix.upload(L.o), rms2=_dev(L.rms2),
                                  gate=DeviceMatrix.upload(L.gate), up=DeviceMatrix.upload(L.up),
                                  down=DeviceMatrix.upload(L.down)))
        dm.rms_final = _dev(model.rms_final)
        dm.head = DeviceMatrix.upload(model.head)
        return dm

    def matrices(self):
        out = []
        for L in self.layers:
            out += [L[k] for k in ("q", "k", "v", "o", "gate", "up", "down")]
        return out + [self.head]

    @property
    def product_bytes(self) -> int:
        """Algorithmic bytes of one token's products: weights, scale, bias, x, xsum and y of each."""
        total = 0
        for m in self.matrices():
            total += m.nbytes + 4 * m.cols + 4 * (m.cols // 64) + 4 * m.rows
        return total


def decode_token_graph(dm: DeviceModel, h0, fused: bool = True, mode: int = TREE, rows_per_warp: int = 0,
                       eps: float = 1e-6, host_io=None):
    """(graph, outputs): the token's stage graph reading h0 and the buffers it writes.

    outputs["logits"] is the head's output; the per-layer buffers are kept in
    outputs["layers"] for inspection.  With host_io = (h_host, logits_host),
    pinned host tensors, every replay first copies h_host into h0 and last
    copies the logits into logits_host (copy nodes of the same graph).
    """
    import torch

    def buf(n):
        return torch.empty(n, dtype=torch.float32, device="cuda")

    nodes, keep = [], [h0]
    layers_out = []
    stage = 0
    if host_io is not None:
        nodes.append(Node.copy(0, host_io[0], h0))
        keep += list(host_io)
        stage = 1
    h = h0
    H, M = dm.hidden, dm.mlp
    for L in dm.layers:
        q, k, v = L["q"], L["k"], L["v"]
        o = dict(q=buf(q.rows), k=buf(k.rows), v=buf(v.rows), o=buf(L["o"].rows), gu=buf(2 * M), h=buf(H))
        if fused:
            for name in ("q", "k", "v"):
                m = L[name]
                nodes.append(Node.q4mv(stage, m.w, m.scale, m.bias, o[name], m.cols, x=h, prologue=PRO_RMSQ,
                                       wt=L["rms1"], eps=eps))
            stage += 1
            m = L["o"]
            nodes.append(Node.q4mv(stage, m.w, m.scale, m.bias, o["o"], m.cols, x=o["q"], prologue=PRO_GSUM))
            stage += 1
            for i, name in enumerate(("gate", "up")):
                m = L[name]
                nodes.append(Node.q4mv(stage, m.w, m.scale, m.bias, o["gu"][i * M:(i + 1) * M], m.cols, x=o["o"],
                                       prologue=PRO_RMSQ, wt=L["rms2"], eps=eps))
            stage += 1
            m = L["down"]
            nodes.append(Node.q4mv(stage, m.w, m.scale, m.bias, o["h"], m.cols, x=o["gu"], prologue=PRO_SWQ))
            stage += 1
        else:
            o.update(xn=buf(H), xs=buf(H // 64), qs=buf(q.rows // 64), xn2=buf(H), xs2=buf(H // 64), s=buf(M),
                     ss=buf(M // 64))
            nodes.append(Node.rmsq(stage, h, L["rms1"], o["xn"], o["xs"], eps=eps))
            stage += 1
            for name in ("q", "k", "v"):
                m = L[name]
                nodes.append(Node.q4mv(stage, m.w, m.scale, m.bias, o[name], m.cols, x=o["xn"], xsum=o["xs"]))
            stage += 1
            nodes.append(Node.gsum(stage, o["q"], o["qs"]))
            stage += 1
            m = L["o"]
            nodes.append(Node.q4mv(stage, m.w, m.scale, m.bias, o["o"], m.cols, x=o["q"], xsum=o["qs"]))
            stage += 1
            nodes.append(Node.rmsq(stage, o["o"], L["rms2"], o["xn2"], o["xs2"], eps=eps))
            stage += 1
            for i, name in enumerate(("gate", "up")):
                m = L[name]
                nodes.append(Node.q4mv(stage, m.w, m.scale, m.bias, o["gu"][i * M:(i + 1) * M], m.cols, x=o["xn2"],
                                       xsum=o["xs2"]))
            stage += 1
            nodes.append(Node.swq(stage, o["gu"], o["s"], o["ss"]))
            stage += 1
            m = L["down"]
            nodes.append(Node.q4mv(stage, m.w, m.scale, m.bias, o["h"], m.cols, x=o["s"], xsum=o["ss"]))
            stage += 1
        layers_out.append(o)
        keep += list(o.values()) + [L[k] for k in L]
        h = o["h"]
    logits = buf(dm.head.rows)
    out = dict(logits=logits, layers=layers_out)
    if fused:
        m = dm.head
        nodes.append(Node.q4mv(stage, m.w, m.scale, m.bias, logits, m.cols, x=h, prologue=PRO_RMSQ,
                               wt=dm.rms_final, eps=eps))
    else:
        out.update(xf=buf(H), xfs=buf(H // 64))
        nodes.append(Node.rmsq(stage, h, dm.rms_final, out["xf"], out["xfs"], eps=eps))
        stage += 1
        m = dm.head
        nodes.append(Node.q4mv(stage, m.w, m.scale, m.bias, logits, m.cols, x=out["xf"], xsum=out["xfs"]))
        keep += [out["xf"], out["xfs"]]
    keep += [logits, dm.rms_final, dm.head]
    if host_io is not None:
        nodes.append(Node.copy(stage + 1, logits, host_io[1]))
    return StageGraph(nodes, mode=mode, rows_per_warp=rows_per_warp, keep=keep), out
