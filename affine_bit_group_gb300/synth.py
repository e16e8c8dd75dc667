"""Seeded synthetic inputs for q4mv / rmsq / swq and the decode-token graph.

This module holds random draws and array shapes only -- none of the product's
arithmetic -- so the CPU oracle and the CUDA library can both be fed from it
without sharing any computation.

Recipe (numpy ``default_rng(seed)``, draws in this order per matrix):

* packed weights: ``integers(0, 2**32, (rows, cols/8), uint32)``.  Each u32 is
  eight independent uniform nibbles 0..15; column 8k+j of a row is nibble j
  of word k, low nibble first (the library's packing).
* scale: ``uniform(0.002, 0.02, (rows, cols/64))`` rounded to f32.
* bias: ``f32(-8 * scale + normal(0, 0.001, (rows, cols/64)))`` -- the affine
  zero point of MLX-style 4-bit weights (the dequantised weight scale*q+bias is
  centred near zero), with the f32 scale widened to f64 before the product.
* activations: ``normal(0, 1, cols)`` rounded to f32.
* RMS-norm weights: ``uniform(0.5, 1.5, n)`` rounded to f32.

Workloads (the pages' shapes: a 4096x2048 product, the 248320x2048 output
head of a 2B-class model, and one decode token's products):

* ``tiny``  seed 0: 13x128 matrix, then x.
* ``mid``   seed 1: 4096x2048 matrix, then x.
* ``head``  seed 2: 248320x2048 matrix, then a N(0,1) hidden vector of 2048,
  then the RMS-norm weights; the product's x is the RMS norm of the hidden.
* ``decode`` seed 3: per layer [rms1 weights, q 4096x2048, k 512x2048,
  v 512x2048, o 2048x4096, rms2 weights, gate 6144x2048, up 6144x2048,
  down 2048x6144], then the final RMS-norm weights, the 248320x2048 head and
  the N(0,1) hidden vector.
* ``sweep`` point (rows, cols): ``default_rng([4, rows, cols])``, matrix then x.

Other formats (group size 32, 64 or 128 columns; scale and bias stored as f32,
bf16 or f16): the same draws with cols/group groups, then the f32 scale and
bias are stored in the 16-bit type -- bf16 as the upper half of the f32 bits
(truncation), f16 by numpy's ``astype(float16)`` -- and passed as uint16 bit
patterns.  ``fmt_case(group, sb, rows, cols)`` uses ``default_rng([5, group,
code(sb), rows, cols])``, matrix then x.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

HIDDEN = 2048
MLP = 6144
HEAD_ROWS = 248320
N_LAYERS = 24
EPS = 1e-6


GROUPS = (32, 64, 128)
SB_TYPES = ("f32", "bf16", "f16")


@dataclass
class Q4Matrix:
    """A packed 4-bit affine matrix: words u32[rows, cols/8], scale/bias [rows, cols/group]
    (f32 values, or uint16 bit patterns of bf16 / f16 values)."""

    w: np.ndarray
    scale: np.ndarray
    bias: np.ndarray
    rows: int
    cols: int
    group: int = 64
    sb: str = "f32"

    def arrays(self):
        return self.w, self.scale, self.bias

    @property
    def nbytes(self) -> int:
        return self.w.nbytes + self.scale.nbytes + self.bias.nbytes


def q4_matrix(rng: np.random.Generator, rows: int, cols: int, group: int = 64, sb: str = "f32") -> Q4Matrix:
    if cols % 64 or group not in GROUPS or cols % group or sb not in SB_TYPES:
        raise ValueError("cols a multiple of 64 and of group; group 32, 64 or 128; sb f32, bf16 or f16")
    G, W = cols // group, cols // 8
    w = rng.integers(0, 2**32, size=(rows, W), dtype=np.uint32)
    scale = rng.uniform(0.002, 0.02, size=(rows, G)).astype(np.float32)
    noise = rng.normal(0.0, 0.001, size=(rows, G))
    bias = (-8.0 * scale.astype(np.float64) + noise).astype(np.float32)
    if sb != "f32":
        scale, bias = store16(scale, sb), store16(bias, sb)
    return Q4Matrix(w, scale, bias, rows, cols, group, sb)


def store16(v: np.ndarray, sb: str) -> np.ndarray:
    """f32 values as bf16 (upper half of the bits) or f16 (numpy rounding) bit patterns."""
    v = np.ascontiguousarray(v, np.float32)
    if sb == "bf16":
        return (v.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    return v.astype(np.float16).view(np.uint16)


def fmt_case(group: int, sb: str, rows: int, cols: int):
    """(matrix, x) in the given format; see the module docstring."""
    rng = np.random.default_rng([5, group, SB_TYPES.index(sb), rows, cols])
    m = q4_matrix(rng, rows, cols, group, sb)
    return m, activations(rng, cols)


def activations(rng: np.random.Generator, n: int) -> np.ndarray:
    return rng.normal(0.0, 1.0, size=n).astype(np.float32)


def rms_weights(rng: np.random.Generator, n: int) -> np.ndarray:
    return rng.uniform(0.5, 1.5, size=n).astype(np.float32)


def tiny():
    rng = np.random.default_rng(0)
    m = q4_matrix(rng, 13, 128)
    return m, activations(rng, 128)


def mid():
    rng = np.random.default_rng(1)
    m = q4_matrix(rng, 4096, 2048)
    return m, activations(rng, 2048)


def head():
    """(matrix, hidden, rms weights); the product's x is rmsq(hidden, weights)."""
    rng = np.random.default_rng(2)
    m = q4_matrix(rng, HEAD_ROWS, HIDDEN)
    hidden = activations(rng, HIDDEN)
    wt = rms_weights(rng, HIDDEN)
    return m, hidden, wt


def sweep_point(rows: int, cols: int):
    rng = np.random.default_rng([4, rows, cols])
    m = q4_matrix(rng, rows, cols)
    return m, activations(rng, cols)


def random_case(seed: int, rows: int, cols: int):
    """Any other shape, same generators (parity and edge-case tests)."""
    rng = np.random.default_rng(seed)
    m = q4_matrix(rng, rows, cols)
    return m, activations(rng, cols)


@dataclass
class Layer:
    rms1: np.ndarray
    q: Q4Matrix
    k: Q4Matrix
    v: Q4Matrix
    o: Q4Matrix
    rms2: np.ndarray
    gate: Q4Matrix
    up: Q4Matrix
    down: Q4Matrix

    def matrices(self):
        return [self.q, self.k, self.v, self.o, self.gate, self.up, self.down]


@dataclass
class DecodeModel:
    layers: list = field(default_factory=list)
    rms_final: np.ndarray = None
    head: Q4Matrix = None
    hidden: int = HIDDEN
    mlp: int = MLP

    def matrices(self):
        out = []
        for L in self.layers:
            out += L.matrices()
        return out + [self.head]

    @property
    def q4_bytes(self) -> int:
        return sum(m.nbytes for m in self.matrices())


def decode_model(seed: int = 3, n_layers: int = N_LAYERS, hidden: int = HIDDEN, mlp: int = MLP,
                 head_rows: int = HEAD_ROWS, q_rows: int = 4096, kv_rows: int = 512):
    """(model, hidden vector) for the synthetic decode token; see the module docstring."""
    rng = np.random.default_rng(seed)
    model = DecodeModel(hidden=hidden, mlp=mlp)
    for _ in range(n_layers):
        rms1 = rms_weights(rng, hidden)
        q = q4_matrix(rng, q_rows, hidden)
        k = q4_matrix(rng, kv_rows, hidden)
        v = q4_matrix(rng, kv_rows, hidden)
        o = q4_matrix(rng, hidden, q_rows)
        rms2 = rms_weights(rng, hidden)
        gate = q4_matrix(rng, mlp, hidden)
        up = q4_matrix(rng, mlp, hidden)
        down = q4_matrix(rng, hidden, mlp)
        model.layers.append(Layer(rms1, q, k, v, o, rms2, gate, up, down))
    model.rms_final = rms_weights(rng, hidden)
    model.head = q4_matrix(rng, head_rows, hidden)
    h = activations(rng, hidden)
    return model, h


# The gated DeltaNet mixer's synthetic token: 16 value heads of 128 columns
# and 4 conv taps (a 2B-class decoder's linear-attention layer; the pages
# give no dimensions).
GDN_HEADS = 16
GDN_DIM = 128
GDN_TAPS = 4


def gdn_case(rng: np.random.Generator, H: int = GDN_HEADS, D: int = GDN_DIM, K: int = GDN_TAPS) -> dict:
    """Inputs of one gdn token (names as abg_gdn): x, conv, state ~ N(0,1)
    scaled 1, 0.5, 1; a, b, z ~ N(0,1); A_log, dt_bias ~ N(0, 0.5);
    nw ~ 1 + N(0, 0.1); S ~ N(0, 0.1), all float32."""
    C = 3 * H * D
    return dict(x=rng.standard_normal(C).astype(np.float32),
                conv=(0.5 * rng.standard_normal((C, K))).astype(np.float32),
                state=rng.standard_normal((C, K - 1)).astype(np.float32),
                a=rng.standard_normal(H).astype(np.float32),
                b=rng.standard_normal(H).astype(np.float32),
                z=rng.standard_normal(H * D).astype(np.float32),
                A_log=(0.5 * rng.standard_normal(H)).astype(np.float32),
                dt_bias=(0.5 * rng.standard_normal(H)).astype(np.float32),
                nw=(1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32),
                S=(0.1 * rng.standard_normal((H, D, D))).astype(np.float32))


# The gated attention token: 8 query heads over 2 key/value heads of 256
# columns, caches of 4096 positions, a mid-context position (the pages give
# no dimensions; Metal's kernel handled positions below 4096).
ATQ_QHEADS = 8
ATQ_KVHEADS = 2
ATQ_DIM = 256
ATQ_CACHE = 4096
ATQ_POS = 2047


def atq_case(rng: np.random.Generator, Hq: int = ATQ_QHEADS, Hkv: int = ATQ_KVHEADS, D: int = ATQ_DIM,
             P: int = ATQ_CACHE, pos: int = ATQ_POS) -> dict:
    """Inputs of one atq token (names as abg_atq): q, gate, k, v ~ N(0,1);
    qn_w, kn_w ~ 1 + N(0, 0.1); cos, sin of angles uniform on [0, 2 pi) per
    column pair; cache rows below pos ~ N(0,1) (rows pos.. zero), float32."""
    ang = rng.uniform(0.0, 2.0 * np.pi, D // 2)
    Kc = np.zeros((Hkv, P, D), np.float32)
    Vc = np.zeros((Hkv, P, D), np.float32)
    Kc[:, :pos] = rng.standard_normal((Hkv, pos, D))
    Vc[:, :pos] = rng.standard_normal((Hkv, pos, D))
    return dict(q=rng.standard_normal(Hq * D).astype(np.float32),
                gate=rng.standard_normal(Hq * D).astype(np.float32),
                k=rng.standard_normal(Hkv * D).astype(np.float32),
                v=rng.standard_normal(Hkv * D).astype(np.float32),
                qn_w=(1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32),
                kn_w=(1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32),
                cos=np.cos(ang).astype(np.float32), sin=np.sin(ang).astype(np.float32),
                Kc=Kc, Vc=Vc, pos=pos)
