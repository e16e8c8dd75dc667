"""CPU oracle for q4mv / rmsq / swq / gsum -- TEST INFRASTRUCTURE ONLY.

This package is the plain, slow definition the CUDA library is checked
against.  Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it; the library never does, and the two share
no code.  The arithmetic lives in ``oracle.c`` (one IEEE binary32 operation per
C operation, built without contraction); this module only marshals numpy
arrays into it and composes the calls into a decode token.

Sources are the three Bend pull-request pages on the 4-bit product:
#1435 "Array.q4mv on Metal: one kernel thread per row ...", #1437
"Array.q4go/Array.q4wait queue Metal Q4 products ...", and #1440 "Metal:
queued rmsq, swq, gdn and atq kernels and a 4-row q4mv ...".

parity unpinned: ``hash32`` against the pages' printed hash (their generator
and hash function are not published).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no contraction, no fast math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            f32p = ctypes.POINTER(ctypes.c_float)
            u32p = ctypes.POINTER(ctypes.c_uint32)
            f64p = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            lib.or_tree.argtypes = [f32p, i64]
            lib.or_tree.restype = ctypes.c_float
            lib.or_gsum.argtypes = [f32p, f32p, i64]
            lib.or_q4mv.argtypes = [u32p, f32p, f32p, f32p, f32p, f32p, i64, i64, i64, i64]
            lib.or_q4mv_absmag.argtypes = [u32p, f32p, f32p, f32p, f32p, f64p, i64, i64, i64, i64]
            lib.or_rmsq.argtypes = [f32p, f32p, ctypes.c_float, f32p, f32p, i64]
            lib.or_exp.argtypes = [ctypes.c_float]
            lib.or_exp.restype = ctypes.c_float
            lib.or_exp_array.argtypes = [f32p, f32p, i64]
            lib.or_swq.argtypes = [f32p, f32p, f32p, i64]
            lib.or_fnv1a.argtypes = [ctypes.c_char_p, i64]
            lib.or_fnv1a.restype = ctypes.c_uint32
            lib.or_hash32.argtypes = [f32p, i64]
            lib.or_hash32.restype = ctypes.c_uint32
            vp = ctypes.c_void_p
            lib.or_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.or_bf16_to_f32.restype = ctypes.c_float
            lib.or_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.or_f16_to_f32.restype = ctypes.c_float
            lib.or_gsum_ex.argtypes = [f32p, f32p, i64, ctypes.c_int]
            lib.or_q4mv_ex.argtypes = [u32p, vp, vp, ctypes.c_int, ctypes.c_int, f32p, f32p, f32p, i64, i64, i64, i64]
            lib.or_log.argtypes = [ctypes.c_float]
            lib.or_log.restype = ctypes.c_float
            lib.or_log_array.argtypes = [f32p, f32p, i64]
            fl = ctypes.c_float
            lib.or_gdn.argtypes = [f32p, f32p, f32p, f32p, f32p, f32p, f32p, f32p, f32p, f32p, f32p, f32p,
                                   i64, i64, i64, fl, fl]
            lib.or_atq.argtypes = [f32p, f32p, f32p, f32p, f32p, f32p, f32p, f32p, f32p, f32p, f32p, f32p,
                                   i64, i64, i64, i64, i64, fl]
            _lib = lib
    return _lib


def _f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _u32(a):
    a = np.ascontiguousarray(a, dtype=np.uint32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32))


def _check_q4(w, scale, bias, x, xsum, rows, cols, row0, n):
    if cols <= 0 or cols % 64:
        raise ValueError("cols must be a positive multiple of 64")
    if row0 < 0 or n < 0 or row0 + n > rows:
        raise ValueError("row range out of bounds")
    G, W = cols // 64, cols // 8
    if w.size != rows * W or scale.size != rows * G or bias.size != rows * G:
        raise ValueError("weight arrays do not match rows x cols")
    if x.size != cols or xsum.size != G:
        raise ValueError("x / xsum do not match cols")


def tree(v) -> np.float32:
    """TREE(v): balanced pairwise sum in index order, odd element carried."""
    v, pv = _f32(v)
    return np.float32(_load().or_tree(pv, v.size))


def gsum(v) -> np.ndarray:
    """s[g] = TREE(v[64g:64g+64])."""
    v, pv = _f32(v)
    if v.size % 64:
        raise ValueError("length must be a multiple of 64")
    s = np.empty(v.size // 64, np.float32)
    _load().or_gsum(pv, _f32(s)[1], v.size)
    return s


def q4mv(w, scale, bias, x, xsum, cols, row0=0, n=None) -> np.ndarray:
    """y[i] = row row0+i of the affine 4-bit product (tree order)."""
    w, pw = _u32(w)
    scale, ps = _f32(scale)
    bias, pb = _f32(bias)
    x, px = _f32(x)
    xsum, pxs = _f32(xsum)
    rows = w.size // (cols // 8)
    n = rows - row0 if n is None else n
    _check_q4(w, scale, bias, x, xsum, rows, cols, row0, n)
    y = np.empty(n, np.float32)
    _load().or_q4mv(pw, ps, pb, px, pxs, _f32(y)[1], rows, cols, row0, n)
    return y


def q4mv_absmag(w, scale, bias, x, xsum, cols, row0=0, n=None) -> np.ndarray:
    """A_r = sum_g |scale*d| + |bias*xsum| in double (scales the fast-mode bound)."""
    w, pw = _u32(w)
    scale, ps = _f32(scale)
    bias, pb = _f32(bias)
    x, px = _f32(x)
    xsum, pxs = _f32(xsum)
    rows = w.size // (cols // 8)
    n = rows - row0 if n is None else n
    _check_q4(w, scale, bias, x, xsum, rows, cols, row0, n)
    a = np.empty(n, np.float64)
    _load().or_q4mv_absmag(pw, ps, pb, px, pxs, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                           rows, cols, row0, n)
    return a


def rmsq(x, wt, eps=1e-6):
    """(xn, xsum): RMS norm with weights, plus the group sums of xn."""
    x, px = _f32(x)
    wt, pwt = _f32(wt)
    if x.size % 64 or x.size == 0 or wt.size != x.size:
        raise ValueError("n must be a positive multiple of 64 and match the weights")
    xn = np.empty(x.size, np.float32)
    xs = np.empty(x.size // 64, np.float32)
    _load().or_rmsq(px, pwt, ctypes.c_float(np.float32(eps)), _f32(xn)[1], _f32(xs)[1], x.size)
    return xn, xs


def exp(v) -> np.ndarray:
    """The specified binary32 exponential, elementwise."""
    v, pv = _f32(v)
    out = np.empty(v.shape, np.float32)
    _load().or_exp_array(pv, _f32(out)[1], v.size)
    return out


def swq(a):
    """(o, osum): o = silu(gate) * up for a = [gate | up], plus group sums."""
    a, pa = _f32(a)
    if a.size % 128 or a.size == 0:
        raise ValueError("a must hold 2n values with n a positive multiple of 64")
    n = a.size // 2
    o = np.empty(n, np.float32)
    os_ = np.empty(n // 64, np.float32)
    _load().or_swq(pa, _f32(o)[1], _f32(os_)[1], n)
    return o, os_


def fnv1a(data: bytes) -> int:
    """32-bit FNV-1a over a byte string."""
    return int(_load().or_fnv1a(data, len(data)))


def hash32(y) -> int:
    """32-bit FNV-1a over y's little-endian binary32 bytes in index order."""
    y, py = _f32(y)
    return int(_load().or_hash32(py, y.size))


def decode_token(model, hidden, eps=1e-6, keep=False):
    """One synthetic decode token: the composition of the calls above.

    ``model`` is a ``synth.DecodeModel``.  Per layer:
    rmsq -> q, k, v products -> group sums of q -> o product (reads q) ->
    rmsq -> gate, up products -> swq -> down product; then a final rmsq and
    the output head.  Returns the head's output (and the per-layer values if
    ``keep``).
    """
    h = np.asarray(hidden, np.float32)
    trace = []
    for L in model.layers:
        xn, xs = rmsq(h, L.rms1, eps)
        q = q4mv(*L.q.arrays(), xn, xs, L.q.cols)
        k = q4mv(*L.k.arrays(), xn, xs, L.k.cols)
        v = q4mv(*L.v.arrays(), xn, xs, L.v.cols)
        qs = gsum(q)
        o = q4mv(*L.o.arrays(), q, qs, L.o.cols)
        xn2, xs2 = rmsq(o, L.rms2, eps)
        gate = q4mv(*L.gate.arrays(), xn2, xs2, L.gate.cols)
        up = q4mv(*L.up.arrays(), xn2, xs2, L.up.cols)
        s, ss = swq(np.concatenate([gate, up]))
        h = q4mv(*L.down.arrays(), s, ss, L.down.cols)
        if keep:
            trace.append(dict(xn=xn, xs=xs, q=q, k=k, v=v, qs=qs, o=o, xn2=xn2, xs2=xs2,
                              gate=gate, up=up, s=s, ss=ss, h=h))
    xf, xfs = rmsq(h, model.rms_final, eps)
    logits = q4mv(*model.head.arrays(), xf, xfs, model.head.cols)
    if keep:
        return logits, trace, (xf, xfs)
    return logits


SB_DTYPES = {"f32": 0, "bf16": 1, "f16": 2}


def half_to_f32(bits, dtype: str) -> np.ndarray:
    """Stored bf16 or f16 bit patterns (uint16) widened to f32, elementwise (exact)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    f = _load().or_bf16_to_f32 if dtype == "bf16" else _load().or_f16_to_f32
    return np.array([f(int(b)) for b in bits], np.float32)


def gsum_ex(v, gs: int) -> np.ndarray:
    """s[g] = TREE(v[gs*g : gs*g + gs])."""
    v, pv = _f32(v)
    if gs not in (32, 64, 128) or v.size % gs:
        raise ValueError("group size 32, 64 or 128 dividing the length")
    s = np.empty(v.size // gs, np.float32)
    _load().or_gsum_ex(pv, _f32(s)[1], v.size, gs)
    return s


def q4mv_ex(w, scale, bias, sb_dtype: str, gs: int, x, xsum, cols, row0=0, n=None) -> np.ndarray:
    """The product for group size gs and scale/bias stored as f32, bf16 or f16
    (scale and bias given as float32 arrays, or as uint16 bit patterns)."""
    if gs not in (32, 64, 128) or cols % gs or cols % 64:
        raise ValueError("group size 32, 64 or 128; cols a multiple of 64 and of gs")
    w, pw = _u32(w)
    dt = SB_DTYPES[sb_dtype]
    if dt == 0:
        scale = np.ascontiguousarray(scale, np.float32)
        bias = np.ascontiguousarray(bias, np.float32)
    else:
        scale = np.ascontiguousarray(scale, np.uint16)
        bias = np.ascontiguousarray(bias, np.uint16)
    x, px = _f32(x)
    xsum, pxs = _f32(xsum)
    rows = w.size // (cols // 8)
    n = rows - row0 if n is None else n
    G = cols // gs
    if scale.size != rows * G or bias.size != rows * G or x.size != cols or xsum.size != G:
        raise ValueError("array sizes do not match rows, cols and gs")
    if row0 < 0 or n < 0 or row0 + n > rows:
        raise ValueError("row range out of bounds")
    y = np.empty(n, np.float32)
    _load().or_q4mv_ex(pw, scale.ctypes.data, bias.ctypes.data, dt, gs, px, pxs, _f32(y)[1], rows, cols, row0, n)
    return y


def q4mm(w, scale, bias, X, XS, cols, row0=0, n=None) -> np.ndarray:
    """Batched product: Y[t] = q4mv(w, scale, bias, X[t], XS[t]) for each of the T
    activation rows of X [T][cols] (group sums XS [T][cols/64]).  A batch of
    decode tokens reads the same weights once for all of them; each token's
    result is by definition its own product, so this is that product applied
    row by row of X (no reordering across tokens)."""
    X = np.atleast_2d(np.asarray(X, np.float32))
    XS = np.atleast_2d(np.asarray(XS, np.float32))
    if X.shape[0] != XS.shape[0]:
        raise ValueError("X and XS hold different token counts")
    return np.stack([q4mv(w, scale, bias, X[t], XS[t], cols, row0=row0, n=n) for t in range(X.shape[0])])


def log(v) -> np.ndarray:
    """The specified binary32 natural logarithm, elementwise (oracle.c LOG)."""
    v, pv = _f32(v)
    out = np.empty(v.shape, np.float32)
    _load().or_log_array(pv, _f32(out)[1], v.size)
    return out


def gdn(x, conv, state, a, b, z, A_log, dt_bias, nw, S, eps=1e-6, eps_n=1e-6):
    """One token of the gated DeltaNet mixer (oracle.c or_gdn): returns
    (y, ysum, S_new, state_new) without touching the inputs.

    Shapes: x [3*H*D] (q | k | v), conv [3*H*D][K], state [3*H*D][K-1],
    a, b, A_log, dt_bias [H], z [H*D], nw [D], S [H][D][D] (keys by values).
    """
    S = np.array(S, dtype=np.float32, copy=True)
    H, D = S.shape[0], S.shape[1]
    if S.shape != (H, D, D) or D % 64 or D > 1024:
        raise ValueError("S must be [H][D][D] with D a multiple of 64, at most 1024")
    conv = np.ascontiguousarray(conv, dtype=np.float32)
    K = conv.shape[-1]
    if conv.shape != (3 * H * D, K) or not 2 <= K <= 8:
        raise ValueError("conv must be [3*H*D][K] with 2 <= K <= 8")
    state = np.array(state, dtype=np.float32, copy=True).reshape(3 * H * D, K - 1)
    x, px = _f32(x)
    if x.size != 3 * H * D:
        raise ValueError("x must hold 3*H*D values")
    a, pa = _f32(a)
    b, pb = _f32(b)
    A_log, pA = _f32(A_log)
    dt_bias, pdt = _f32(dt_bias)
    z, pz = _f32(z)
    nw, pn = _f32(nw)
    if a.size != H or b.size != H or A_log.size != H or dt_bias.size != H or z.size != H * D or nw.size != D:
        raise ValueError("a, b, A_log, dt_bias must hold H values, z H*D, nw D")
    y = np.empty(H * D, np.float32)
    ys = np.empty(H * D // 64, np.float32)
    _load().or_gdn(px, _f32(conv)[1], _f32(state)[1], pa, pb, pz, pA, pdt, pn, _f32(S)[1], _f32(y)[1],
                   _f32(ys)[1], H, D, K, ctypes.c_float(np.float32(eps)), ctypes.c_float(np.float32(eps_n)))
    return y, ys, S, state


def atq(q, gate, k, v, qn_w, kn_w, cos, sin, Kc, Vc, pos: int, eps=1e-6):
    """One token of gated attention at position pos (oracle.c or_atq): returns
    (y, ysum, Kc_new, Vc_new) without touching the inputs.

    Shapes: q, gate [Hq*D]; k, v [Hkv*D]; qn_w, kn_w [D]; cos, sin [D/2];
    Kc, Vc [Hkv][P][D] with rows < pos filled.
    """
    Kc = np.array(Kc, dtype=np.float32, copy=True)
    Vc = np.array(Vc, dtype=np.float32, copy=True)
    Hkv, P, D = Kc.shape
    q, pq = _f32(q)
    Hq = q.size // D
    if Vc.shape != Kc.shape or D % 64 or D > 1024 or q.size != Hq * D or Hq % Hkv or not 0 <= pos < P:
        raise ValueError("bad atq shapes")
    gate, pg = _f32(gate)
    k, pk = _f32(k)
    v, pv = _f32(v)
    qn_w, pqn = _f32(qn_w)
    kn_w, pkn = _f32(kn_w)
    cos, pc = _f32(cos)
    sin, ps = _f32(sin)
    if gate.size != Hq * D or k.size != Hkv * D or v.size != Hkv * D or qn_w.size != D or kn_w.size != D or \
            cos.size != D // 2 or sin.size != D // 2:
        raise ValueError("bad atq shapes")
    y = np.empty(Hq * D, np.float32)
    ys = np.empty(Hq * D // 64, np.float32)
    _load().or_atq(pq, pg, pk, pv, pqn, pkn, pc, ps, _f32(Kc)[1], _f32(Vc)[1], _f32(y)[1], _f32(ys)[1],
                   Hq, Hkv, D, P, pos, ctypes.c_float(np.float32(eps)))
    return y, ys, Kc, Vc
