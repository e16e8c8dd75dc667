"""Python binding of libabg.so: the GB300 affine 4-bit group-quantized
matrix-vector product (q4mv), its activation producers (rmsq, swq, gsum) and
the decode-token stage graph.

This module only marshals arguments: tensors become device pointers, the
current torch stream becomes a cudaStream_t, and status codes become
exceptions.  Every step of the computation runs in the library's CUDA kernels;
there is no CPU path.  PyTorch supplies device memory and streams.

The C declarations, with the meaning, layout, ownership and error behaviour
of every argument, are in include/abg.h.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "TREE", "FAST", "AbgError", "library", "q4mv", "q4mv_ex", "q4mm", "gsum", "rmsq", "swq", "StageGraph", "Node",
    "device_status", "set_q4mv_tuning", "MAX_COLS", "SB_F32", "SB_BF16", "SB_F16", "SB_TYPES", "swiglu_mlp_static",
]

TREE, FAST = 0, 1
MAX_COLS = 16384
NODE_Q4MV, NODE_RMSQ, NODE_SWQ, NODE_GSUM, NODE_GDN, NODE_ATQ, NODE_COPY = 0, 1, 2, 3, 4, 5, 6
PRO_NONE, PRO_GSUM, PRO_RMSQ, PRO_SWQ = 0, 1, 2, 3
SB_F32, SB_BF16, SB_F16 = 0, 1, 2
SB_TYPES = {"f32": SB_F32, "bf16": SB_BF16, "f16": SB_F16}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libabg.so")
_lock = threading.Lock()
_lib = None

_STATUS = {0: "ok", 1: "invalid argument", 2: "misaligned pointer", 3: "bad shape", 4: "output overlaps an input",
           5: "CUDA error", 6: "device wait timed out"}


class AbgError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {_STATUS.get(status, 'unknown status')} ({status})"
        if status == 5 and _lib is not None:
            msg += ": " + _lib.abg_last_cuda_error().decode()
        super().__init__(msg)


class _Node(ctypes.Structure):
    """Mirror of struct abg_node in include/abg.h."""
    _fields_ = [
        ("kind", ctypes.c_int32), ("stage", ctypes.c_int32),
        ("w", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("bias", ctypes.c_void_p),
        ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("row0", ctypes.c_int64), ("n", ctypes.c_int64),
        ("y", ctypes.c_void_p),
        ("prologue", ctypes.c_int32), ("eps", ctypes.c_float),
        ("x", ctypes.c_void_p), ("xsum", ctypes.c_void_p), ("wt", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("out_sum", ctypes.c_void_p),
        ("len", ctypes.c_int64),
        ("group", ctypes.c_int32), ("sb_type", ctypes.c_int32),
        ("args", ctypes.c_void_p),
    ]


class _GdnArgs(ctypes.Structure):
    """Mirror of struct abg_gdn_args in include/abg.h."""
    _fields_ = [(f, ctypes.c_void_p) for f in ("x", "conv", "state", "a", "b", "z", "A_log", "dt_bias", "nw", "S",
                                               "y", "ysum")] + \
               [("H", ctypes.c_int64), ("D", ctypes.c_int64), ("K", ctypes.c_int64),
                ("eps", ctypes.c_float), ("eps_n", ctypes.c_float)]


class _AtqArgs(ctypes.Structure):
    """Mirror of struct abg_atq_args in include/abg.h."""
    _fields_ = [(f, ctypes.c_void_p) for f in ("q", "gate", "k", "v", "qn_w", "kn_w", "cos", "sin", "Kc", "Vc", "y",
                                               "ysum")] + \
               [(f, ctypes.c_int64) for f in ("Hq", "Hkv", "D", "P", "pos")] + [("eps", ctypes.c_float)]


def library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Loads libabg.so (building it with nvcc first if it is missing or stale)."""
    global _lib
    if _lib is not None:  # loaded: no lock on the per-call path
        return _lib
    with _lock:
        if _lib is None:
            if build_if_missing:
                from . import _build
                if _build.stale():
                    _build.build()
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"the CUDA library {_LIB_PATH} is not built")
            lib = ctypes.CDLL(_LIB_PATH)
            P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            lib.abg_q4mv.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, I, I, P]
            lib.abg_gsum.argtypes = [P, P, I64, I, P]
            lib.abg_rmsq.argtypes = [P, P, ctypes.c_float, P, P, I64, I, P]
            lib.abg_swq.argtypes = [P, P, P, I64, I, P]
            lib.abg_q4mv_ex.argtypes = [P, P, P, I, I, P, P, P, I64, I64, I64, I64, I, I, P]
            lib.abg_q4mm.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, I64, I, I, P]
            lib.abg_gsum_ex.argtypes = [P, P, I64, I, I, P]
            lib.abg_rmsq_ex.argtypes = [P, P, ctypes.c_float, P, P, I64, I, I, P]
            lib.abg_swq_ex.argtypes = [P, P, P, I64, I, I, P]
            lib.abg_stage_graph_create.argtypes = [ctypes.POINTER(_Node), I64, I, I, ctypes.POINTER(P)]
            lib.abg_stage_graph_launch.argtypes = [P, P]
            lib.abg_stage_graph_launches.argtypes = [P, ctypes.POINTER(I64)]
            lib.abg_stage_graph_swiglu_pairs.argtypes = [P, ctypes.POINTER(I64)]
            lib.abg_swiglu_mlp_static.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, I64, I64, I64, I, P]
            lib.abg_stage_graph_destroy.argtypes = [P]
            F = ctypes.c_float
            lib.abg_gdn.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, I64, I64, I64, F, F, I, P]
            lib.abg_atq.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, I64, I64, I64, I64, I64, F, I, P]
            lib.abg_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), I]
            lib.abg_selftest_wait_timeout.argtypes = [P]
            lib.abg_set_q4mv_tuning.argtypes = [I, I, I, I]
            lib.abg_status_str.argtypes = [I]
            lib.abg_status_str.restype = ctypes.c_char_p
            lib.abg_last_cuda_error.argtypes = []
            lib.abg_last_cuda_error.restype = ctypes.c_char_p
            for f in ("abg_q4mv", "abg_q4mm", "abg_gsum", "abg_rmsq", "abg_swq", "abg_q4mv_ex", "abg_gsum_ex", "abg_rmsq_ex",
                      "abg_swq_ex", "abg_stage_graph_create",
                      "abg_stage_graph_launch", "abg_stage_graph_launches", "abg_stage_graph_swiglu_pairs",
                      "abg_stage_graph_destroy", "abg_swiglu_mlp_static", "abg_gdn", "abg_atq",
                      "abg_device_status", "abg_set_q4mv_tuning", "abg_selftest_wait_timeout"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _check(status: int, what: str):
    if status != 0:
        raise AbgError(status, what)


def _ptr(t, dtype=None, numel=None, name="tensor"):
    """Device pointer of a CUDA tensor (or an int address, passed through)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype and not (dtype == "word" and t.element_size() == 4 and
                                                         not t.is_floating_point()) \
            and not (dtype == "half" and t.element_size() == 2):
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {numel}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


_DTYPES = None


def _dtypes():
    global _DTYPES
    if _DTYPES is None:
        import torch
        _DTYPES = (torch.int32, torch.float32)
    return _DTYPES


def q4mv(w, scale, bias, x, xsum, y, cols: int, row0: int = 0, n: int | None = None, mode: int = TREE,
         rows_per_warp: int = 0, stream=None):
    """y[i] = row row0+i of the packed (rows x cols) matrix times x (see abg_q4mv)."""
    _, f32 = _dtypes()
    rows = w.shape[0] if w.dim() == 2 else w.numel() // (cols // 8)
    n = rows - row0 if n is None else n
    G, W = cols // 64, cols // 8
    st = library().abg_q4mv(
        _ptr(w, "word", rows * W, "w"), _ptr(scale, f32, rows * G, "scale"), _ptr(bias, f32, rows * G, "bias"),
        _ptr(x, f32, cols, "x"), _ptr(xsum, f32, G, "xsum"), _ptr(y, f32, n, "y"),
        rows, cols, row0, n, mode, rows_per_warp, _stream(stream))
    _check(st, "abg_q4mv")
    return y


def q4mv_ex(w, scale, bias, sb_type, group: int, x, xsum, y, cols: int, row0: int = 0, n: int | None = None,
            mode: int = TREE, rows_per_warp: int = 0, stream=None):
    """The product for groups of `group` columns with scale/bias stored as sb_type
    ("f32", "bf16", "f16" or an SB_* code); 16-bit scale and bias may be any
    2-byte tensor holding the bit patterns (see abg_q4mv_ex)."""
    _, f32 = _dtypes()
    sb = SB_TYPES[sb_type] if isinstance(sb_type, str) else sb_type
    rows = w.shape[0] if w.dim() == 2 else w.numel() // (cols // 8)
    n = rows - row0 if n is None else n
    G, W = cols // group, cols // 8
    sdt = f32 if sb == SB_F32 else "half"
    st = library().abg_q4mv_ex(
        _ptr(w, "word", rows * W, "w"), _ptr(scale, sdt, rows * G, "scale"), _ptr(bias, sdt, rows * G, "bias"),
        sb, group, _ptr(x, f32, cols, "x"), _ptr(xsum, f32, G, "xsum"), _ptr(y, f32, n, "y"),
        rows, cols, row0, n, mode, rows_per_warp, _stream(stream))
    _check(st, "abg_q4mv_ex")
    return y


def q4mm(w, scale, bias, X, XS, Y, cols: int, row0: int = 0, n: int | None = None, mode: int = TREE,
         rows_per_warp: int = 0, stream=None):
    """Y[t] = the product for token t of X [T][cols] (group sums XS [T][cols/64]),
    Y [T][n]; the weights are read once for the batch (see abg_q4mm)."""
    _, f32 = _dtypes()
    T = X.shape[0] if X.dim() == 2 else 1
    rows = w.shape[0] if w.dim() == 2 else w.numel() // (cols // 8)
    n = rows - row0 if n is None else n
    G, W = cols // 64, cols // 8
    st = library().abg_q4mm(
        _ptr(w, "word", rows * W, "w"), _ptr(scale, f32, rows * G, "scale"), _ptr(bias, f32, rows * G, "bias"),
        _ptr(X, f32, T * cols, "X"), _ptr(XS, f32, T * G, "XS"), _ptr(Y, f32, T * n, "Y"),
        rows, cols, row0, n, T, mode, rows_per_warp, _stream(stream))
    _check(st, "abg_q4mm")
    return Y


def _gdn_args(x, conv, state, a, b, z, A_log, dt_bias, nw, S, y, ysum, eps, eps_n):
    _, f32 = _dtypes()
    H, D = S.shape[0], S.shape[1]
    K = conv.shape[-1]
    C = 3 * H * D
    return _GdnArgs(
        _ptr(x, f32, C, "x"), _ptr(conv, f32, C * K, "conv"), _ptr(state, f32, C * (K - 1), "state"),
        _ptr(a, f32, H, "a"), _ptr(b, f32, H, "b"), _ptr(z, f32, H * D, "z"), _ptr(A_log, f32, H, "A_log"),
        _ptr(dt_bias, f32, H, "dt_bias"), _ptr(nw, f32, D, "nw"), _ptr(S, f32, H * D * D, "S"),
        _ptr(y, f32, H * D, "y"), _ptr(ysum, f32, H * D // 64, "ysum"), H, D, K, eps, eps_n)


def _atq_args(q, gate, k, v, qn_w, kn_w, cos, sin, Kc, Vc, y, ysum, pos, eps):
    _, f32 = _dtypes()
    Hkv, P, D = Kc.shape
    Hq = q.numel() // D
    return _AtqArgs(
        _ptr(q, f32, Hq * D, "q"), _ptr(gate, f32, Hq * D, "gate"), _ptr(k, f32, Hkv * D, "k"),
        _ptr(v, f32, Hkv * D, "v"), _ptr(qn_w, f32, D, "qn_w"), _ptr(kn_w, f32, D, "kn_w"),
        _ptr(cos, f32, D // 2, "cos"), _ptr(sin, f32, D // 2, "sin"), _ptr(Kc, f32, Hkv * P * D, "Kc"),
        _ptr(Vc, f32, Hkv * P * D, "Vc"), _ptr(y, f32, Hq * D, "y"), _ptr(ysum, f32, Hq * D // 64, "ysum"),
        Hq, Hkv, D, P, pos, eps)


def gdn(x, conv, state, a, b, z, A_log, dt_bias, nw, S, y, ysum, eps: float = 1e-6, eps_n: float = 1e-6,
        mode: int = TREE, stream=None):
    """One token of the gated DeltaNet mixer (see abg_gdn): S [H][D][D] and
    state [3*H*D][K-1] are updated in place; y [H*D] and ysum [H*D/64] written."""
    g = _gdn_args(x, conv, state, a, b, z, A_log, dt_bias, nw, S, y, ysum, eps, eps_n)
    st = library().abg_gdn(g.x, g.conv, g.state, g.a, g.b, g.z, g.A_log, g.dt_bias, g.nw, g.S, g.y, g.ysum,
                           g.H, g.D, g.K, ctypes.c_float(eps), ctypes.c_float(eps_n), mode, _stream(stream))
    _check(st, "abg_gdn")
    return y


def atq(q, gate, k, v, qn_w, kn_w, cos, sin, Kc, Vc, y, ysum, pos: int, eps: float = 1e-6, mode: int = TREE,
        stream=None):
    """One token of gated attention at position pos (see abg_atq): row pos of
    Kc and Vc [Hkv][P][D] is written; y [Hq*D] and ysum [Hq*D/64] written."""
    t = _atq_args(q, gate, k, v, qn_w, kn_w, cos, sin, Kc, Vc, y, ysum, pos, eps)
    st = library().abg_atq(t.q, t.gate, t.k, t.v, t.qn_w, t.kn_w, t.cos, t.sin, t.Kc, t.Vc, t.y, t.ysum,
                           t.Hq, t.Hkv, t.D, t.P, t.pos, ctypes.c_float(eps), mode, _stream(stream))
    _check(st, "abg_atq")
    return y


def swiglu_mlp_static(gate, up, down, x, xsum, y, cols: int, mode: int = TREE, stream=None):
    """y = down(silu(gate x) * (up x)) with no device allocation (abg_swiglu_mlp_static).

    gate, up, down are (w, scale, bias) triples of CUDA tensors: gate and up
    n x cols, down rows x n, with n <= 16384.  The intermediate vectors live in
    a static device array inside the library, shared by every call (see
    include/abg.h for who needs this and the ordering rule).
    """
    (wg, sg, bg), (wu, su, bu), (wd, sd, bd) = gate, up, down
    n = wg.numel() * 8 // cols
    rows = y.numel()
    _check(library().abg_swiglu_mlp_static(
        _ptr(wg, name="gate w"), _ptr(sg, name="gate scale"), _ptr(bg, name="gate bias"),
        _ptr(wu, name="up w"), _ptr(su, name="up scale"), _ptr(bu, name="up bias"),
        _ptr(wd, name="down w"), _ptr(sd, name="down scale"), _ptr(bd, name="down bias"),
        _ptr(x, name="x"), _ptr(xsum, name="xsum"), _ptr(y, name="y"), n, cols, rows, mode, _stream(stream)),
        "abg_swiglu_mlp_static")


def gsum(v, s, mode: int = TREE, stream=None, group: int = 64):
    """s[g] = tree sum of v[group*g : group*g+group]."""
    _, f32 = _dtypes()
    n = v.numel()
    st = library().abg_gsum_ex(_ptr(v, f32, n, "v"), _ptr(s, f32, n // group, "s"), n, group, mode, _stream(stream))
    _check(st, "abg_gsum_ex")
    return s


def rmsq(x, wt, xn, xsum, eps: float = 1e-6, mode: int = TREE, stream=None, group: int = 64):
    """RMS norm with weights into xn, and the group sums of xn into xsum."""
    _, f32 = _dtypes()
    n = x.numel()
    st = library().abg_rmsq_ex(_ptr(x, f32, n, "x"), _ptr(wt, f32, n, "wt"), ctypes.c_float(eps),
                               _ptr(xn, f32, n, "xn"), _ptr(xsum, f32, n // group, "xsum"), n, group, mode,
                               _stream(stream))
    _check(st, "abg_rmsq_ex")
    return xn, xsum


def swq(a, o, osum, mode: int = TREE, stream=None, group: int = 64):
    """o = silu(a[:n]) * a[n:], and the group sums of o into osum."""
    _, f32 = _dtypes()
    n = a.numel() // 2
    st = library().abg_swq_ex(_ptr(a, f32, 2 * n, "a"), _ptr(o, f32, n, "o"), _ptr(osum, f32, n // group, "osum"), n,
                              group, mode, _stream(stream))
    _check(st, "abg_swq_ex")
    return o, osum


class Node:
    """Builders for the stage-graph node kinds (fields as in struct abg_node)."""

    @staticmethod
    def q4mv(stage, w, scale, bias, y, cols, x, xsum=None, prologue=PRO_NONE, wt=None, eps=1e-6, row0=0, n=None,
             group=64, sb_type=SB_F32):
        rows = w.shape[0] if w.dim() == 2 else w.numel() // (cols // 8)
        n = rows - row0 if n is None else n
        sb = SB_TYPES[sb_type] if isinstance(sb_type, str) else sb_type
        nd = _Node(kind=NODE_Q4MV, stage=stage, w=_ptr(w, name="w"), scale=_ptr(scale, name="scale"),
                   bias=_ptr(bias, name="bias"), rows=rows, cols=cols, row0=row0, n=n, y=_ptr(y, name="y"),
                   prologue=prologue, eps=eps, x=_ptr(x, name="x"), xsum=_ptr(xsum, name="xsum"),
                   wt=_ptr(wt, name="wt"), group=group, sb_type=sb)
        return nd

    @staticmethod
    def rmsq(stage, x, wt, out, out_sum, eps=1e-6, group=64):
        return _Node(kind=NODE_RMSQ, stage=stage, x=_ptr(x, name="x"), wt=_ptr(wt, name="wt"), out=_ptr(out, name="out"),
                     out_sum=_ptr(out_sum, name="out_sum"), eps=eps, len=x.numel(), group=group)

    @staticmethod
    def swq(stage, a, out, out_sum, group=64):
        return _Node(kind=NODE_SWQ, stage=stage, x=_ptr(a, name="a"), out=_ptr(out, name="out"),
                     out_sum=_ptr(out_sum, name="out_sum"), len=a.numel() // 2, group=group)

    @staticmethod
    def gsum(stage, v, out_sum, group=64):
        return _Node(kind=NODE_GSUM, stage=stage, x=_ptr(v, name="v"), out_sum=_ptr(out_sum, name="out_sum"),
                     len=v.numel(), group=group)

    @staticmethod
    def gdn(stage, x, conv, state, a, b, z, A_log, dt_bias, nw, S, y, ysum, eps=1e-6, eps_n=1e-6):
        """A gdn node: arguments as gdn()."""
        g = _gdn_args(x, conv, state, a, b, z, A_log, dt_bias, nw, S, y, ysum, eps, eps_n)
        nd = _Node(kind=NODE_GDN, stage=stage, args=ctypes.addressof(g))
        nd._args = g  # read when the graph is created
        return nd

    @staticmethod
    def atq(stage, q, gate, k, v, qn_w, kn_w, cos, sin, Kc, Vc, y, ysum, pos, eps=1e-6):
        """An atq node for position pos (fixed in the graph): arguments as atq()."""
        t = _atq_args(q, gate, k, v, qn_w, kn_w, cos, sin, Kc, Vc, y, ysum, pos, eps)
        nd = _Node(kind=NODE_ATQ, stage=stage, args=ctypes.addressof(t))
        nd._args = t
        return nd

    @staticmethod
    def copy(stage, src, dst):
        """A copy node: src's float32 values into dst.  Each is a CUDA tensor or
        a pinned CPU tensor, so that a replay can take its inputs from host
        memory and hand its results back there."""
        import torch
        for t, name in ((src, "src"), (dst, "dst")):
            if t.dtype != torch.float32 or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous float32 tensor")
            if not t.is_cuda and not t.is_pinned():
                raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
        if dst.numel() < src.numel():
            raise ValueError(f"dst holds {dst.numel()} elements, needs {src.numel()}")
        return _Node(kind=NODE_COPY, stage=stage, x=src.data_ptr(), out=dst.data_ptr(), len=src.numel())


class StageGraph:
    """A decode token's stages recorded into one CUDA graph (abg_stage_graph_*).

    ``keep`` holds references to the tensors the nodes point at, so they stay
    allocated as long as the graph (the lifetime rule of abg.h).
    """

    def __init__(self, nodes, mode: int = TREE, rows_per_warp: int = 0, keep=()):
        arr = (_Node * len(nodes))(*nodes)
        h = ctypes.c_void_p()
        _check(library().abg_stage_graph_create(arr, len(nodes), mode, rows_per_warp, ctypes.byref(h)),
               "abg_stage_graph_create")
        self._h = h
        self._keep = list(keep)
        n = ctypes.c_int64()
        _check(library().abg_stage_graph_launches(self._h, ctypes.byref(n)), "abg_stage_graph_launches")
        self.launches = n.value
        _check(library().abg_stage_graph_swiglu_pairs(self._h, ctypes.byref(n)), "abg_stage_graph_swiglu_pairs")
        self.swiglu_pairs = n.value

    def launch(self, stream=None):
        _check(library().abg_stage_graph_launch(self._h, _stream(stream)), "abg_stage_graph_launch")

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _check(library().abg_stage_graph_destroy(self._h), "abg_stage_graph_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def device_status(clear: bool = True) -> int:
    """The device status word's bits (bit 0: a bounded device wait timed out)."""
    bits = ctypes.c_uint32()
    st = library().abg_device_status(ctypes.byref(bits), 1 if clear else 0)
    if st not in (0, 6):
        _check(st, "abg_device_status")
    return bits.value


def selftest_wait_timeout(stream=None):
    """Enqueues the failure-detection self-test (abg_selftest_wait_timeout): a product
    whose bounded waits run out after about 0.5 s; read the result with device_status()."""
    _check(library().abg_selftest_wait_timeout(_stream(stream)), "abg_selftest_wait_timeout")


def set_q4mv_tuning(smem_kb: int = 0, consumer_warps: int = 0, blocks_per_sm: int = 0, stage_kb: int = 0):
    _check(library().abg_set_q4mv_tuning(smem_kb, consumer_warps, blocks_per_sm, stage_kb), "abg_set_q4mv_tuning")
