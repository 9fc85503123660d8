"""FP64 CPU oracle for convolution forward, input gradient, and weight and bias gradients.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the package smoke check
and by the benchmark's CPU-baseline leg, never by the product path.  It shares
no code with the CUDA library; the only thing both sides take is the seeded
input generator in ``synth``.

The arithmetic lives in ``conv_oracle.c`` (plain nested loops, double
accumulation); this module compiles it with gcc when needed and marshals numpy
arrays through ctypes.  See that file's header for the definitions it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


class _Desc(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int64) for name in (
        "n", "c_in", "c_out", "groups", "in_h", "in_w", "k_h", "k_w",
        "s_h", "s_w", "p_h", "p_w", "d_h", "d_w", "p_h_end", "p_w_end",
        "in_d", "k_d", "s_d", "p_d", "p_d_end", "d_d")] + [
        ("nhwc", ctypes.c_int32), ("w_ohwi", ctypes.c_int32)]


@dataclass(frozen=True)
class Conv:
    """Shape of one convolution as the oracle sees it.

    ``spatial_dims`` is 1 for conv1d (NCL / NLC; ``in_hw = (1, L)``), 2 for
    conv2d and 3 for conv3d (then ``in_hw``, ``k``, ``stride``, ``pad``, ``dil`` and
    ``pad_end`` are (depth, height, width) triples).  ``nhwc`` selects channels-last
    activations, ``w_ohwi`` selects the [C_out, (KD,) KH, KW, C_in/G] weight order
    instead of [C_out, C_in/G, (KD,) KH, KW].
    """
    n: int
    c_in: int
    c_out: int
    in_hw: tuple
    k: tuple
    stride: tuple = (1, 1)
    pad: tuple = (0, 0)
    dil: tuple = (1, 1)
    groups: int = 1
    nhwc: bool = False
    w_ohwi: bool = False
    spatial_dims: int = 2
    pad_end: tuple = None   # padding after each axis; None: the same as ``pad`` (symmetric)

    def pads_end(self):
        return tuple(self.pad) if self.pad_end is None else tuple(self.pad_end)

    def _full(self, t, default):
        """A per-axis tuple with one entry per axis of ``in_hw`` (defaults, such as stride (1, 1),
        are pairs: a 3-D shape takes the default for its leading depth entry)."""
        t = tuple(t)
        return (default,) * (len(self.in_hw) - len(t)) + t

    def _dhw(self, t, depth_default):
        """(depth, height, width) of a per-axis tuple; depth_default for 1-D and 2-D shapes."""
        t = self._full(t, depth_default)
        return t if self.spatial_dims == 3 else (depth_default,) + t

    def _c(self) -> _Desc:
        ind, inh, inw = self._dhw(self.in_hw, 1)
        kd, kh, kw = self._dhw(self.k, 1)
        sd, sh, sw = self._dhw(self.stride, 1)
        pd, ph, pw = self._dhw(self.pad, 0)
        dd, dh, dw = self._dhw(self.dil, 1)
        ped, peh, pew = self._dhw(self.pads_end(), 0)
        return _Desc(self.n, self.c_in, self.c_out, self.groups, inh, inw, kh, kw, sh, sw, ph, pw, dh, dw,
                     peh, pew, ind, kd, sd, pd, ped, dd, int(self.nhwc), int(self.w_ohwi))

    def out_hw(self):
        """Output extent per spatial axis: (oh, ow), or (od, oh, ow) for 3-D shapes."""
        k, s, p, d = self._full(self.k, 1), self._full(self.stride, 1), self._full(self.pad, 0), self._full(self.dil, 1)
        pe = self._full(self.pads_end(), 0)
        return tuple(out_size2(self.in_hw[i], k[i], s[i], p[i], pe[i], d[i]) for i in range(len(self.in_hw)))

    def x_shape(self):
        return _act_shape(self, self.c_in, self.in_hw)

    def y_shape(self):
        return _act_shape(self, self.c_out, self.out_hw())

    def w_shape(self):
        cpg = self.c_in // self.groups
        if self.spatial_dims == 1:
            return (self.c_out, self.k[1], cpg) if self.w_ohwi else (self.c_out, cpg, self.k[1])
        if self.w_ohwi:
            return (self.c_out,) + tuple(self.k) + (cpg,)
        return (self.c_out, cpg) + tuple(self.k)


def _act_shape(c: Conv, ch: int, hw):
    if c.spatial_dims == 1:
        return (c.n, hw[1], ch) if c.nhwc else (c.n, ch, hw[1])
    return (c.n,) + tuple(hw) + (ch,) if c.nhwc else (c.n, ch) + tuple(hw)


def build(force: bool = False) -> str:
    """Compile conv_oracle.c into liboracle.so next to it (plain -O2, no tuning)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + ".tmp.%d" % os.getpid()
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER
        f32p, f64p, i64p = P(ctypes.c_float), P(ctypes.c_double), P(ctypes.c_int64)
        lib.oracle_out_size.argtypes = [ctypes.c_int64] * 5 + [i64p]
        lib.oracle_out_size.restype = ctypes.c_int
        lib.oracle_out_size2.argtypes = [ctypes.c_int64] * 6 + [i64p]
        lib.oracle_out_size2.restype = ctypes.c_int
        lib.oracle_check.argtypes = [P(_Desc), i64p, i64p]
        lib.oracle_check.restype = ctypes.c_int
        for name in ("oracle_conv_fwd",):
            getattr(lib, name).argtypes = [P(_Desc), f32p, f32p, f32p, f64p]
            getattr(lib, name).restype = ctypes.c_int
        for name in ("oracle_conv_dgrad", "oracle_conv_dgrad_scatter"):
            getattr(lib, name).argtypes = [P(_Desc), f32p, f32p, f64p]
            getattr(lib, name).restype = ctypes.c_int
        lib.oracle_conv_fwd_points.argtypes = [P(_Desc), f32p, f32p, f32p, i64p, ctypes.c_int64, f64p]
        lib.oracle_conv_fwd_points.restype = None
        lib.oracle_conv_fwd_points3.argtypes = [P(_Desc), f32p, f32p, f32p, i64p, ctypes.c_int64, f64p]
        lib.oracle_conv_fwd_points3.restype = None
        lib.oracle_conv_dgrad_points3.argtypes = [P(_Desc), f32p, f32p, i64p, ctypes.c_int64, f64p]
        lib.oracle_conv_dgrad_points3.restype = None
        lib.oracle_conv_wgrad_points3.argtypes = [P(_Desc), f32p, f32p, i64p, ctypes.c_int64, f64p]
        lib.oracle_conv_wgrad_points3.restype = None
        lib.oracle_conv_dgrad_points.argtypes = [P(_Desc), f32p, f32p, i64p, ctypes.c_int64, f64p]
        lib.oracle_conv_dgrad_points.restype = None
        lib.oracle_conv_wgrad.argtypes = [P(_Desc), f32p, f32p, f64p]
        lib.oracle_conv_wgrad.restype = ctypes.c_int
        lib.oracle_conv_bgrad.argtypes = [P(_Desc), f32p, f64p]
        lib.oracle_conv_bgrad.restype = ctypes.c_int
        lib.oracle_conv_wgrad_points.argtypes = [P(_Desc), f32p, f32p, i64p, ctypes.c_int64, f64p]
        lib.oracle_conv_wgrad_points.restype = None
        _lib = lib
    return _lib


def _f32(a, shape=None):
    a = np.ascontiguousarray(a, dtype=np.float32)
    if shape is not None and a.size != int(np.prod(shape)):
        raise ValueError("array has %d elements, expected shape %s" % (a.size, shape))
    return a


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def out_size(in_: int, k: int, s: int, p: int, d: int):
    """Output length along one axis, or None when the shape is rejected."""
    out = ctypes.c_int64(0)
    rc = _load().oracle_out_size(in_, k, s, p, d, ctypes.byref(out))
    return None if rc != 0 else out.value


def out_size2(in_: int, k: int, s: int, p_begin: int, p_end: int, d: int):
    """Output length along one axis with (begin, end) padding, or None when the shape is rejected."""
    out = ctypes.c_int64(0)
    rc = _load().oracle_out_size2(in_, k, s, p_begin, p_end, d, ctypes.byref(out))
    return None if rc != 0 else out.value


def check(c: Conv) -> bool:
    """True when the oracle accepts the shape (nonzero extents, divisibility, kernel fits)."""
    oh, ow = ctypes.c_int64(0), ctypes.c_int64(0)
    return _load().oracle_check(ctypes.byref(c._c()), ctypes.byref(oh), ctypes.byref(ow)) == 0


def conv_fwd(c: Conv, x, w, bias=None) -> np.ndarray:
    """Whole forward output in fp64, shaped like the layout ``c`` names."""
    x, w = _f32(x, c.x_shape()), _f32(w, c.w_shape())
    b = None if bias is None else _f32(bias, (c.c_out,))
    y = np.empty(c.y_shape(), dtype=np.float64)
    rc = _load().oracle_conv_fwd(ctypes.byref(c._c()), _ptr(x, ctypes.c_float), _ptr(w, ctypes.c_float),
                                 _ptr(b, ctypes.c_float), _ptr(y, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle rejected the shape")
    return y


def conv_dgrad(c: Conv, dy, w, scatter: bool = False) -> np.ndarray:
    """Whole input gradient in fp64 (gather form, or the scatter form when asked)."""
    dy, w = _f32(dy, c.y_shape()), _f32(w, c.w_shape())
    dx = np.empty(c.x_shape(), dtype=np.float64)
    fn = _load().oracle_conv_dgrad_scatter if scatter else _load().oracle_conv_dgrad
    rc = fn(ctypes.byref(c._c()), _ptr(dy, ctypes.c_float), _ptr(w, ctypes.c_float), _ptr(dx, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle rejected the shape")
    return dx


def conv_transpose(c: Conv, x, w, bias=None) -> np.ndarray:
    """Transposed convolution forward in fp64, by its definition: the input gradient of the
    convolution ``c`` applied to ``x``, then ``bias[channel]`` added to every output element of
    that channel (oarust ``conv_transpose_2d`` runs the same two steps: the transposed scatter,
    then a separate bias pass).  ``x`` has c's output shape, the result c's input shape, and the
    bias has ``c.c_in`` entries (the transposed convolution's output channels)."""
    y = conv_dgrad(c, x, w)
    if bias is not None:
        b = _f32(bias, (c.c_in,)).astype(np.float64)
        axis = y.ndim - 1 if c.nhwc else 1
        shape = [1] * y.ndim
        shape[axis] = c.c_in
        y = y + b.reshape(shape)
    return y


def conv_fwd_points(c: Conv, x, w, bias, idx) -> np.ndarray:
    """Forward outputs at an (count, 4) array of (n, c_out, oh, ow) indices, or for a 3-D shape an
    (count, 5) array of (n, c_out, od, oh, ow) indices."""
    x, w = _f32(x, c.x_shape()), _f32(w, c.w_shape())
    b = None if bias is None else _f32(bias, (c.c_out,))
    k = 5 if c.spatial_dims == 3 else 4
    idx = np.ascontiguousarray(idx, dtype=np.int64).reshape(-1, k)
    out = np.empty(idx.shape[0], dtype=np.float64)
    fn = _load().oracle_conv_fwd_points3 if k == 5 else _load().oracle_conv_fwd_points
    fn(ctypes.byref(c._c()), _ptr(x, ctypes.c_float), _ptr(w, ctypes.c_float), _ptr(b, ctypes.c_float),
       _ptr(idx, ctypes.c_int64), idx.shape[0], _ptr(out, ctypes.c_double))
    return out


def conv_dgrad_points(c: Conv, dy, w, idx) -> np.ndarray:
    """Input-gradient elements at an (count, 4) array of (n, c_in, ih, iw) indices, or for a 3-D
    shape an (count, 5) array of (n, c_in, id, ih, iw) indices."""
    dy, w = _f32(dy, c.y_shape()), _f32(w, c.w_shape())
    k = 5 if c.spatial_dims == 3 else 4
    idx = np.ascontiguousarray(idx, dtype=np.int64).reshape(-1, k)
    out = np.empty(idx.shape[0], dtype=np.float64)
    fn = _load().oracle_conv_dgrad_points3 if k == 5 else _load().oracle_conv_dgrad_points
    fn(ctypes.byref(c._c()), _ptr(dy, ctypes.c_float), _ptr(w, ctypes.c_float), _ptr(idx, ctypes.c_int64),
       idx.shape[0], _ptr(out, ctypes.c_double))
    return out


def conv_wgrad(c: Conv, x, dy) -> np.ndarray:
    """Whole weight gradient in fp64, shaped like the weight layout ``c`` names: every
    (c_out, c_in_local, kh, kw) element is the sum over batch and output positions of the output
    gradient times the input element the forward multiplied by that weight."""
    x, dy = _f32(x, c.x_shape()), _f32(dy, c.y_shape())
    dw = np.empty(c.w_shape(), dtype=np.float64)
    rc = _load().oracle_conv_wgrad(ctypes.byref(c._c()), _ptr(x, ctypes.c_float), _ptr(dy, ctypes.c_float),
                                   _ptr(dw, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle rejected the shape")
    return dw


def conv_bgrad(c: Conv, dy) -> np.ndarray:
    """Bias gradient in fp64: the output gradient summed over batch and positions, per channel."""
    dy = _f32(dy, c.y_shape())
    db = np.empty((c.c_out,), dtype=np.float64)
    rc = _load().oracle_conv_bgrad(ctypes.byref(c._c()), _ptr(dy, ctypes.c_float), _ptr(db, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle rejected the shape")
    return db


def conv_wgrad_points(c: Conv, x, dy, idx) -> np.ndarray:
    """Weight-gradient elements at an (count, 4) array of (c_out, c_in_local, kh, kw) indices, or for a
    3-D shape an (count, 5) array of (c_out, c_in_local, kd, kh, kw) indices."""
    x, dy = _f32(x, c.x_shape()), _f32(dy, c.y_shape())
    k = 5 if c.spatial_dims == 3 else 4
    idx = np.ascontiguousarray(idx, dtype=np.int64).reshape(-1, k)
    out = np.empty(idx.shape[0], dtype=np.float64)
    fn = _load().oracle_conv_wgrad_points3 if k == 5 else _load().oracle_conv_wgrad_points
    fn(ctypes.byref(c._c()), _ptr(x, ctypes.c_float), _ptr(dy, ctypes.c_float), _ptr(idx, ctypes.c_int64),
       idx.shape[0], _ptr(out, ctypes.c_double))
    return out
