"""Python binding of the gbconv C ABI (include/gbconv.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libgbconv.so.  The raw entry points keep the C names
(``gbconv_fwd``, ``gbconv_bwd_data`` ...) and take integer device addresses;
``conv_fwd`` / ``conv_bwd_data`` wrap them for torch tensors (device memory
and the current stream come from PyTorch; nothing else does).

Importing this module loads libgbconv.so and fails loudly if it has not been
built (``python convolution_conv_fwd_gb300/build.py``): there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgbconv.so")

# status codes
GBCONV_OK, GBCONV_EINVAL, GBCONV_EUNSUPPORTED, GBCONV_ECUDA, GBCONV_ETIMEOUT = range(5)
# layouts / dtypes
GBCONV_NCHW, GBCONV_NHWC = 0, 1
GBCONV_W_OIHW, GBCONV_W_OHWI = 0, 1
GBCONV_F32, GBCONV_BF16 = 0, 1
GBCONV_PAD_SYMMETRIC, GBCONV_PAD_BEGIN_END = 0, 1
# kernel families
KERNELS = {0: "direct", 1: "depthwise", 2: "pointwise", 3: "implicit", 4: "dgrad", 5: "direct_dgrad",
           6: "depthwise_dgrad", 7: "direct_wgrad", 8: "wgrad", 9: "smallgroup", 10: "smallgroup_dgrad"}
GBCONV_OP_FWD, GBCONV_OP_BWD_DATA, GBCONV_OP_BWD_FILTER = 0, 1, 2

EXPORTS = ("gbconv_out_shape", "gbconv_select", "gbconv_describe", "gbconv_fwd", "gbconv_bwd_data", "gbconv_conv_transpose",
           "gbconv_bwd_filter_workspace", "gbconv_bwd_filter", "gbconv_bwd_filter_noalloc",
           "gbconv_pack_weight", "gbconv_device_status", "gbconv_set_wait_limit_ns", "gbconv_kernels_launched",
           "gbconv_status_string", "gbconv_host_staging_bytes", "gbconv_fwd_host", "gbconv_bwd_data_host",
           "gbconv_conv_transpose_host")


class Desc(ctypes.Structure):
    """Mirror of gbconv_desc."""
    _fields_ = [("spatial_dims", ctypes.c_int32), ("layout", ctypes.c_int32), ("wlayout", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("n", ctypes.c_int64), ("c_in", ctypes.c_int64),
                ("c_out", ctypes.c_int64), ("groups", ctypes.c_int64), ("in_", ctypes.c_int64 * 3),
                ("k", ctypes.c_int64 * 3), ("stride", ctypes.c_int64 * 3), ("pad", ctypes.c_int64 * 3),
                ("dil", ctypes.c_int64 * 3), ("pad_end", ctypes.c_int64 * 3), ("pad_mode", ctypes.c_int32)]


class GbconvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s: %s (status %d)" % (what, status_string(status), status))
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libgbconv.so is not built at %s; run `python convolution_conv_fwd_gb300/build.py`"
                          % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    vp, st = ctypes.c_void_p, ctypes.c_int
    lib.gbconv_out_shape.argtypes = [P(Desc), P(ctypes.c_int64)]
    lib.gbconv_select.argtypes = [P(Desc), ctypes.c_int32, P(ctypes.c_int32)]
    lib.gbconv_describe.argtypes = [P(Desc), ctypes.c_int32, ctypes.c_char_p, ctypes.c_int64]
    lib.gbconv_fwd.argtypes = [P(Desc), vp, vp, vp, vp, vp]
    lib.gbconv_bwd_data.argtypes = [P(Desc), vp, vp, vp, vp]
    lib.gbconv_conv_transpose.argtypes = [P(Desc), vp, vp, vp, vp, vp]
    lib.gbconv_bwd_filter_workspace.argtypes = [P(Desc), P(ctypes.c_int64)]
    lib.gbconv_bwd_filter.argtypes = [P(Desc), vp, vp, vp, vp, vp, ctypes.c_int64, vp]
    lib.gbconv_bwd_filter_noalloc.argtypes = [P(Desc), vp, vp, vp, vp, vp]
    lib.gbconv_pack_weight.argtypes = [P(Desc), vp, vp, vp]
    lib.gbconv_device_status.argtypes = [vp]
    lib.gbconv_host_staging_bytes.argtypes = [P(Desc), ctypes.c_int32, ctypes.c_int32, P(ctypes.c_int64)]
    lib.gbconv_fwd_host.argtypes = [P(Desc), vp, vp, vp, vp, vp, ctypes.c_int64, ctypes.c_int32, vp, vp]
    lib.gbconv_bwd_data_host.argtypes = [P(Desc), vp, vp, vp, vp, ctypes.c_int64, ctypes.c_int32, vp, vp]
    lib.gbconv_conv_transpose_host.argtypes = [P(Desc), vp, vp, vp, vp, vp, ctypes.c_int64, ctypes.c_int32, vp, vp]
    for f in ("gbconv_out_shape", "gbconv_select", "gbconv_describe", "gbconv_conv_transpose", "gbconv_fwd",
              "gbconv_bwd_data", "gbconv_bwd_filter_workspace", "gbconv_bwd_filter", "gbconv_bwd_filter_noalloc",
              "gbconv_pack_weight", "gbconv_device_status", "gbconv_host_staging_bytes", "gbconv_fwd_host",
              "gbconv_bwd_data_host", "gbconv_conv_transpose_host"):
        getattr(lib, f).restype = st
    lib.gbconv_set_wait_limit_ns.argtypes = [ctypes.c_int64]
    lib.gbconv_set_wait_limit_ns.restype = ctypes.c_int64
    lib.gbconv_kernels_launched.argtypes = []
    lib.gbconv_kernels_launched.restype = ctypes.c_uint64
    lib.gbconv_status_string.argtypes = [st]
    lib.gbconv_status_string.restype = ctypes.c_char_p
    return lib


_lib = _load()


# ---------------------------------------------------------------- raw C entry points

def gbconv_out_shape(desc: Desc):
    """(OH, OW) for 2-D, (L_out, 1) for 1-D, (OD, OH, OW) for 3-D descriptors."""
    out = (ctypes.c_int64 * 3)()
    s = _lib.gbconv_out_shape(ctypes.byref(desc), out)
    if s != GBCONV_OK:
        raise GbconvError(s, "gbconv_out_shape")
    if desc.spatial_dims == 3:
        return int(out[0]), int(out[1]), int(out[2])
    return int(out[0]), int(out[1])


def gbconv_select(desc: Desc, op: int) -> str:
    k = ctypes.c_int32(-1)
    s = _lib.gbconv_select(ctypes.byref(desc), op, ctypes.byref(k))
    if s != GBCONV_OK:
        raise GbconvError(s, "gbconv_select")
    return KERNELS[k.value]


def gbconv_describe(desc: Desc, op: int) -> str:
    buf = ctypes.create_string_buffer(256)
    s = _lib.gbconv_describe(ctypes.byref(desc), op, buf, len(buf))
    if s != GBCONV_OK:
        raise GbconvError(s, "gbconv_describe")
    return buf.value.decode()


def gbconv_fwd(desc: Desc, x: int, w: int, bias: int | None, y: int, stream: int) -> int:
    return _lib.gbconv_fwd(ctypes.byref(desc), x, w, bias or None, y, stream or None)


def gbconv_bwd_data(desc: Desc, dy: int, w: int, dx: int, stream: int) -> int:
    return _lib.gbconv_bwd_data(ctypes.byref(desc), dy, w, dx, stream or None)


def gbconv_conv_transpose(desc: Desc, x: int, w: int, bias: int | None, y: int, stream: int) -> int:
    return _lib.gbconv_conv_transpose(ctypes.byref(desc), x, w, bias or None, y, stream or None)


def gbconv_bwd_filter_workspace(desc: Desc) -> int:
    b = ctypes.c_int64(0)
    s = _lib.gbconv_bwd_filter_workspace(ctypes.byref(desc), ctypes.byref(b))
    if s != GBCONV_OK:
        raise GbconvError(s, "gbconv_bwd_filter_workspace")
    return int(b.value)


def gbconv_bwd_filter(desc: Desc, x: int, dy: int, dw: int, db: int | None, workspace: int | None,
                      workspace_bytes: int, stream: int) -> int:
    return _lib.gbconv_bwd_filter(ctypes.byref(desc), x, dy, dw, db or None, workspace or None, workspace_bytes,
                                  stream or None)


# Size of the library's static scratch array (GBCONV_NOALLOC_WORKSPACE_BYTES in include/gbconv.h).
NOALLOC_WORKSPACE_BYTES = 32 << 20


def gbconv_bwd_filter_noalloc(desc: Desc, x: int, dy: int, dw: int, db: int | None, stream: int) -> int:
    """The weight gradient on the library's own static scratch array, for callers that cannot
    allocate device memory (no workspace argument; see include/gbconv.h)."""
    return _lib.gbconv_bwd_filter_noalloc(ctypes.byref(desc), x, dy, dw, db or None, stream or None)


def gbconv_pack_weight(desc: Desc, w_oihw: int, w_ohwi: int, stream: int) -> int:
    return _lib.gbconv_pack_weight(ctypes.byref(desc), w_oihw, w_ohwi, stream or None)


def gbconv_host_staging_bytes(desc: Desc, op: int, with_bias: bool = False) -> int:
    b = ctypes.c_int64(0)
    s = _lib.gbconv_host_staging_bytes(ctypes.byref(desc), op, int(bool(with_bias)), ctypes.byref(b))
    if s != GBCONV_OK:
        raise GbconvError(s, "gbconv_host_staging_bytes")
    return int(b.value)


def gbconv_fwd_host(desc: Desc, x: int, w: int, bias: int | None, y: int, staging: int, staging_bytes: int,
                    slices: int, stream: int, done_event: int | None = None) -> int:
    """gbconv_fwd on host buffers (x, w, bias, y host addresses), pipelined in batch slices through the
    device staging buffer: synchronous, or recording ``done_event`` (a raw cudaEvent_t) at the end."""
    return _lib.gbconv_fwd_host(ctypes.byref(desc), x, w, bias or None, y, staging, staging_bytes, slices,
                                stream or None, done_event or None)


def gbconv_bwd_data_host(desc: Desc, dy: int, w: int, dx: int, staging: int, staging_bytes: int, slices: int,
                         stream: int, done_event: int | None = None) -> int:
    return _lib.gbconv_bwd_data_host(ctypes.byref(desc), dy, w, dx, staging, staging_bytes, slices, stream or None,
                                     done_event or None)


def gbconv_conv_transpose_host(desc: Desc, x: int, w: int, bias: int | None, y: int, staging: int,
                               staging_bytes: int, slices: int, stream: int, done_event: int | None = None) -> int:
    return _lib.gbconv_conv_transpose_host(ctypes.byref(desc), x, w, bias or None, y, staging, staging_bytes, slices,
                                           stream or None, done_event or None)


def gbconv_device_status(stream: int) -> int:
    return _lib.gbconv_device_status(stream or None)


def gbconv_set_wait_limit_ns(ns: int) -> int:
    """Bound of the kernels' internal waits for later launches (<= 0: the 2 s default); returns the
    previous bound."""
    return int(_lib.gbconv_set_wait_limit_ns(int(ns)))


def gbconv_kernels_launched() -> int:
    return int(_lib.gbconv_kernels_launched())


def status_string(status: int) -> str:
    return _lib.gbconv_status_string(status).decode()


# ---------------------------------------------------------------- descriptors

def make_desc(n, c_in, c_out, in_size, k, stride=1, pad=0, dil=1, groups=1, *, spatial_dims=2,
              layout="nhwc", wlayout="ohwi", dtype="bf16", pad_end=None) -> Desc:
    """Build a gbconv_desc.  Sizes are ints (1-D), pairs (2-D: height, width) or triples (3-D: depth,
    height, width); an int is used on every axis.  ``pad`` is the padding before each axis, and after
    it too unless ``pad_end`` gives the padding after (begin, end padding)."""
    def pair(v):
        if isinstance(v, (tuple, list)):
            t = [int(e) for e in v][:3]
        else:
            t = [int(v)] * spatial_dims
        return tuple(t + [1] * (3 - len(t)))
    d = Desc()
    d.spatial_dims = spatial_dims
    d.layout = {"nchw": GBCONV_NCHW, "ncl": GBCONV_NCHW, "ncdhw": GBCONV_NCHW, "nhwc": GBCONV_NHWC, "nlc": GBCONV_NHWC,
                "ndhwc": GBCONV_NHWC}[layout]
    d.wlayout = {"oihw": GBCONV_W_OIHW, "oik": GBCONV_W_OIHW, "oidhw": GBCONV_W_OIHW, "ohwi": GBCONV_W_OHWI,
                 "oki": GBCONV_W_OHWI, "odhwi": GBCONV_W_OHWI}[wlayout]
    d.dtype = {"f32": GBCONV_F32, "bf16": GBCONV_BF16}[dtype]
    d.n, d.c_in, d.c_out, d.groups = int(n), int(c_in), int(c_out), int(groups)
    for name, v in (("in_", in_size), ("k", k), ("stride", stride), ("pad", pad), ("dil", dil)):
        t = pair(v)
        for i in range(3):
            getattr(d, name)[i] = t[i]
    if pad_end is not None:
        d.pad_mode = GBCONV_PAD_BEGIN_END
        t = pair(pad_end)
        for i in range(3):
            d.pad_end[i] = t[i]
    return d


_shape_cache = {}


def desc_shapes(d: Desc):
    """(x_shape, w_shape, y_shape) in the layouts the descriptor names (kept per descriptor value)."""
    key = bytes(d)
    hit = _shape_cache.get(key)
    if hit is None:
        if len(_shape_cache) > 4096:
            _shape_cache.clear()
        hit = _shape_cache[key] = _desc_shapes(d)
    return hit


def _desc_shapes(d: Desc):
    out = gbconv_out_shape(d)
    oh, ow = out[0], out[1]
    cpg = d.c_in // d.groups
    if d.spatial_dims == 1:
        L, K = d.in_[0], d.k[0]
        x = (d.n, L, d.c_in) if d.layout == GBCONV_NHWC else (d.n, d.c_in, L)
        y = (d.n, oh, d.c_out) if d.layout == GBCONV_NHWC else (d.n, d.c_out, oh)
        w = (d.c_out, K, cpg) if d.wlayout == GBCONV_W_OHWI else (d.c_out, cpg, K)
        return x, w, y
    if d.spatial_dims == 3:
        sp_in, sp_k, sp_out = tuple(d.in_[:3]), tuple(d.k[:3]), out
    else:
        sp_in, sp_k, sp_out = tuple(d.in_[:2]), tuple(d.k[:2]), (oh, ow)
    nhwc = d.layout == GBCONV_NHWC
    x = (d.n,) + sp_in + (d.c_in,) if nhwc else (d.n, d.c_in) + sp_in
    y = (d.n,) + sp_out + (d.c_out,) if nhwc else (d.n, d.c_out) + sp_out
    w = (d.c_out,) + sp_k + (cpg,) if d.wlayout == GBCONV_W_OHWI else (d.c_out, cpg) + sp_k
    return x, w, y


# ---------------------------------------------------------------- torch helpers

def _torch():
    import torch
    return torch


def _check(t, shape, dtype, name):
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA %s tensor" % (name, dtype))
    return t


def _one_device(**tensors):
    """The one CUDA device every given tensor (None entries skipped) lives on.  The C ABI launches on
    the current device with device pointers, so tensors on different GPUs are refused here and the
    wrappers make this device current for the call."""
    dev = None
    for name, t in tensors.items():
        if t is None:
            continue
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("%s is on %s, but the other tensors are on %s: one call takes one device"
                             % (name, t.device, dev))
    return dev


def _dtype(d: Desc):
    torch = _torch()
    return torch.bfloat16 if d.dtype == GBCONV_BF16 else torch.float32


def _check_host(t, shape, dtype, name):
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    if t.dtype != dtype or t.is_cuda or not t.is_contiguous():
        raise ValueError("%s must be a contiguous host %s tensor" % (name, dtype))
    return t


# Calls on host tensors go to the library's host entry points (gbconv_fwd_host, gbconv_bwd_data_host),
# which pipeline the batch through a device staging buffer in slices: the copy in of slice i+1, the
# kernel of slice i and the copy out of slice i-1 run at the same time.  The staging buffer comes from
# torch's caching allocator; the library allocates nothing.  HOST_SLICES = 0 lets the library choose
# (about 4 MiB of copies per slice).
HOST_SLICES = 0
_staging_cache = {}


class HostCall:
    """A host-buffer call in flight (``conv_fwd_async`` and the like).  ``wait()`` blocks until the
    result is in host memory and returns it; until then the call holds its host tensors and device
    staging buffer, which must not be modified."""

    def __init__(self, result, keep, event):
        self._result, self._keep, self._event = result, keep, event

    def done(self) -> bool:
        return self._event is None or self._event.query()

    def wait(self):
        if self._event is not None:
            self._event.synchronize()
            self._event = self._keep = None
        return self._result

    def __del__(self):
        # the copies still read and write the tensors this object holds
        if getattr(self, "_event", None) is not None:
            try:
                self._event.synchronize()
            except Exception:  # interpreter shutdown: the CUDA context may already be gone
                pass


def _host_call(d: Desc, op: int, src, w, bias, out_shape, out=None, wait=True):
    """One call on host tensors.  Synchronous (wait=True): returns the result as a pinned host tensor
    (or ``out``).  Else returns a HostCall whose completion event the library records.  op
    GBCONV_OP_BWD_DATA with a bias is the transposed convolution."""
    torch = _torch()
    dt = _dtype(d)
    dev = torch.device("cuda", torch.cuda.current_device())
    res = out if out is not None else torch.empty(out_shape, dtype=dt, pin_memory=True)
    _check_host(res, out_shape, dt, "result")
    key = (bytes(d), op, bias is not None)
    nbytes = _staging_cache.get(key)
    if nbytes is None:
        if len(_staging_cache) > 4096:
            _staging_cache.clear()
        nbytes = _staging_cache[key] = gbconv_host_staging_bytes(d, op, bias is not None)
    staging = torch.empty((max(nbytes, 1),), dtype=torch.uint8, device=dev)
    cur = torch.cuda.current_stream(dev)
    event = None
    if not wait:
        event = torch.cuda.Event()
        event.record(cur)  # creates the event; the library records it again at the call's end
    done = None if event is None else event.cuda_event
    stream = cur.cuda_stream
    if op == GBCONV_OP_FWD:
        st = gbconv_fwd_host(d, src.data_ptr(), w.data_ptr(), None if bias is None else bias.data_ptr(),
                             res.data_ptr(), staging.data_ptr(), nbytes, HOST_SLICES, stream, done)
        what = "gbconv_fwd_host"
    elif bias is not None:
        st = gbconv_conv_transpose_host(d, src.data_ptr(), w.data_ptr(), bias.data_ptr(), res.data_ptr(),
                                        staging.data_ptr(), nbytes, HOST_SLICES, stream, done)
        what = "gbconv_conv_transpose_host"
    else:
        st = gbconv_bwd_data_host(d, src.data_ptr(), w.data_ptr(), res.data_ptr(), staging.data_ptr(), nbytes,
                                  HOST_SLICES, stream, done)
        what = "gbconv_bwd_data_host"
    if st != GBCONV_OK:
        if event is not None:
            event.synchronize()  # recorded after whatever was enqueued
        raise GbconvError(st, what)
    if wait:
        return res
    return HostCall(res, (src, w, bias, staging), event)


def _host_args(d: Desc, op: int, src, w, bias):
    """Checks host tensors against the descriptor; returns the result's shape."""
    torch = _torch()
    xs, ws, ys = desc_shapes(d)
    dt = _dtype(d)
    _check_host(src, xs if op == GBCONV_OP_FWD else ys, dt, "x" if op == GBCONV_OP_FWD else "dy")
    _check_host(w, ws, dt, "w")
    if bias is not None:
        _check_host(bias, (d.c_out if op == GBCONV_OP_FWD else d.c_in,), torch.float32, "bias")
    return ys if op == GBCONV_OP_FWD else xs


def conv_fwd_async(d: Desc, x, w, bias=None, y=None) -> HostCall:
    """``conv_fwd`` on host tensors without waiting: the copies and kernels are enqueued and a HostCall
    is returned at once.  Independent calls made this way keep the host link busy back to back (one
    call's last copy out overlaps the next call's copies in); ``wait()`` returns the result."""
    ys = _host_args(d, GBCONV_OP_FWD, x, w, bias)
    return _host_call(d, GBCONV_OP_FWD, x, w, bias, ys, y, wait=False)


def conv_bwd_data_async(d: Desc, dy, w, dx=None) -> HostCall:
    """``conv_bwd_data`` on host tensors without waiting (see ``conv_fwd_async``)."""
    xs = _host_args(d, GBCONV_OP_BWD_DATA, dy, w, None)
    return _host_call(d, GBCONV_OP_BWD_DATA, dy, w, None, xs, dx, wait=False)


def conv_transpose_async(d: Desc, x, w, bias=None, y=None) -> HostCall:
    """``conv_transpose`` on host tensors without waiting (see ``conv_fwd_async``)."""
    xs = _host_args(d, GBCONV_OP_BWD_DATA, x, w, bias)
    return _host_call(d, GBCONV_OP_BWD_DATA, x, w, bias, xs, y, wait=False)


def conv_fwd(d: Desc, x, w, bias=None, y=None):
    """y = conv(x, w) (+ bias) on the current CUDA stream.

    x, w (and y if given) are contiguous CUDA tensors in the descriptor's
    layouts and dtype; bias is a float32 CUDA tensor [C_out] or None.  Host
    (CPU) tensors are copied to the current device first and the result is
    copied back, so the same call serves device-resident and host data (in batch slices whose
    copies overlap the kernels; the result is then a pinned host tensor, or ``y`` if given).
    """
    torch = _torch()
    xs, ws, ys = desc_shapes(d)
    dt = _dtype(d)
    if not x.is_cuda:
        _check_host(x, xs, dt, "x")
        _check_host(w, ws, dt, "w")
        if bias is not None:
            _check_host(bias, (d.c_out,), torch.float32, "bias")
        return _host_call(d, GBCONV_OP_FWD, x, w, bias, ys, y)
    _check(x, xs, dt, "x")
    _check(w, ws, dt, "w")
    if bias is not None:
        _check(bias, (d.c_out,), torch.float32, "bias")
    out = y if y is not None else torch.empty(ys, dtype=dt, device=x.device)
    _check(out, ys, dt, "y")
    dev = _one_device(x=x, w=w, bias=bias, y=out)
    with torch.cuda.device(dev):
        s = gbconv_fwd(d, x.data_ptr(), w.data_ptr(), None if bias is None else bias.data_ptr(), out.data_ptr(),
                       torch.cuda.current_stream(dev).cuda_stream)
    if s != GBCONV_OK:
        raise GbconvError(s, "gbconv_fwd")
    return out


def conv_bwd_data(d: Desc, dy, w, dx=None):
    """Input gradient of the forward convolution ``d`` on the current CUDA stream.

    dy has the forward output's shape, w the forward weight's; the result has
    the forward input's shape (the descriptor fixes it).  Host tensors are
    staged through the device as in ``conv_fwd``.
    """
    torch = _torch()
    xs, ws, ys = desc_shapes(d)
    dt = _dtype(d)
    if not dy.is_cuda:
        _check_host(dy, ys, dt, "dy")
        _check_host(w, ws, dt, "w")
        return _host_call(d, GBCONV_OP_BWD_DATA, dy, w, None, xs, dx)
    _check(dy, ys, dt, "dy")
    _check(w, ws, dt, "w")
    out = dx if dx is not None else torch.empty(xs, dtype=dt, device=dy.device)
    _check(out, xs, dt, "dx")
    dev = _one_device(dy=dy, w=w, dx=out)
    with torch.cuda.device(dev):
        s = gbconv_bwd_data(d, dy.data_ptr(), w.data_ptr(), out.data_ptr(), torch.cuda.current_stream(dev).cuda_stream)
    if s != GBCONV_OK:
        raise GbconvError(s, "gbconv_bwd_data")
    return out


def conv_bwd_filter(d: Desc, x, dy, dw=None, db=None, workspace=None, want_db=False):
    """Weight gradient (and bias gradient) of the forward convolution ``d`` on the current stream.

    x has the forward input's shape, dy the forward output's; returns ``dw`` (the forward weight's
    shape and dtype) when no bias gradient is asked for, else ``(dw, db)`` with db float32 [C_out].
    A bias gradient is asked for by passing ``db`` or ``want_db=True``.  The workspace is a CUDA
    uint8 tensor of at least ``gbconv_bwd_filter_workspace(d)`` bytes; one is allocated (by torch,
    not by the library) when none is given.
    """
    torch = _torch()
    xs, ws_, ys = desc_shapes(d)
    dt = _dtype(d)
    _check(x, xs, dt, "x")
    _check(dy, ys, dt, "dy")
    out = dw if dw is not None else torch.empty(ws_, dtype=dt, device=x.device)
    _check(out, ws_, dt, "dw")
    want_db = want_db or db is not None
    if want_db:
        db = db if db is not None else torch.empty((d.c_out,), dtype=torch.float32, device=x.device)
        _check(db, (d.c_out,), torch.float32, "db")
    dev = _one_device(x=x, dy=dy, dw=out, db=db if want_db else None, workspace=workspace)
    with torch.cuda.device(dev):
        # the workspace size follows the SM count of the device the call runs on
        need = gbconv_bwd_filter_workspace(d)
        if workspace is None:
            workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=dev)
        if workspace.dtype != torch.uint8 or not workspace.is_cuda or workspace.numel() < need:
            raise ValueError("workspace must be a CUDA uint8 tensor of at least %d bytes" % need)
        s = gbconv_bwd_filter(d, x.data_ptr(), dy.data_ptr(), out.data_ptr(), db.data_ptr() if want_db else None,
                              workspace.data_ptr(), workspace.numel(), torch.cuda.current_stream(dev).cuda_stream)
    if s != GBCONV_OK:
        raise GbconvError(s, "gbconv_bwd_filter")
    return (out, db) if want_db else out


def conv_transpose(d: Desc, x, w, bias=None, y=None):
    """Transposed convolution forward: the input gradient of the convolution ``d`` applied to x,
    plus a float32 bias over its C_in output channels, on the current CUDA stream.

    x has d's output shape, w d's weight shape (with OIHW this is the transposed convolution's
    own [C_in_t, C_out_t/G, KH, KW] weight), the result d's input shape.  Host tensors are staged
    through the device as in ``conv_fwd``.
    """
    torch = _torch()
    xs, ws, ys = desc_shapes(d)
    dt = _dtype(d)
    if not x.is_cuda:
        _check_host(x, ys, dt, "x")
        _check_host(w, ws, dt, "w")
        if bias is not None:
            _check_host(bias, (d.c_in,), torch.float32, "bias")
        return _host_call(d, GBCONV_OP_BWD_DATA, x, w, bias, xs, y)
    _check(x, ys, dt, "x")
    _check(w, ws, dt, "w")
    if bias is not None:
        _check(bias, (d.c_in,), torch.float32, "bias")
    out = y if y is not None else torch.empty(xs, dtype=dt, device=x.device)
    _check(out, xs, dt, "y")
    dev = _one_device(x=x, w=w, bias=bias, y=out)
    with torch.cuda.device(dev):
        s = gbconv_conv_transpose(d, x.data_ptr(), w.data_ptr(), None if bias is None else bias.data_ptr(),
                                  out.data_ptr(), torch.cuda.current_stream(dev).cuda_stream)
    if s != GBCONV_OK:
        raise GbconvError(s, "gbconv_conv_transpose")
    return out


def pack_weight(d: Desc, w_oihw):
    """OIHW -> OHWI copy of a weight, on the device ([C_out, C_in/G, K...] -> [C_out, K..., C_in/G] for
    1-D, 2-D and 3-D descriptors)."""
    torch = _torch()
    dt = _dtype(d)
    cpg = d.c_in // d.groups
    k = tuple(int(v) for v in d.k[:d.spatial_dims])
    src_shape, dst_shape = (d.c_out, cpg) + k, (d.c_out,) + k + (cpg,)
    _check(w_oihw, src_shape, dt, "w_oihw")
    out = torch.empty(dst_shape, dtype=dt, device=w_oihw.device)
    with torch.cuda.device(w_oihw.device):
        s = gbconv_pack_weight(d, w_oihw.data_ptr(), out.data_ptr(), torch.cuda.current_stream(w_oihw.device).cuda_stream)
    if s != GBCONV_OK:
        raise GbconvError(s, "gbconv_pack_weight")
    return out


def device_status():
    """Raise if a kernel of this library recorded an expired internal wait."""
    torch = _torch()
    s = gbconv_device_status(torch.cuda.current_stream().cuda_stream)
    if s != GBCONV_OK:
        raise GbconvError(s, "gbconv_device_status")
