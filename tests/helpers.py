"""Test-side glue: descriptors for both sides, tensor transfer, error metrics.

The oracle and the CUDA path each get the convolution shape in their own
vocabulary (``oracle.Conv`` and the C ABI's ``gbconv_desc``); only the seeded
values from ``synth`` are shared.
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import os

import numpy as np

import oracle
import synth

# Parity bars.  FP32 CUDA-core paths: max relative error 1e-5 against the
# dot-product scale.  BF16 tensor-core paths: normwise relative error 2e-2,
# plus a per-element bound derived from the arithmetic: the output is one
# RNE rounding of an fp32 sum, so |gpu - ref| <= 2^-8 |ref| (the bf16 half-ulp
# with margin for a sum that lands near a rounding boundary) + 2^-16 * scale
# (fp32 accumulation over up to a few thousand terms, scale = sum |x*w| + |b|).
F32_REL = 1e-5
BF16_NORMWISE = 2e-2
BF16_ELEM_REL = 2.0 ** -8
BF16_ELEM_SCALE = 2.0 ** -16


def oracle_conv(wl_or_kw) -> oracle.Conv:
    """oracle.Conv from a synth Workload or a dict with the same fields."""
    g = wl_or_kw if isinstance(wl_or_kw, dict) else wl_or_kw.__dict__
    sd = g["spatial_dims"]
    pe = g.get("pad_end")
    if sd == 3:
        return oracle.Conv(n=g["n"], c_in=g["c_in"], c_out=g["c_out"], in_hw=tuple(g["in_size"]), k=tuple(g["k"]),
                           stride=tuple(g["stride"]), pad=tuple(g["pad"]), dil=tuple(g["dil"]), groups=g["groups"],
                           nhwc=g["layout"] in ("nhwc", "ndhwc"), w_ohwi=g["wlayout"] in ("ohwi", "odhwi"),
                           spatial_dims=3, pad_end=None if pe is None else tuple(pe))
    if sd == 1:
        return oracle.Conv(n=g["n"], c_in=g["c_in"], c_out=g["c_out"], in_hw=(1, g["in_size"][0]),
                           k=(1, g["k"][0]), stride=(1, g["stride"][0]), pad=(0, g["pad"][0]),
                           dil=(1, g["dil"][0]), groups=g["groups"], nhwc=g["layout"] in ("nhwc", "nlc"),
                           w_ohwi=g["wlayout"] in ("ohwi", "oki"), spatial_dims=1,
                           pad_end=None if pe is None else (0, pe[0]))
    return oracle.Conv(n=g["n"], c_in=g["c_in"], c_out=g["c_out"], in_hw=tuple(g["in_size"]), k=tuple(g["k"]),
                       stride=tuple(g["stride"]), pad=tuple(g["pad"]), dil=tuple(g["dil"]), groups=g["groups"],
                       nhwc=g["layout"] in ("nhwc", "nlc"), w_ohwi=g["wlayout"] in ("ohwi", "oki"), spatial_dims=2,
                       pad_end=None if pe is None else tuple(pe))


def lib_desc(gb, wl_or_kw):
    """The binding's gbconv_desc for the same shape."""
    g = wl_or_kw if isinstance(wl_or_kw, dict) else wl_or_kw.__dict__
    sd = g["spatial_dims"]
    one = (lambda t: t[0]) if sd == 1 else (lambda t: tuple(t))
    pe = g.get("pad_end")
    return gb.make_desc(g["n"], g["c_in"], g["c_out"], one(g["in_size"]), one(g["k"]), one(g["stride"]),
                        one(g["pad"]), one(g["dil"]), g["groups"], spatial_dims=sd, layout=g["layout"],
                        wlayout=g["wlayout"], dtype=g["dtype"], pad_end=None if pe is None else one(pe))


def shape_kw(**kw):
    """A dict describing one convolution, with defaults."""
    d = dict(spatial_dims=2, n=1, c_in=16, c_out=16, in_size=(8, 8), k=(3, 3), stride=(1, 1), pad=(1, 1),
             dil=(1, 1), groups=1, layout="nhwc", wlayout="ohwi", dtype="bf16", bias=False)
    d.update(kw)
    return d


def draw(c: oracle.Conv, dtype: str, seed: int, op: str = "fwd", bias: bool = False, kind: str = "normal"):
    """Seeded inputs for a shape: dict with float32 values (and bf16 bits for bf16)."""
    out = {}
    src = ("g", c.y_shape()) if op == "dgrad" else ("x", c.x_shape())
    for i, (name, shape) in enumerate([src, ("w", c.w_shape())]):
        if kind == "int":
            lo, hi = (-3, 3) if name != "w" else (-2, 2)
            v = synth.integers(seed * 16 + i, shape, lo, hi)
        else:
            v = synth.normal(seed * 16 + i, shape, 1.0 if name != "w" else 0.25)
        if dtype == "bf16":
            out[name + "_bits"], out[name] = synth.as_bf16(v)
        else:
            out[name] = v.astype(np.float32)
    if bias:
        b = synth.integers(seed * 16 + 7, (c.c_out,), -4, 4) if kind == "int" else synth.normal(seed * 16 + 7, (c.c_out,), 0.5)
        out["b"] = b.astype(np.float32)
    return out


def to_device(torch, arr_f32, bits=None, device="cuda"):
    """Device tensor holding exactly these values (bf16 from bits, else float32)."""
    if bits is not None:
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr_f32, dtype=np.float32)).to(device)


def to_host_f64(torch, t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def scale_fwd(c, x, w, b):
    """Per-output condition scale |b| + sum |x*w| (the oracle run on absolute values)."""
    return oracle.conv_fwd(c, np.abs(x), np.abs(w), None if b is None else np.abs(b))


def scale_dgrad(c, g, w):
    return oracle.conv_dgrad(c, np.abs(g), np.abs(w))


def check_f32(got, ref, scale):
    err = np.abs(got - ref) / np.maximum(scale, 1e-30)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= F32_REL, "fp32 max relative error %.3e > %.1e" % (worst, F32_REL)
    return worst


def check_bf16(got, ref, scale):
    num = float(np.linalg.norm((got - ref).ravel()))
    den = float(np.linalg.norm(ref.ravel()))
    normwise = num / den if den > 0 else num
    assert normwise <= BF16_NORMWISE, "bf16 normwise error %.3e > %.1e" % (normwise, BF16_NORMWISE)
    bound = BF16_ELEM_REL * np.abs(ref) + BF16_ELEM_SCALE * scale + 1e-30
    bad = np.abs(got - ref) > bound
    assert not bad.any(), "%d elements outside the per-element bound, first at %s: got %r ref %r" % (
        int(bad.sum()), np.argwhere(bad)[0], got[bad][0], ref[bad][0])
    return normwise


def bf16_round(a):
    """Exact bf16 RNE rounding of float64 values that are exact in float32."""
    return synth.bf16_to_f32(synth.bf16_bits(np.asarray(a, dtype=np.float32))).astype(np.float64)


# ---------------------------------------------------------------- whole oracle outputs on every host core

def host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _pool_map(fn, items):
    with cf.ThreadPoolExecutor(max_workers=min(len(items), host_threads())) as ex:
        return list(ex.map(fn, items))


def _batch_bounds(n, parts):
    parts = max(1, min(n, parts))
    b = [n * i // parts for i in range(parts + 1)]
    return [(lo, hi) for lo, hi in zip(b[:-1], b[1:]) if hi > lo]


def _points_whole(c, shape, query, parts):
    """Every element of an NC... shaped result by point queries, the flat index range split in parts."""
    total = int(np.prod(shape))
    bounds = [(total * i // parts, total * (i + 1) // parts) for i in range(parts)]

    def run(lohi):
        lo, hi = lohi
        idx = np.stack(np.unravel_index(np.arange(lo, hi, dtype=np.int64), shape), axis=1).astype(np.int64)
        return query(idx)

    return np.concatenate(_pool_map(run, bounds)).reshape(shape)


def oracle_whole(c: oracle.Conv, op: str, a, b, bias=None):
    """The oracle's whole result for ``op`` on the host's cores.

    op 'fwd' (a = x, b = w), 'dgrad' (a = dy, b = w) or 'wgrad' (a = x, b = dy).  Images are
    independent in the forward and input gradient, so 1-D and 2-D shapes split over batch slices
    (each slice one oracle call); the weight gradient is the fp64 sum of its batch slices' weight
    gradients.  3-D shapes have small batches, so they run as point queries over slices of the
    flat output index.  Returns the array in ``c``'s layout (fwd: y, dgrad: dx, wgrad: dw)."""
    t = host_threads()
    if c.spatial_dims == 3:
        parts = 4 * t
        if op == "fwd":
            shape = (c.n, c.c_out) + tuple(c.out_hw())
            r = _points_whole(c, shape, lambda i: oracle.conv_fwd_points(c, a, b, bias, i), parts)
        elif op == "dgrad":
            shape = (c.n, c.c_in) + tuple(c.in_hw)
            r = _points_whole(c, shape, lambda i: oracle.conv_dgrad_points(c, a, b, i), parts)
        else:
            shape = (c.c_out, c.c_in // c.groups) + tuple(c.k)
            r = _points_whole(c, shape, lambda i: oracle.conv_wgrad_points(c, a, b, i), parts)
            return r.transpose(0, 2, 3, 4, 1) if c.w_ohwi else r
        return r.transpose(0, 2, 3, 4, 1) if c.nhwc else r
    slices = _batch_bounds(c.n, t)

    def run(lohi):
        lo, hi = lohi
        cs = dataclasses.replace(c, n=hi - lo)
        if op == "fwd":
            return oracle.conv_fwd(cs, a[lo:hi], b, bias)
        if op == "dgrad":
            return oracle.conv_dgrad(cs, a[lo:hi], b)
        return oracle.conv_wgrad(cs, a[lo:hi], b[lo:hi])

    parts = _pool_map(run, slices)
    if op == "wgrad":
        return np.sum(np.stack(parts), axis=0)
    return np.concatenate(parts, axis=0)
