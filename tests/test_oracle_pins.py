"""Pins for the FP64 oracle, checked against things other than the oracle itself.

Each test ties the oracle to a fact the pages or the mathematics fix:
hand-worked examples (tests/golden), the output-size rule, the 1x1 = matmul
identity, delta kernels, constant-input closed forms, an independent library
convolution (PyTorch CPU, float64), the adjoint identity between forward and
input gradient (and in w, for the weight gradient), scatter == gather, a
one-hot output gradient, and rejection of degenerate shapes.
A plausible slip in the oracle (dropped bias, a flipped kernel, a wrong group
window, a sign or stride error in the gather) fails at least one of them.
"""
import dataclasses
import json
import os

import numpy as np
import pytest

import oracle
import synth
from oracle import Conv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- golden cases

def test_golden_conv1d_dilated_padded():
    g = _golden("conv1d_dilated_padded.json")
    s = g["shape"]
    c = Conv(n=1, c_in=1, c_out=1, in_hw=(1, s["length"]), k=(1, s["k"]), stride=(1, s["stride"]),
             pad=(0, s["pad"]), dil=(1, s["dil"]), spatial_dims=1)
    y = oracle.conv_fwd(c, np.array(g["x"]).reshape(1, 1, 5), np.array(g["w"]).reshape(1, 1, 3), g["bias"])
    assert y.reshape(-1).tolist() == g["y"]


def test_golden_conv2d_grouped_strided():
    g = _golden("conv2d_grouped_strided.json")
    s = g["shape"]
    c = Conv(n=1, c_in=2, c_out=2, in_hw=(3, 3), k=(2, 2), stride=(2, 2), pad=(1, 1), groups=2)
    y = oracle.conv_fwd(c, np.array(g["x_nchw"], dtype=np.float32)[None], np.array(g["w_oihw"]))
    assert y[0].tolist() == g["y_nchw"]


def test_golden_conv1d_dgrad_strided():
    g = _golden("conv1d_dgrad_strided.json")
    c = Conv(n=1, c_in=1, c_out=1, in_hw=(1, 5), k=(1, 3), stride=(1, 2), pad=(0, 1), spatial_dims=1)
    dx = oracle.conv_dgrad(c, np.array(g["dy"]).reshape(1, 1, 3), np.array(g["w"]).reshape(1, 1, 3))
    assert dx.reshape(-1).tolist() == g["dx"]
    dxs = oracle.conv_dgrad(c, np.array(g["dy"]).reshape(1, 1, 3), np.array(g["w"]).reshape(1, 1, 3), scatter=True)
    assert dxs.reshape(-1).tolist() == g["dx"]


# ------------------------------------------------------------ output-size rule

@pytest.mark.parametrize("in_,k,s,p,d,expect", [
    (32, 3, 1, 2, 2, 32),     # conv1d NCL fp32 workload: eff 5, (32+4-5)/1+1
    (56, 1, 1, 0, 1, 56),     # pointwise 1x1
    (56, 3, 1, 1, 1, 56),     # dense 3x3 pad 1
    (112, 3, 2, 1, 1, 56),    # depthwise 3x3 stride 2: (112+2-3)//2+1
    (64, 3, 2, 1, 1, 32),     # dgrad forward shape
    (63, 3, 2, 1, 1, 32),     # ... and a different input giving the same output
    (5, 5, 1, 0, 1, 1),       # kernel exactly fills the input
    (4, 3, 1, 0, 2, None),    # eff 5 > 4: rejected
    (1, 3, 1, 1, 1, 1),       # padding makes it fit
    (7, 3, 3, 0, 1, 2),       # floor: last input position never read
    (10, 4, 3, 2, 3, 2),      # eff 10, (10+4-10)//3+1 = 2
    (0, 1, 1, 0, 1, None),
    (8, 0, 1, 0, 1, None),
    (8, 3, 0, 0, 1, None),
    (8, 3, 1, 0, 0, None),
])
def test_out_size_table(in_, k, s, p, d, expect):
    assert oracle.out_size(in_, k, s, p, d) == expect


# --------------------------------------------------------- 1x1 conv == matmul

@pytest.mark.parametrize("nhwc", [True, False])
def test_pointwise_is_matmul(nhwc):
    n, h, w, ci, co = 2, 5, 3, 12, 7
    c = Conv(n=n, c_in=ci, c_out=co, in_hw=(h, w), k=(1, 1), nhwc=nhwc, w_ohwi=True)
    x = synth.normal(11, c.x_shape()).astype(np.float32)
    wt = synth.normal(12, c.w_shape()).astype(np.float32)
    y = oracle.conv_fwd(c, x, wt)
    xm = x.astype(np.float64)
    if not nhwc:
        xm = xm.transpose(0, 2, 3, 1)
    ref = xm.reshape(-1, ci) @ wt.astype(np.float64).reshape(co, ci).T
    got = y if nhwc else y.transpose(0, 2, 3, 1)
    np.testing.assert_allclose(got.reshape(-1, co), ref, rtol=1e-12, atol=1e-12)
    # data gradient of the same 1x1: dy[M, C_out] @ W[C_out, C_in]
    dy = synth.normal(13, c.y_shape()).astype(np.float32)
    dx = oracle.conv_dgrad(c, dy, wt)
    dym = dy.astype(np.float64) if nhwc else dy.astype(np.float64).transpose(0, 2, 3, 1)
    refdx = dym.reshape(-1, co) @ wt.astype(np.float64).reshape(co, ci)
    gotdx = dx if nhwc else dx.transpose(0, 2, 3, 1)
    np.testing.assert_allclose(gotdx.reshape(-1, ci), refdx, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- delta kernels

@pytest.mark.parametrize("k,d", [(3, 1), (5, 1), (3, 2), (3, 3)])
@pytest.mark.parametrize("nhwc", [False, True])
def test_delta_kernel_reproduces_input(k, d, nhwc):
    ch, kc = 4, (k - 1) // 2
    c = Conv(n=2, c_in=ch, c_out=ch, in_hw=(6, 7), k=(k, k), pad=(d * kc, d * kc), dil=(d, d), nhwc=nhwc)
    w = np.zeros(c.w_shape())
    for i in range(ch):
        w[i, i, kc, kc] = 1.0
    x = synth.normal(21, c.x_shape())
    y = oracle.conv_fwd(c, x, w)
    np.testing.assert_array_equal(y, x.astype(np.float32).astype(np.float64))


def test_delta_kernel_depthwise():
    ch = 5
    c = Conv(n=1, c_in=ch, c_out=ch, in_hw=(4, 9), k=(3, 3), pad=(1, 1), groups=ch)
    w = np.zeros(c.w_shape())
    w[:, 0, 1, 1] = 1.0
    x = synth.normal(22, c.x_shape())
    np.testing.assert_array_equal(oracle.conv_fwd(c, x, w), x.astype(np.float32).astype(np.float64))


@pytest.mark.parametrize("k0,s,p,d", [(0, 1, 2, 2), (2, 1, 2, 2), (1, 2, 1, 3), (2, 3, 0, 2)])
def test_delta_tap_1d_shift(k0, s, p, d):
    L, K = 13, 3
    c = Conv(n=1, c_in=1, c_out=1, in_hw=(1, L), k=(1, K), stride=(1, s), pad=(0, p), dil=(1, d), spatial_dims=1)
    w = np.zeros((1, 1, K))
    w[0, 0, k0] = 1.0
    x = np.arange(1, L + 1, dtype=np.float64).reshape(1, 1, L)
    y = oracle.conv_fwd(c, x, w).reshape(-1)
    lout = oracle.out_size(L, K, s, p, d)
    for l in range(lout):
        src = l * s + k0 * d - p
        assert y[l] == (src + 1 if 0 <= src < L else 0.0)


# ---------------------------------------------------- closed form, constants

def test_constant_input_border_counts():
    # x = 1, w = 1, 3x3 pad 1 stride 1: each output is bias + (C_in/G) * (taps inside the image):
    # 4 at corners, 6 on edges, 9 inside.
    g, ci, co = 2, 6, 4
    c = Conv(n=1, c_in=ci, c_out=co, in_hw=(5, 6), k=(3, 3), pad=(1, 1), groups=g, nhwc=True, w_ohwi=True)
    b = np.array([0.25, -1.0, 2.0, 0.0])
    y = oracle.conv_fwd(c, np.ones(c.x_shape()), np.ones(c.w_shape()), b)
    cpg = ci // g
    taps = np.full((5, 6), 9.0)
    taps[0, :] = taps[-1, :] = 6.0
    taps[:, 0] = taps[:, -1] = 6.0
    taps[0, 0] = taps[0, -1] = taps[-1, 0] = taps[-1, -1] = 4.0
    for o in range(co):
        np.testing.assert_array_equal(y[0, :, :, o], b[o] + cpg * taps)


# ------------------------------------------- independent library convolution

torch = pytest.importorskip("torch")


def _to_nchw(a, c):
    return a.transpose(0, 3, 1, 2) if (c.nhwc and c.spatial_dims == 2) else (
        a.transpose(0, 2, 1) if (c.nhwc and c.spatial_dims == 1) else a)


def _w_to_oihw(w, c):
    if not c.w_ohwi:
        return w
    return w.transpose(0, 3, 1, 2) if c.spatial_dims == 2 else w.transpose(0, 2, 1)


CASES = [
    Conv(n=2, c_in=4, c_out=8, in_hw=(1, 32), k=(1, 3), stride=(1, 1), pad=(0, 2), dil=(1, 2), spatial_dims=1),
    Conv(n=1, c_in=6, c_out=4, in_hw=(1, 17), k=(1, 4), stride=(1, 3), pad=(0, 1), dil=(1, 2), groups=2,
         spatial_dims=1, nhwc=True, w_ohwi=True),
    Conv(n=2, c_in=6, c_out=9, in_hw=(7, 9), k=(3, 2), stride=(2, 1), pad=(1, 0), dil=(1, 2), groups=3),
    Conv(n=1, c_in=8, c_out=8, in_hw=(9, 8), k=(3, 3), stride=(2, 2), pad=(1, 1), groups=8, nhwc=True, w_ohwi=True),
    Conv(n=2, c_in=4, c_out=6, in_hw=(6, 5), k=(5, 3), stride=(1, 2), pad=(2, 1), dil=(1, 1), nhwc=True),
    Conv(n=1, c_in=3, c_out=2, in_hw=(10, 10), k=(3, 3), stride=(3, 3), pad=(0, 0), dil=(2, 2), w_ohwi=True),
]


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_matches_torch_float64(ci):
    c = CASES[ci]
    F = torch.nn.functional
    x = synth.normal(31 + ci, c.x_shape()).astype(np.float32)
    w = synth.normal(41 + ci, c.w_shape()).astype(np.float32)
    b = synth.normal(51 + ci, (c.c_out,)).astype(np.float32)
    xt = torch.from_numpy(_to_nchw(x, c).astype(np.float64).copy())
    wt = torch.from_numpy(_w_to_oihw(w, c).astype(np.float64).copy())
    bt = torch.from_numpy(b.astype(np.float64))
    if c.spatial_dims == 1:
        ref = F.conv1d(xt, wt, bt, stride=c.stride[1], padding=c.pad[1], dilation=c.dil[1], groups=c.groups)
    else:
        ref = F.conv2d(xt, wt, bt, stride=c.stride, padding=c.pad, dilation=c.dil, groups=c.groups)
    y = oracle.conv_fwd(c, x, w, b)
    np.testing.assert_allclose(_to_nchw(y, c), ref.numpy(), rtol=1e-12, atol=1e-12)
    # input gradient against torch's own backward-data routine
    dy = synth.normal(61 + ci, c.y_shape()).astype(np.float32)
    dyt = torch.from_numpy(_to_nchw(dy, c).astype(np.float64).copy())
    if c.spatial_dims == 1:
        refdx = torch.nn.grad.conv1d_input(xt.shape, wt, dyt, stride=c.stride[1], padding=c.pad[1],
                                           dilation=c.dil[1], groups=c.groups)
    else:
        refdx = torch.nn.grad.conv2d_input(xt.shape, wt, dyt, stride=c.stride, padding=c.pad,
                                           dilation=c.dil, groups=c.groups)
    dx = oracle.conv_dgrad(c, dy, w)
    np.testing.assert_allclose(_to_nchw(dx, c), refdx.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_conv_transpose_matches_torch_float64(ci):
    # The transposed convolution of the forward c: torch's conv_transpose with c's weight as its
    # [C_in_t = C_out, C_out_t / G, KH, KW] weight, and the output_padding that lands on c's input
    # extent (the trailing positions no stride reaches).
    c = CASES[ci]
    F = torch.nn.functional
    x = synth.normal(91 + ci, c.y_shape()).astype(np.float32)
    w = synth.normal(92 + ci, c.w_shape()).astype(np.float32)
    b = synth.normal(93 + ci, (c.c_in,)).astype(np.float32)
    xt = torch.from_numpy(_to_nchw(x, c).astype(np.float64).copy())
    wt = torch.from_numpy(_w_to_oihw(w, c).astype(np.float64).copy())
    bt = torch.from_numpy(b.astype(np.float64))
    oh, ow = c.out_hw()
    def opad(axis, o):
        return c.in_hw[axis] - ((o - 1) * c.stride[axis] - 2 * c.pad[axis] + c.dil[axis] * (c.k[axis] - 1) + 1)
    if c.spatial_dims == 1:
        ref = F.conv_transpose1d(xt, wt, bt, stride=c.stride[1], padding=c.pad[1], output_padding=opad(1, ow),
                                 groups=c.groups, dilation=c.dil[1])
    else:
        ref = F.conv_transpose2d(xt, wt, bt, stride=c.stride, padding=c.pad, output_padding=(opad(0, oh), opad(1, ow)),
                                 groups=c.groups, dilation=c.dil)
    y = oracle.conv_transpose(c, x, w, b)
    np.testing.assert_allclose(_to_nchw(y, c), ref.numpy(), rtol=1e-12, atol=1e-12)


# --------------------------------------------- adjoint and scatter == gather

@pytest.mark.parametrize("ci", range(len(CASES)))
def test_adjoint_identity(ci):
    # <conv(x, w), dy> == <x, dgrad(dy, w)> for the bias-free convolution
    c = CASES[ci]
    x = synth.normal(71 + ci, c.x_shape())
    w = synth.normal(72 + ci, c.w_shape())
    dy = synth.normal(73 + ci, c.y_shape())
    lhs = float(np.sum(oracle.conv_fwd(c, x, w) * dy.astype(np.float32)))
    rhs = float(np.sum(x.astype(np.float32).astype(np.float64) * oracle.conv_dgrad(c, dy, w)))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs)) * 10


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_scatter_equals_gather(ci):
    c = CASES[ci]
    dy = synth.normal(81 + ci, c.y_shape())
    w = synth.normal(82 + ci, c.w_shape())
    np.testing.assert_allclose(oracle.conv_dgrad(c, dy, w), oracle.conv_dgrad(c, dy, w, scatter=True),
                               rtol=1e-12, atol=1e-12)


def test_unreached_input_has_zero_gradient():
    # in=7, k=3, s=3, p=0: out=2 reads positions 0..5; position 6 gets no gradient.
    c = Conv(n=1, c_in=2, c_out=3, in_hw=(1, 7), k=(1, 3), stride=(1, 3), spatial_dims=1)
    dx = oracle.conv_dgrad(c, synth.normal(91, c.y_shape()), synth.normal(92, c.w_shape()))
    assert np.all(dx[:, :, 6] == 0.0) and np.all(dx[:, :, :6] != 0.0)


# ------------------------------------------------------- degenerate rejection

@pytest.mark.parametrize("kw", [
    dict(n=0), dict(c_in=0), dict(c_out=0), dict(groups=0), dict(groups=3),
    dict(stride=(0, 1)), dict(dil=(1, 0)), dict(k=(9, 3)), dict(in_hw=(0, 5)),
])
def test_degenerate_shapes_rejected(kw):
    base = dict(n=1, c_in=4, c_out=4, in_hw=(6, 5), k=(3, 3), stride=(1, 1), pad=(1, 1), dil=(1, 1), groups=2)
    base.update(kw)
    c = Conv(**base)
    assert not oracle.check(c)


# ------------------------------------------------------- weight and bias gradients

@pytest.mark.parametrize("ci", range(len(CASES)))
def test_wgrad_matches_torch_float64(ci):
    # torch's own weight-gradient routine, in float64, on the NCHW / OIHW view of the same case
    c = CASES[ci]
    x = synth.normal(101 + ci, c.x_shape()).astype(np.float32)
    dy = synth.normal(102 + ci, c.y_shape()).astype(np.float32)
    xt = torch.from_numpy(_to_nchw(x, c).astype(np.float64).copy())
    dyt = torch.from_numpy(_to_nchw(dy, c).astype(np.float64).copy())
    w_oihw_shape = (c.c_out, c.c_in // c.groups) + ((c.k[1],) if c.spatial_dims == 1 else tuple(c.k))
    if c.spatial_dims == 1:
        ref = torch.nn.grad.conv1d_weight(xt, w_oihw_shape, dyt, stride=c.stride[1], padding=c.pad[1],
                                          dilation=c.dil[1], groups=c.groups)
    else:
        ref = torch.nn.grad.conv2d_weight(xt, w_oihw_shape, dyt, stride=c.stride, padding=c.pad,
                                          dilation=c.dil, groups=c.groups)
    dw = oracle.conv_wgrad(c, x, dy)
    np.testing.assert_allclose(_w_to_oihw(dw, c), ref.numpy(), rtol=1e-12, atol=1e-12)
    axes = tuple(a for a in range(dyt.ndim) if a != 1)
    np.testing.assert_allclose(oracle.conv_bgrad(c, dy), dyt.sum(dim=axes).numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_wgrad_adjoint_identity(ci):
    # The forward is linear in w: <conv(x, w), dy> == <w, wgrad(x, dy)>
    c = CASES[ci]
    x = synth.normal(111 + ci, c.x_shape())
    w = synth.normal(112 + ci, c.w_shape())
    dy = synth.normal(113 + ci, c.y_shape())
    lhs = float(np.sum(oracle.conv_fwd(c, x, w) * dy.astype(np.float32)))
    rhs = float(np.sum(w.astype(np.float32).astype(np.float64) * oracle.conv_wgrad(c, x, dy)))
    assert abs(lhs - rhs) <= 1e-11 * max(1.0, abs(lhs))


@pytest.mark.parametrize("nhwc", [False, True])
def test_pointwise_wgrad_is_matmul(nhwc):
    # 1x1, stride 1, no padding: dW[co, ci] = sum over pixels m of dy[m, co] * x[m, ci]
    c = Conv(n=2, c_in=5, c_out=3, in_hw=(4, 3), k=(1, 1), nhwc=nhwc, w_ohwi=nhwc)
    x = synth.normal(121, c.x_shape())
    dy = synth.normal(122, c.y_shape())
    X = x if nhwc else x.transpose(0, 2, 3, 1)
    G = dy if nhwc else dy.transpose(0, 2, 3, 1)
    X = X.astype(np.float32).astype(np.float64).reshape(-1, c.c_in)
    G = G.astype(np.float32).astype(np.float64).reshape(-1, c.c_out)
    ref = np.zeros((c.c_out, c.c_in))
    for m in range(X.shape[0]):
        for co in range(c.c_out):
            for ci_ in range(c.c_in):
                ref[co, ci_] += G[m, co] * X[m, ci_]
    np.testing.assert_allclose(oracle.conv_wgrad(c, x, dy).reshape(c.c_out, c.c_in), ref, rtol=1e-12, atol=1e-12)


def test_wgrad_constant_counts():
    # x = 1, dy = 1: dW[co, cl, kh, kw] = N * (output rows whose tap kh lands in the image) *
    # (output columns whose tap kw lands in the image); db[co] = N * OH * OW.
    c = Conv(n=3, c_in=4, c_out=6, in_hw=(7, 6), k=(3, 2), stride=(2, 1), pad=(1, 1), dil=(1, 2), groups=2,
             nhwc=True, w_ohwi=True)
    oh_n, ow_n = c.out_hw()
    dw = oracle.conv_wgrad(c, np.ones(c.x_shape()), np.ones(c.y_shape()))
    for kh in range(3):
        rows = sum(1 for oh in range(oh_n) if 0 <= oh * 2 + kh * 1 - 1 < 7)
        for kw in range(2):
            cols = sum(1 for ow in range(ow_n) if 0 <= ow * 1 + kw * 2 - 1 < 6)
            np.testing.assert_array_equal(dw[:, kh, kw, :], 3.0 * rows * cols)
    np.testing.assert_array_equal(oracle.conv_bgrad(c, np.ones(c.y_shape())), 3.0 * oh_n * ow_n)


def test_wgrad_of_one_hot_output_gradient_is_the_input_patch():
    # dy = 1 at (n0, co0, oh0, ow0) only: dW[co0, cl, kh, kw] is the input element the forward read
    # for that output with that weight (zero outside the image); every other output channel is 0.
    c = Conv(n=2, c_in=6, c_out=4, in_hw=(6, 7), k=(3, 3), stride=(2, 1), pad=(1, 2), dil=(1, 2), groups=2)
    x = synth.normal(131, c.x_shape()).astype(np.float32)
    n0, co0, oh0, ow0 = 1, 3, 2, 4
    dy = np.zeros(c.y_shape())
    dy[n0, co0, oh0, ow0] = 1.0
    dw = oracle.conv_wgrad(c, x, dy)
    g = co0 // (c.c_out // c.groups)
    cpg = c.c_in // c.groups
    for cl in range(cpg):
        for kh in range(3):
            for kw in range(3):
                ih, iw = oh0 * 2 + kh - 1, ow0 + kw * 2 - 2
                want = x[n0, g * cpg + cl, ih, iw] if (0 <= ih < 6 and 0 <= iw < 7) else 0.0
                assert dw[co0, cl, kh, kw] == want
    assert np.all(np.delete(dw, co0, axis=0) == 0.0)


# ------------------------------------------------------- (begin, end) padding

ASYM = [
    Conv(n=2, c_in=4, c_out=6, in_hw=(7, 8), k=(3, 3), stride=(2, 2), pad=(0, 1), pad_end=(1, 0), groups=2),
    Conv(n=1, c_in=3, c_out=5, in_hw=(1, 13), k=(1, 4), stride=(1, 3), pad=(0, 2), pad_end=(0, 0), dil=(1, 2),
         spatial_dims=1, nhwc=True, w_ohwi=True),
    Conv(n=2, c_in=5, c_out=4, in_hw=(6, 9), k=(2, 3), stride=(1, 1), pad=(1, 0), pad_end=(0, 2), nhwc=True),
    Conv(n=1, c_in=2, c_out=3, in_hw=(5, 5), k=(1, 1), stride=(1, 1), pad=(0, 0), pad_end=(1, 2), w_ohwi=True),
]


@pytest.mark.parametrize("in_,k,s,pb,pe,d,expect", [
    (7, 3, 2, 0, 1, 1, 3), (8, 3, 2, 0, 1, 1, 4), (8, 3, 2, 1, 0, 1, 4), (8, 3, 2, 0, 0, 1, 3),
    (5, 1, 1, 0, 2, 1, 7), (13, 4, 3, 2, 0, 2, 3), (4, 5, 1, 0, 0, 1, None), (4, 5, 1, 0, 1, 1, 1),
    (4, 5, 1, 1, 1, 1, 2), (5, 3, 1, 0, -1, 1, None),
])
def test_out_size_begin_end(in_, k, s, pb, pe, d, expect):
    # (in + begin + end - (k-1)*d - 1) // s + 1, and rejected when the padded input is shorter
    # than the effective kernel
    assert oracle.out_size2(in_, k, s, pb, pe, d) == expect


@pytest.mark.parametrize("ci", range(len(ASYM)))
def test_begin_end_padding_matches_torch_float64(ci):
    # torch on an explicitly zero-padded input (F.pad), convolution without padding; the input,
    # weight and bias gradients by autograd through the same graph
    c = ASYM[ci]
    F = torch.nn.functional
    x = synth.normal(141 + ci, c.x_shape()).astype(np.float32)
    w = synth.normal(142 + ci, c.w_shape()).astype(np.float32)
    b = synth.normal(143 + ci, (c.c_out,)).astype(np.float32)
    dy = synth.normal(144 + ci, c.y_shape()).astype(np.float32)
    xt = torch.from_numpy(_to_nchw(x, c).astype(np.float64).copy()).requires_grad_(True)
    wt = torch.from_numpy(_w_to_oihw(w, c).astype(np.float64).copy()).requires_grad_(True)
    bt = torch.from_numpy(b.astype(np.float64)).requires_grad_(True)
    pe = c.pads_end()
    if c.spatial_dims == 1:
        yt = F.conv1d(F.pad(xt, (c.pad[1], pe[1])), wt, bt, stride=c.stride[1], dilation=c.dil[1], groups=c.groups)
    else:
        yt = F.conv2d(F.pad(xt, (c.pad[1], pe[1], c.pad[0], pe[0])), wt, bt, stride=c.stride, dilation=c.dil,
                      groups=c.groups)
    np.testing.assert_allclose(_to_nchw(oracle.conv_fwd(c, x, w, b), c), yt.detach().numpy(), rtol=1e-12, atol=1e-12)
    dyt = torch.from_numpy(_to_nchw(dy, c).astype(np.float64).copy())
    gx, gw, gb_ = torch.autograd.grad(yt, (xt, wt, bt), dyt)
    np.testing.assert_allclose(_to_nchw(oracle.conv_dgrad(c, dy, w), c), gx.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(_w_to_oihw(oracle.conv_wgrad(c, x, dy), c), gw.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.conv_bgrad(c, dy), gb_.numpy(), rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------- 3-D convolution

CASES3 = [
    Conv(n=2, c_in=4, c_out=6, in_hw=(5, 6, 7), k=(3, 3, 3), stride=(1, 2, 1), pad=(1, 1, 0), dil=(1, 1, 2),
         groups=2, spatial_dims=3),
    Conv(n=1, c_in=3, c_out=4, in_hw=(4, 5, 6), k=(2, 3, 1), stride=(2, 1, 1), pad=(0, 1, 0), pad_end=(1, 0, 2),
         spatial_dims=3, nhwc=True, w_ohwi=True),
    Conv(n=2, c_in=6, c_out=6, in_hw=(3, 4, 5), k=(3, 3, 3), stride=(1, 1, 1), pad=(1, 1, 1), groups=6,
         spatial_dims=3, nhwc=True),
]


def _to_ncdhw(a, c):
    return a.transpose(0, 4, 1, 2, 3) if c.nhwc else a


def _w_to_oidhw(w, c):
    return w.transpose(0, 4, 1, 2, 3) if c.w_ohwi else w


@pytest.mark.parametrize("ci", range(len(CASES3)))
def test_conv3d_matches_torch_float64(ci):
    # torch conv3d on the explicitly padded input, and its autograd input, weight and bias gradients
    c = CASES3[ci]
    F = torch.nn.functional
    x = synth.normal(151 + ci, c.x_shape()).astype(np.float32)
    w = synth.normal(152 + ci, c.w_shape()).astype(np.float32)
    b = synth.normal(153 + ci, (c.c_out,)).astype(np.float32)
    dy = synth.normal(154 + ci, c.y_shape()).astype(np.float32)
    xt = torch.from_numpy(_to_ncdhw(x, c).astype(np.float64).copy()).requires_grad_(True)
    wt = torch.from_numpy(_w_to_oidhw(w, c).astype(np.float64).copy()).requires_grad_(True)
    bt = torch.from_numpy(b.astype(np.float64)).requires_grad_(True)
    pad, pe = c._full(c.pad, 0), c._full(c.pads_end(), 0)
    xp = F.pad(xt, (pad[2], pe[2], pad[1], pe[1], pad[0], pe[0]))
    yt = F.conv3d(xp, wt, bt, stride=c._full(c.stride, 1), dilation=c._full(c.dil, 1), groups=c.groups)
    np.testing.assert_allclose(_to_ncdhw(oracle.conv_fwd(c, x, w, b), c), yt.detach().numpy(), rtol=1e-12, atol=1e-12)
    dyt = torch.from_numpy(_to_ncdhw(dy, c).astype(np.float64).copy())
    gx, gw, gb_ = torch.autograd.grad(yt, (xt, wt, bt), dyt)
    np.testing.assert_allclose(_to_ncdhw(oracle.conv_dgrad(c, dy, w), c), gx.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(_to_ncdhw(oracle.conv_dgrad(c, dy, w, scatter=True), c), gx.numpy(),
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(_w_to_oidhw(oracle.conv_wgrad(c, x, dy), c), gw.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.conv_bgrad(c, dy), gb_.numpy(), rtol=1e-12, atol=1e-12)
    # the point queries the full-size checks use, at every third (n, c, d, h, w) element
    yi = np.argwhere(np.ones(yt.shape, dtype=bool))[::3]
    np.testing.assert_allclose(oracle.conv_fwd_points(c, x, w, b, yi), yt.detach().numpy()[tuple(yi.T)],
                               rtol=1e-12, atol=1e-12)
    xi = np.argwhere(np.ones(gx.shape, dtype=bool))[::3]
    np.testing.assert_allclose(oracle.conv_dgrad_points(c, dy, w, xi), gx.numpy()[tuple(xi.T)], rtol=1e-12,
                               atol=1e-12)
    wi = np.argwhere(np.ones(gw.shape, dtype=bool))[::3]  # (co, c_local, kd, kh, kw) of the OIDHW gradient
    np.testing.assert_allclose(oracle.conv_wgrad_points(c, x, dy, wi), gw.numpy()[tuple(wi.T)], rtol=1e-12,
                               atol=1e-12)


def test_conv3d_with_unit_depth_is_conv2d():
    # depth 1, kernel depth 1: the 3-D sums are the 2-D ones
    c2 = Conv(n=2, c_in=4, c_out=6, in_hw=(6, 7), k=(3, 2), stride=(2, 1), pad=(1, 0), dil=(1, 2), groups=2, nhwc=True,
              w_ohwi=True)
    c3 = Conv(n=2, c_in=4, c_out=6, in_hw=(1, 6, 7), k=(1, 3, 2), stride=(1, 2, 1), pad=(0, 1, 0), dil=(1, 1, 2),
              groups=2, nhwc=True, w_ohwi=True, spatial_dims=3)
    x = synth.normal(161, c2.x_shape()).astype(np.float32)
    w = synth.normal(162, c2.w_shape()).astype(np.float32)
    dy = synth.normal(163, c2.y_shape()).astype(np.float32)
    x3, w3, dy3 = x.reshape(c3.x_shape()), w.reshape(c3.w_shape()), dy.reshape(c3.y_shape())
    np.testing.assert_array_equal(oracle.conv_fwd(c3, x3, w3).reshape(c2.y_shape()), oracle.conv_fwd(c2, x, w))
    np.testing.assert_array_equal(oracle.conv_dgrad(c3, dy3, w3).reshape(c2.x_shape()), oracle.conv_dgrad(c2, dy, w))
    np.testing.assert_array_equal(oracle.conv_wgrad(c3, x3, dy3).reshape(c2.w_shape()), oracle.conv_wgrad(c2, x, dy))


# ------------------------------------------------- 2-D and 1-D point queries

def _torch_fwd_and_grads(c, x, w, b, dy):
    """torch float64 forward on the explicitly padded NCHW / NCL view, and its autograd input, weight
    and bias gradients (all in the NCHW / OIHW view)."""
    F = torch.nn.functional
    xt = torch.from_numpy(_to_nchw(x, c).astype(np.float64).copy()).requires_grad_(True)
    wt = torch.from_numpy(_w_to_oihw(w, c).astype(np.float64).copy()).requires_grad_(True)
    bt = torch.from_numpy(b.astype(np.float64)).requires_grad_(True)
    pe = c.pads_end()
    if c.spatial_dims == 1:
        yt = F.conv1d(F.pad(xt, (c.pad[1], pe[1])), wt, bt, stride=c.stride[1], dilation=c.dil[1], groups=c.groups)
    else:
        yt = F.conv2d(F.pad(xt, (c.pad[1], pe[1], c.pad[0], pe[0])), wt, bt, stride=c.stride, dilation=c.dil,
                      groups=c.groups)
    dyt = torch.from_numpy(_to_nchw(dy, c).astype(np.float64).copy())
    gx, gw, _ = torch.autograd.grad(yt, (xt, wt, bt), dyt)
    return yt.detach().numpy(), gx.numpy(), gw.numpy()


def _as4(idx, c):
    """Indices of an NCL / OIK tensor as the 4-index (n, c, 0, l) / (co, cl, 0, k) form the 2-D point
    queries take; 2-D indices unchanged."""
    if c.spatial_dims == 1:
        return np.stack([idx[:, 0], idx[:, 1], np.zeros_like(idx[:, 0]), idx[:, 2]], axis=1)
    return idx


@pytest.mark.parametrize("ci", range(len(CASES) + len(ASYM)))
def test_points_2d_match_torch_float64(ci):
    # The batched 4-index point queries (forward, input gradient, weight gradient) that the full-size
    # checks of 2-D workloads use, against torch at every third element: grouped, strided, dilated,
    # symmetric and (begin, end) padded, both activation layouts and both weight orders, 1-D and 2-D.
    # Indices are (n, c, h, w) of the NCHW view and (co, c_local, kh, kw) of the OIHW view whatever
    # the layout, so a swapped index order or layout slip fails here.
    c = (CASES + ASYM)[ci]
    x = synth.normal(171 + ci, c.x_shape()).astype(np.float32)
    w = synth.normal(172 + ci, c.w_shape()).astype(np.float32)
    b = synth.normal(173 + ci, (c.c_out,)).astype(np.float32)
    dy = synth.normal(174 + ci, c.y_shape()).astype(np.float32)
    y_ref, gx_ref, gw_ref = _torch_fwd_and_grads(c, x, w, b, dy)
    for ref, query in ((y_ref, lambda i: oracle.conv_fwd_points(c, x, w, b, i)),
                       (gx_ref, lambda i: oracle.conv_dgrad_points(c, dy, w, i)),
                       (gw_ref, lambda i: oracle.conv_wgrad_points(c, x, dy, i))):
        idx = np.argwhere(np.ones(ref.shape, dtype=bool))[ci % 3::3]
        np.testing.assert_allclose(query(_as4(idx, c)), ref[tuple(idx.T)], rtol=1e-12, atol=1e-12)
    # and without a bias the forward points are the bias-free sums
    idx = np.argwhere(np.ones(y_ref.shape, dtype=bool))[::5]
    got = oracle.conv_fwd_points(c, x, w, None, _as4(idx, c))
    bias_at = b.astype(np.float64)[idx[:, 1]]
    np.testing.assert_allclose(got, y_ref[tuple(idx.T)] - bias_at, rtol=1e-12, atol=1e-12)


# ------------------------------------------- the tests' whole-output oracle on many cores

@pytest.mark.parametrize("ci", range(len(CASES) + len(CASES3)))
def test_whole_on_host_threads_equals_one_call(ci):
    # the full-size parity tests split the oracle over batch slices (1-D / 2-D) or flat index ranges
    # of point queries (3-D) on every host core; the pieces must put back the one-call result
    from tests.helpers import oracle_whole
    c = (CASES + CASES3)[ci]
    c = dataclasses.replace(c, n=3)
    x = synth.normal(181 + ci, c.x_shape()).astype(np.float32)
    w = synth.normal(182 + ci, c.w_shape()).astype(np.float32)
    b = synth.normal(183 + ci, (c.c_out,)).astype(np.float32)
    dy = synth.normal(184 + ci, c.y_shape()).astype(np.float32)
    np.testing.assert_allclose(oracle_whole(c, "fwd", x, w, b), oracle.conv_fwd(c, x, w, b), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(oracle_whole(c, "dgrad", dy, w), oracle.conv_dgrad(c, dy, w), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(oracle_whole(c, "wgrad", x, dy), oracle.conv_wgrad(c, x, dy), rtol=1e-13, atol=1e-13)
