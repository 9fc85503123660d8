"""The benchmark workloads: tensor shapes and value recipes, nothing else.

Shapes are stated explicitly (including the output-gradient shape of the dgrad
workload, which its description gives); no convolution arithmetic lives here.
Values come from ``synth`` with seed ``1000 + index`` unless a caller passes
another seed; bf16 workloads round the drawn values to bf16 (RNE) and hand the
same bits to the GPU and the oracle.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import as_bf16, normal, uniform


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    op: str                 # "fwd", "dgrad" or "wgrad"
    dtype: str              # "f32" or "bf16"
    spatial_dims: int
    layout: str             # "ncl" / "nhwc" / "ndhwc"
    wlayout: str            # "oik" / "ohwi" / "odhwi"
    n: int
    c_in: int
    c_out: int
    in_size: tuple          # (L,), (H, W) or (D, H, W)
    k: tuple
    stride: tuple
    pad: tuple
    dil: tuple
    groups: int
    bias: bool
    x_shape: tuple          # forward input (fwd) -- or dx shape (dgrad)
    w_shape: tuple
    g_shape: tuple          # output gradient shape (dgrad and wgrad)
    recipe: dict = field(default_factory=dict)
    describe: str = ""


WORKLOADS = [
    Workload("conv1d_ncl_f32", 0, "fwd", "f32", 1, "ncl", "oik", 2, 4, 8, (32,), (3,), (1,), (2,), (2,), 1, True,
             (2, 4, 32), (8, 4, 3), (),
             {"x": ("uniform", -1, 1), "w": ("uniform", -1, 1), "b": ("uniform", -1, 1)},
             "conv1d NCL fp32, N=2, C_in=4, C_out=8, L=32, K=3, stride 1, pad 2, dilation 2, bias"),
    Workload("pointwise_1x1_nhwc_bf16", 1, "fwd", "bf16", 2, "nhwc", "ohwi", 32, 256, 64, (56, 56), (1, 1), (1, 1),
             (0, 0), (1, 1), 1, False, (32, 56, 56, 256), (64, 1, 1, 256), (),
             {"x": ("normal", 1.0), "w": ("normal", (1.0 / 256) ** 0.5)},
             "pointwise 1x1 conv2d NHWC bf16, N=32, 56x56, C 256->64, no bias"),
    Workload("dense3x3_nhwc_bf16", 2, "fwd", "bf16", 2, "nhwc", "ohwi", 32, 64, 64, (56, 56), (3, 3), (1, 1),
             (1, 1), (1, 1), 1, True, (32, 56, 56, 64), (64, 3, 3, 64), (),
             {"x": ("normal", 1.0), "w": ("normal", (2.0 / (64 * 9)) ** 0.5), "b": ("normal", 0.1)},
             "dense 3x3 conv2d NHWC bf16, N=32, 56x56, C 64->64, stride 1, pad 1, fp32 bias"),
    Workload("depthwise3x3_s2_nhwc_bf16", 3, "fwd", "bf16", 2, "nhwc", "ohwi", 32, 256, 256, (112, 112), (3, 3),
             (2, 2), (1, 1), (1, 1), 256, False, (32, 112, 112, 256), (256, 3, 3, 1), (),
             {"x": ("normal", 1.0), "w": ("normal", (2.0 / 9) ** 0.5)},
             "depthwise 3x3 conv2d NHWC bf16, N=32, 112x112, C=G=256, stride 2, pad 1, no bias"),
    Workload("dgrad3x3_s2_nhwc_bf16", 4, "dgrad", "bf16", 2, "nhwc", "ohwi", 16, 128, 256, (64, 64), (3, 3),
             (2, 2), (1, 1), (1, 1), 1, False, (16, 64, 64, 128), (256, 3, 3, 128), (16, 32, 32, 256),
             {"g": ("normal", 1.0), "w": ("normal", (2.0 / (128 * 9)) ** 0.5)},
             "conv2d backward-data NHWC bf16, 3x3 stride 2 pad 1, x 16x64x64x128, dy 16x32x32x256"),
]

# Widening beyond the five: the depthwise input gradient, the transpose of the depthwise workload
# (dy 32x56x56x256 -> dx 32x112x112x256).
EXTRA_WORKLOADS = [
    Workload("depthwise3x3_s2_dgrad_nhwc_bf16", 5, "dgrad", "bf16", 2, "nhwc", "ohwi", 32, 256, 256, (112, 112),
             (3, 3), (2, 2), (1, 1), (1, 1), 256, False, (32, 112, 112, 256), (256, 3, 3, 1), (32, 56, 56, 256),
             {"g": ("normal", 1.0), "w": ("normal", (2.0 / 9) ** 0.5)},
             "depthwise 3x3 stride-2 pad-1 backward-data NHWC bf16, dx 32x112x112x256, dy 32x56x56x256"),
    # a strided dense forward (ResNet-style downsampling): four stride-phase sources per tile
    Workload("dense3x3_s2_nhwc_bf16", 6, "fwd", "bf16", 2, "nhwc", "ohwi", 32, 128, 128, (56, 56), (3, 3), (2, 2),
             (1, 1), (1, 1), 1, True, (32, 56, 56, 128), (128, 3, 3, 128), (),
             {"x": ("normal", 1.0), "w": ("normal", (2.0 / (128 * 9)) ** 0.5), "b": ("normal", 0.1)},
             "dense 3x3 conv2d NHWC bf16, N=32, 56x56 -> 28x28, C 128->128, stride 2, pad 1, fp32 bias"),
    # the weight gradient of the dense 3x3 workload: dW [64, 3, 3, 64] from x and dy, both 32x56x56x64
    Workload("wgrad3x3_nhwc_bf16", 7, "wgrad", "bf16", 2, "nhwc", "ohwi", 32, 64, 64, (56, 56), (3, 3), (1, 1),
             (1, 1), (1, 1), 1, False, (32, 56, 56, 64), (64, 3, 3, 64), (32, 56, 56, 64),
             {"x": ("normal", 1.0), "g": ("normal", 1.0)},
             "conv2d backward-filter NHWC bf16, 3x3 stride 1 pad 1, x and dy 32x56x56x64 -> dW 64x3x3x64"),
    # a 3-D convolution layer: 3x3x3, N=2, 16x56x56, C 64->64, pad 1, fp32 bias
    Workload("dense3x3x3_ndhwc_bf16", 8, "fwd", "bf16", 3, "ndhwc", "odhwi", 2, 64, 64, (16, 56, 56), (3, 3, 3),
             (1, 1, 1), (1, 1, 1), (1, 1, 1), 1, True, (2, 16, 56, 56, 64), (64, 3, 3, 3, 64), (),
             {"x": ("normal", 1.0), "w": ("normal", (2.0 / (64 * 27)) ** 0.5), "b": ("normal", 0.1)},
             "dense 3x3x3 conv3d NDHWC bf16, N=2, 16x56x56, C 64->64, stride 1, pad 1, fp32 bias"),
    # the input gradient of that layer: dx 2x16x56x56x64 from dy of the same shape
    Workload("dgrad3x3x3_ndhwc_bf16", 9, "dgrad", "bf16", 3, "ndhwc", "odhwi", 2, 64, 64, (16, 56, 56), (3, 3, 3),
             (1, 1, 1), (1, 1, 1), (1, 1, 1), 1, False, (2, 16, 56, 56, 64), (64, 3, 3, 3, 64), (2, 16, 56, 56, 64),
             {"g": ("normal", 1.0), "w": ("normal", (2.0 / (64 * 27)) ** 0.5)},
             "conv3d backward-data NDHWC bf16, 3x3x3 stride 1 pad 1, dx and dy 2x16x56x56x64"),
    # and its weight gradient: dW 64x3x3x3x64 from x and dy, both 2x16x56x56x64
    Workload("wgrad3x3x3_ndhwc_bf16", 10, "wgrad", "bf16", 3, "ndhwc", "odhwi", 2, 64, 64, (16, 56, 56), (3, 3, 3),
             (1, 1, 1), (1, 1, 1), (1, 1, 1), 1, False, (2, 16, 56, 56, 64), (64, 3, 3, 3, 64), (2, 16, 56, 56, 64),
             {"x": ("normal", 1.0), "g": ("normal", 1.0)},
             "conv3d backward-filter NDHWC bf16, 3x3x3 stride 1 pad 1, x and dy 2x16x56x56x64 -> dW 64x3x3x3x64"),
    # the weight gradient of the strided dense workload (ResNet-style downsampling): dW [128, 3, 3, 128]
    # from x 32x56x56x128 and dy 32x28x28x128
    Workload("wgrad3x3_s2_nhwc_bf16", 11, "wgrad", "bf16", 2, "nhwc", "ohwi", 32, 128, 128, (56, 56), (3, 3), (2, 2),
             (1, 1), (1, 1), 1, False, (32, 56, 56, 128), (128, 3, 3, 128), (32, 28, 28, 128),
             {"x": ("normal", 1.0), "g": ("normal", 1.0)},
             "conv2d backward-filter NHWC bf16, 3x3 stride 2 pad 1, x 32x56x56x128, dy 32x28x28x128 -> dW 128x3x3x128"),
    # a small-group layer (ResNeXt-style grouped 3x3): C 256 in 64 groups of 4 channels, 56x56, fp32 bias
    Workload("smallgroup3x3_g64_nhwc_bf16", 12, "fwd", "bf16", 2, "nhwc", "ohwi", 32, 256, 256, (56, 56), (3, 3),
             (1, 1), (1, 1), (1, 1), 64, True, (32, 56, 56, 256), (256, 3, 3, 4), (),
             {"x": ("normal", 1.0), "w": ("normal", (2.0 / (4 * 9)) ** 0.5), "b": ("normal", 0.1)},
             "grouped 3x3 conv2d NHWC bf16, N=32, 56x56, C 256->256, G=64 (4 channels per group), stride 1, pad 1, "
             "fp32 bias"),
    # its input gradient: dx 32x56x56x256 from dy of the same shape
    Workload("smallgroup3x3_g64_dgrad_nhwc_bf16", 13, "dgrad", "bf16", 2, "nhwc", "ohwi", 32, 256, 256, (56, 56),
             (3, 3), (1, 1), (1, 1), (1, 1), 64, False, (32, 56, 56, 256), (256, 3, 3, 4), (32, 56, 56, 256),
             {"g": ("normal", 1.0), "w": ("normal", (2.0 / (4 * 9)) ** 0.5)},
             "grouped 3x3 conv2d backward-data NHWC bf16, G=64 (4 channels per group), dx and dy 32x56x56x256"),
    # a grouped dense layer on the tensor cores: C 128 in 2 groups of 64 channels, 56x56, fp32 bias
    Workload("grouped3x3_g2_nhwc_bf16", 14, "fwd", "bf16", 2, "nhwc", "ohwi", 32, 128, 128, (56, 56), (3, 3),
             (1, 1), (1, 1), (1, 1), 2, True, (32, 56, 56, 128), (128, 3, 3, 64), (),
             {"x": ("normal", 1.0), "w": ("normal", (2.0 / (64 * 9)) ** 0.5), "b": ("normal", 0.1)},
             "grouped 3x3 conv2d NHWC bf16, N=32, 56x56, C 128->128, G=2 (64 channels per group), stride 1, pad 1, "
             "fp32 bias"),
]

BY_NAME = {w.name: w for w in WORKLOADS + EXTRA_WORKLOADS}


def _draw(spec, seed, shape):
    kind = spec[0]
    if kind == "uniform":
        return uniform(seed, shape, spec[1], spec[2])
    if kind == "normal":
        return normal(seed, shape, spec[1])
    raise ValueError(kind)


def make_inputs(wl: Workload, seed: int | None = None) -> dict:
    """Draw the workload's inputs.

    Returns float32 arrays of the operation's inputs: ``x`` and ``w`` (forward), ``g`` and ``w``
    (input gradient) or ``x`` and ``g`` (weight gradient), and, when the workload has one, float32
    ``b``; for bf16 workloads also the uint16 bit patterns (``x_bits``, ``g_bits``, ``w_bits``) of the
    same values.
    """
    base = 1000 + wl.index if seed is None else seed
    out = {}
    if wl.op == "dgrad":
        names = [("g", wl.g_shape), ("w", wl.w_shape)]
    elif wl.op == "wgrad":
        names = [("x", wl.x_shape), ("g", wl.g_shape)]
    else:
        names = [("x", wl.x_shape), ("w", wl.w_shape)]
    for i, (name, shape) in enumerate(names):
        v = _draw(wl.recipe[name], base * 16 + i, shape)
        if wl.dtype == "bf16":
            bits, f = as_bf16(v)
            out[name + "_bits"] = bits
            out[name] = f
        else:
            out[name] = v.astype(np.float32)
    if wl.bias:
        out["b"] = _draw(wl.recipe["b"], base * 16 + 7, (wl.c_out,)).astype(np.float32)
    return out
