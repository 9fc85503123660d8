"""GPU parity: every kernel family, through the C ABI, against the FP64 oracle.

Small shapes (several tiles, ragged tails, odd extents, zero-tap phases) are
compared element by element with the whole oracle output.  The benchmark
workloads run at full size in the launch configuration the benchmark times
and are compared element by element with the whole oracle output too (the
oracle split over the host's cores).  Integer-valued inputs make every
product and partial sum exact, so those runs, small and full size, must match
the oracle bit for bit (after the one bf16 rounding of the output).
"""
import numpy as np
import pytest

import oracle
import synth
from synth.workloads import EXTRA_WORKLOADS, WORKLOADS, make_inputs
from tests.helpers import (bf16_round, check_bf16, check_f32, draw, lib_desc, oracle_conv, oracle_whole, scale_dgrad,
                           scale_fwd, shape_kw, to_device, to_host_f64)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
GUARD = 64  # elements of sentinel on each side of every output buffer


@pytest.fixture(scope="module")
def gb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import convolution_conv_fwd_gb300 as gb
    return gb


def _guarded(shape, dtype):
    numel = int(np.prod(shape))
    buf = torch.full((numel + 2 * GUARD,), 7.0, dtype=dtype, device="cuda")
    return buf, buf[GUARD:GUARD + numel].view(shape)


def _guards_intact(buf):
    g = torch.cat([buf[:GUARD], buf[-GUARD:]]).float()
    return bool((g == 7.0).all())


def run_fwd(gb, kw, inp):
    d = lib_desc(gb, kw)
    bits = kw["dtype"] == "bf16"
    x = to_device(torch, inp["x"], inp.get("x_bits") if bits else None)
    w = to_device(torch, inp["w"], inp.get("w_bits") if bits else None)
    b = to_device(torch, inp["b"]) if "b" in inp else None
    _, _, ys = gb.desc_shapes(d)
    buf, y = _guarded(ys, torch.bfloat16 if bits else torch.float32)
    gb.conv_fwd(d, x, w, b, y=y)
    gb.device_status()
    assert _guards_intact(buf), "kernel wrote outside y"
    return to_host_f64(torch, y)


def run_dgrad(gb, kw, inp):
    d = lib_desc(gb, kw)
    bits = kw["dtype"] == "bf16"
    g = to_device(torch, inp["g"], inp.get("g_bits") if bits else None)
    w = to_device(torch, inp["w"], inp.get("w_bits") if bits else None)
    xs, _, _ = gb.desc_shapes(d)
    buf, dx = _guarded(xs, torch.bfloat16 if bits else torch.float32)
    gb.conv_bwd_data(d, g, w, dx=dx)
    gb.device_status()
    assert _guards_intact(buf), "kernel wrote outside dx"
    return to_host_f64(torch, dx)


# (shape, op, expected kernel family)
SMALL = [
    # implicit GEMM forward (tcgen05), resident and streamed weights, ragged tiles, dilation, K-block tails
    (shape_kw(n=2, in_size=(9, 11), c_in=64, c_out=64, bias=True), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(7, 5), c_in=32, c_out=96), "fwd", "implicit"),
    (shape_kw(n=3, in_size=(12, 12), c_in=128, c_out=128, dil=(2, 2), pad=(2, 2), bias=True), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(6, 20), c_in=16, c_out=256, k=(5, 3), pad=(2, 1)), "fwd", "implicit"),
    (shape_kw(n=2, in_size=(10, 10), c_in=48, c_out=32, pad=(0, 0)), "fwd", "implicit"),
    (shape_kw(n=2, in_size=(9, 9), c_in=64, c_out=96, k=(1, 1), pad=(0, 0)), "fwd", "implicit"),
    (shape_kw(spatial_dims=1, n=3, in_size=(37,), c_in=32, c_out=64, k=(3,), stride=(1,), pad=(2,), dil=(2,),
              layout="nlc", wlayout="oki", bias=True), "fwd", "implicit"),
    # channel tails: 80 input channels (second 64-block zero-filled by TMA), 72 outputs (masked N columns)
    (shape_kw(n=2, in_size=(7, 9), c_in=80, c_out=72, bias=True), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(6, 7), c_in=64, c_out=192, bias=True), "fwd", "implicit"),
    # resident weights with two 64-channel k-blocks (every (k-block, tap) tile stays in shared memory)
    (shape_kw(n=2, in_size=(11, 12), c_in=128, c_out=64, k=(2, 2), pad=(0, 0), bias=True), "fwd", "implicit"),
    # small C_out at unit stride: dilation 2, a 1x2 kernel at dilation 3, a 3x2 kernel over two
    # k-blocks, 8 channels, and many items per image with a ragged last one
    (shape_kw(n=2, in_size=(13, 17), c_in=64, c_out=64, dil=(2, 2), pad=(2, 2), bias=True), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(9, 30), c_in=64, c_out=16, k=(1, 2), pad=(0, 1), dil=(1, 3)), "fwd", "implicit"),
    (shape_kw(n=2, in_size=(10, 9), c_in=96, c_out=48, k=(3, 2), pad=(1, 0), bias=True), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(12, 7), c_in=8, c_out=8), "fwd", "implicit"),
    (shape_kw(n=3, in_size=(60, 60), c_in=64, c_out=64, bias=True), "fwd", "implicit"),
    # C_out = 64 (64-wide N tiles): odd output widths, KW = 2 and 5, a row stride, two k-blocks, a
    # k-block tail, (begin, end) padding, row dilation
    (shape_kw(n=2, in_size=(9, 13), c_in=64, c_out=64, bias=True), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(10, 12), c_in=64, c_out=64, k=(2, 2), pad=(0, 0)), "fwd", "implicit"),
    (shape_kw(n=2, in_size=(11, 15), c_in=128, c_out=64, k=(3, 5), pad=(1, 2), bias=True), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(17, 14), c_in=72, c_out=64, stride=(2, 1), bias=True), "fwd", "implicit"),
    (shape_kw(n=2, in_size=(12, 11), c_in=64, c_out=64, pad=(0, 1), pad_end=(2, 0)), "fwd", "implicit"),
    (shape_kw(n=2, in_size=(30, 25), c_in=64, c_out=64, k=(3, 3), pad=(2, 1), dil=(2, 1)), "fwd", "implicit"),
    # images wider than one halo box: column strips (each with its own virtual grid), the last strip
    # narrower; strided forward, grouped, 3-D, dilation, C_out tails
    (shape_kw(n=1, in_size=(9, 150), c_in=64, c_out=64, bias=True), "fwd", "implicit"),
    (shape_kw(n=2, in_size=(6, 113), c_in=128, c_out=96, k=(3, 5), pad=(1, 2), bias=True), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(11, 230), c_in=64, c_out=128, stride=(2, 2), bias=True), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(7, 171), c_in=64, c_out=64, dil=(1, 2), pad=(1, 2)), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(6, 140), c_in=128, c_out=128, groups=2, bias=True), "fwd", "implicit"),
    (shape_kw(spatial_dims=3, n=1, in_size=(3, 5, 130), c_in=64, c_out=64, k=(3, 3, 3), stride=(1, 1, 1),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(10, 150), c_in=128, c_out=128, stride=(2, 2)), "dgrad", "dgrad"),
    (shape_kw(n=2, in_size=(5, 121), c_in=64, c_out=128), "dgrad", "dgrad"),
    (shape_kw(n=1, in_size=(9, 233), c_in=64, c_out=64, stride=(2, 1), k=(3, 2), pad=(1, 0)), "dgrad", "dgrad"),
    # pointwise TMA GEMM: ragged M, K tail inside a 64-wide block, every N tile width
    (shape_kw(n=2, in_size=(9, 7), c_in=256, c_out=64, k=(1, 1), pad=(0, 0)), "fwd", "pointwise"),
    # more 128-row tiles than SMs (a second round on a few CTAs) and a ragged last tile
    (shape_kw(n=2, in_size=(110, 89), c_in=64, c_out=64, k=(1, 1), pad=(0, 0)), "fwd", "pointwise"),
    # 252 tiles: two tiles on each of 126 CTAs (the grid is sized for equal rounds), ragged last tile
    # 128-channel tiles with channels on M: a grouped forward (128 channels per group, bias) and five
    # output tiles of one plan
    (shape_kw(n=2, in_size=(9, 11), c_in=256, c_out=256, groups=2, bias=True), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(7, 6), c_in=64, c_out=640, bias=True), "fwd", "implicit"),
    (shape_kw(n=2, in_size=(126, 128), c_in=64, c_out=32, k=(1, 1), pad=(0, 0), bias=True), "fwd", "pointwise"),
    (shape_kw(n=1, in_size=(13, 13), c_in=72, c_out=128, k=(1, 1), pad=(0, 0), bias=True), "fwd", "pointwise"),
    (shape_kw(n=3, in_size=(10, 10), c_in=64, c_out=256, k=(1, 1), pad=(0, 0)), "fwd", "pointwise"),
    (shape_kw(n=1, in_size=(5, 9), c_in=8, c_out=32, k=(1, 1), pad=(0, 0)), "fwd", "pointwise"),
    # depthwise
    (shape_kw(n=2, in_size=(15, 13), c_in=64, c_out=64, groups=64, stride=(2, 2), bias=True), "fwd", "depthwise"),
    (shape_kw(n=1, in_size=(8, 8), c_in=24, c_out=24, groups=24, k=(5, 5), pad=(2, 2)), "fwd", "depthwise"),
    (shape_kw(n=2, in_size=(9, 9), c_in=256, c_out=256, groups=256, dil=(2, 2), pad=(1, 1)), "fwd", "depthwise"),
    (shape_kw(n=2, in_size=(11, 10), c_in=32, c_out=32, groups=32, bias=True), "fwd", "depthwise"),
    (shape_kw(n=1, in_size=(10, 9), c_in=16, c_out=16, groups=16, stride=(2, 2), pad=(0, 0)), "fwd", "depthwise"),
    (shape_kw(n=1, in_size=(21, 19), c_in=40, c_out=40, groups=40, stride=(2, 2), pad=(2, 2)), "fwd", "depthwise"),
    # TMA-fed 3x3 path (64-channel chunks): stride 1 and 2, several tiles, ragged tile edges, wide padding
    (shape_kw(n=2, in_size=(13, 37), c_in=128, c_out=128, groups=128, bias=True), "fwd", "depthwise"),
    (shape_kw(n=3, in_size=(19, 35), c_in=64, c_out=64, groups=64, stride=(2, 2), pad=(0, 0)), "fwd", "depthwise"),
    (shape_kw(n=1, in_size=(10, 41), c_in=192, c_out=192, groups=192, stride=(2, 2), pad=(2, 2), bias=True),
     "fwd", "depthwise"),
    # strided 1x1 forward through a strided TMA view (ResNet-style downsampling): stride 2, uneven
    # strides with an odd extent, a K tail, several n-tiles
    (shape_kw(n=2, in_size=(15, 14), c_in=64, c_out=128, k=(1, 1), pad=(0, 0), stride=(2, 2), bias=True),
     "fwd", "implicit"),
    (shape_kw(n=1, in_size=(23, 9), c_in=256, c_out=64, k=(1, 1), pad=(0, 0), stride=(2, 3)), "fwd", "implicit"),
    (shape_kw(n=3, in_size=(8, 8), c_in=72, c_out=40, k=(1, 1), pad=(0, 0), stride=(2, 2)), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(28, 28), c_in=128, c_out=512, k=(1, 1), pad=(0, 0), stride=(2, 2), bias=True),
     "fwd", "implicit"),
    # strided forwards through stride-phase views (several sources per item): 3x3 s2 p1 (ResNet
    # downsampling), odd extents, dilation, 5x5 s2, 3x3 s3 (nine sources), mixed strides, 4x4 s2,
    # and a padded strided 1x1
    (shape_kw(n=2, in_size=(16, 15), c_in=64, c_out=128, stride=(2, 2), bias=True), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(13, 11), c_in=128, c_out=64, stride=(2, 2), dil=(2, 1), pad=(2, 1)), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(17, 14), c_in=32, c_out=64, k=(5, 5), pad=(2, 2), stride=(2, 2)), "fwd", "implicit"),
    (shape_kw(n=2, in_size=(14, 13), c_in=64, c_out=64, stride=(3, 3), pad=(1, 1)), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(12, 17), c_in=72, c_out=96, stride=(1, 2), bias=True), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(18, 18), c_in=64, c_out=256, k=(4, 4), pad=(1, 1), stride=(2, 2)), "fwd", "implicit"),
    (shape_kw(n=2, in_size=(9, 10), c_in=64, c_out=64, k=(1, 1), pad=(1, 1), stride=(2, 2)), "fwd", "implicit"),
    # stride-phase dgrad (tcgen05): one phase, four uneven phases, zero-tap phases, even kernel, N tiles
    (shape_kw(n=2, in_size=(9, 11), c_in=64, c_out=64), "dgrad", "dgrad"),
    (shape_kw(n=2, in_size=(13, 10), c_in=128, c_out=256, stride=(2, 2)), "dgrad", "dgrad"),
    (shape_kw(n=1, in_size=(8, 8), c_in=32, c_out=32, k=(1, 1), pad=(0, 0), stride=(2, 2)), "dgrad", "dgrad"),
    (shape_kw(n=1, in_size=(11, 9), c_in=64, c_out=32, k=(4, 4), stride=(2, 2), pad=(1, 1)), "dgrad", "dgrad"),
    (shape_kw(n=1, in_size=(7, 7), c_in=96, c_out=48, dil=(2, 2), pad=(1, 1)), "dgrad", "dgrad"),
    (shape_kw(n=2, in_size=(9, 9), c_in=72, c_out=40, stride=(2, 2)), "dgrad", "dgrad"),
    (shape_kw(n=1, in_size=(8, 6), c_in=192, c_out=64), "dgrad", "dgrad"),
    # wider dgrad: an odd m-tile count per phase, several rounds, BN = 256 with two n-tiles, a ragged
    # output-channel tail, a 2x2 kernel at stride 2 (four one-tap phases)
    (shape_kw(n=1, in_size=(11, 13), c_in=128, c_out=64, stride=(2, 2)), "dgrad", "dgrad"),
    (shape_kw(n=3, in_size=(40, 37), c_in=128, c_out=72, stride=(2, 2)), "dgrad", "dgrad"),
    (shape_kw(n=1, in_size=(12, 12), c_in=512, c_out=64, stride=(2, 2)), "dgrad", "dgrad"),
    (shape_kw(n=2, in_size=(9, 10), c_in=256, c_out=136, k=(2, 2), pad=(0, 0), stride=(2, 2)), "dgrad", "dgrad"),
    # depthwise dgrad gather (G = C): stride 2 (the transpose of the depthwise workload), stride 1,
    # mixed strides with dilation, a 5x5 kernel, 1x1, many channel chunks
    (shape_kw(n=2, in_size=(14, 15), c_in=64, c_out=64, groups=64, stride=(2, 2)), "dgrad", "depthwise_dgrad"),
    (shape_kw(n=1, in_size=(9, 13), c_in=40, c_out=40, groups=40), "dgrad", "depthwise_dgrad"),
    (shape_kw(n=1, in_size=(12, 11), c_in=24, c_out=24, groups=24, stride=(2, 1), dil=(2, 1), pad=(2, 1)),
     "dgrad", "depthwise_dgrad"),
    (shape_kw(n=1, in_size=(10, 10), c_in=16, c_out=16, groups=16, k=(5, 5), pad=(2, 2), stride=(3, 2)),
     "dgrad", "depthwise_dgrad"),
    (shape_kw(n=2, in_size=(6, 7), c_in=8, c_out=8, groups=8, k=(1, 1), pad=(0, 0), stride=(2, 2)),
     "dgrad", "depthwise_dgrad"),
    (shape_kw(n=1, in_size=(8, 9), c_in=512, c_out=512, groups=512, stride=(2, 2)), "dgrad", "depthwise_dgrad"),
    # the generic direct forward beyond the shared-memory-staged small path (x + w above 8192
    # elements): fp32 NCHW grouped, strided, dilated; bf16 NCHW; fp32 3-D
    (shape_kw(n=2, in_size=(40, 37), c_in=6, c_out=9, groups=3, k=(3, 2), stride=(2, 1), pad=(1, 1), dil=(1, 2),
              layout="nchw", wlayout="oihw", dtype="f32", bias=True), "fwd", "direct"),
    (shape_kw(n=2, in_size=(30, 29), c_in=16, c_out=8, layout="nchw", wlayout="oihw"), "fwd", "direct"),
    (shape_kw(spatial_dims=3, n=1, in_size=(6, 20, 21), c_in=8, c_out=4, k=(3, 3, 3), stride=(1, 1, 1), pad=(1, 1, 1),
              dil=(1, 1, 1), layout="ncdhw", wlayout="oidhw", dtype="f32"), "fwd", "direct"),
    # the TMA-fed depthwise forward at unit stride with 4 x 16 output tiles (4 rows: one tile row)
    (shape_kw(n=2, in_size=(4, 30), c_in=64, c_out=64, groups=64), "fwd", "depthwise"),
    # the TMA-fed stride-2 gather: several 4x16 dy tiles each way, ragged in both, odd H
    (shape_kw(n=3, in_size=(37, 70), c_in=128, c_out=128, groups=128, stride=(2, 2)), "dgrad", "depthwise_dgrad"),
    # (begin, end) padding: implicit forward one-sided, strided with padding after only (the usual
    # 'same' padding of an even input at stride 2), a 1x1 with padding after, the depthwise
    # generic kernel, the stride-phase dgrad, the depthwise dgrad, and the generic direct kernels
    (shape_kw(n=2, in_size=(9, 11), c_in=64, c_out=64, pad=(1, 0), pad_end=(0, 1), bias=True), "fwd", "implicit"),
    (shape_kw(n=2, in_size=(16, 14), c_in=64, c_out=128, stride=(2, 2), pad=(0, 0), pad_end=(1, 1)), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(7, 9), c_in=64, c_out=64, k=(1, 1), pad=(0, 0), pad_end=(1, 2), bias=True),
     "fwd", "implicit"),
    (shape_kw(n=2, in_size=(14, 15), c_in=64, c_out=64, groups=64, stride=(2, 2), pad=(0, 0), pad_end=(1, 1),
              bias=True), "fwd", "depthwise"),
    (shape_kw(n=2, in_size=(16, 13), c_in=128, c_out=64, stride=(2, 2), pad=(0, 1), pad_end=(1, 0)), "dgrad", "dgrad"),
    (shape_kw(n=1, in_size=(14, 12), c_in=32, c_out=32, groups=32, stride=(2, 2), pad=(0, 0), pad_end=(1, 1)),
     "dgrad", "depthwise_dgrad"),
    (shape_kw(n=2, in_size=(9, 8), c_in=6, c_out=4, groups=2, k=(3, 2), stride=(2, 1), pad=(2, 0), pad_end=(0, 1),
              layout="nchw", wlayout="oihw", dtype="f32", bias=True), "fwd", "direct"),
    (shape_kw(n=1, in_size=(10, 7), c_in=8, c_out=12, stride=(2, 2), pad=(1, 0), pad_end=(0, 2), layout="nchw",
              wlayout="oihw", dtype="f32"), "dgrad", "direct_dgrad"),
    # 3-D: a depth kernel (generic kernels: fp32 NCDHW with groups, stride, dilation and begin/end
    # padding; bf16 NDHWC), and depth-1 kernels at unit depth stride, which the 2-D families run
    # on N*D images (implicit GEMM, 1x1 GEMM, depthwise, stride-phase dgrad)
    (shape_kw(spatial_dims=3, n=2, in_size=(5, 6, 7), c_in=4, c_out=6, groups=2, k=(3, 2, 3), stride=(2, 1, 2),
              pad=(1, 0, 1), pad_end=(0, 1, 1), dil=(1, 2, 1), layout="ncdhw", wlayout="oidhw", dtype="f32",
              bias=True), "fwd", "direct"),
    (shape_kw(spatial_dims=3, n=1, in_size=(4, 6, 5), c_in=16, c_out=8, k=(3, 3, 3), stride=(1, 1, 1),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "fwd", "implicit"),
    # 3-D forwards on the implicit GEMM (one activation source per kernel-depth tap, 5-D TMA boxes):
    # depth stride, depth dilation with (begin, end) depth padding, several k-blocks and N tiles,
    # kernel depth 2 with an H/W stride (two stride phases per depth tap)
    (shape_kw(spatial_dims=3, n=2, in_size=(5, 9, 11), c_in=64, c_out=64, k=(3, 3, 3), stride=(2, 1, 1),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi", bias=True), "fwd", "implicit"),
    (shape_kw(spatial_dims=3, n=1, in_size=(6, 7, 8), c_in=32, c_out=64, k=(3, 3, 3), stride=(1, 1, 1),
              pad=(2, 1, 1), pad_end=(0, 1, 1), dil=(2, 1, 1), layout="ndhwc", wlayout="odhwi"), "fwd", "implicit"),
    (shape_kw(spatial_dims=3, n=1, in_size=(3, 6, 7), c_in=128, c_out=192, k=(2, 2, 3), stride=(1, 1, 1),
              pad=(0, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi", bias=True), "fwd", "implicit"),
    (shape_kw(spatial_dims=3, n=1, in_size=(4, 9, 10), c_in=64, c_out=64, k=(2, 3, 3), stride=(1, 2, 1),
              pad=(0, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "fwd", "implicit"),
    (shape_kw(spatial_dims=3, n=2, in_size=(3, 7, 6), c_in=64, c_out=64, k=(1, 3, 3), stride=(1, 1, 1),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi", bias=True), "fwd", "implicit"),
    (shape_kw(spatial_dims=3, n=2, in_size=(5, 6, 7), c_in=4, c_out=6, groups=2, k=(3, 2, 3), stride=(2, 1, 2),
              pad=(1, 0, 1), dil=(1, 2, 1), layout="ncdhw", wlayout="oidhw", dtype="f32"), "dgrad", "direct_dgrad"),
    (shape_kw(spatial_dims=3, n=1, in_size=(4, 6, 5), c_in=16, c_out=8, k=(3, 3, 3), stride=(2, 1, 1),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "dgrad", "dgrad"),
    (shape_kw(spatial_dims=3, n=2, in_size=(3, 9, 11), c_in=64, c_out=64, k=(1, 3, 3), stride=(1, 1, 1),
              pad=(0, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi", bias=True), "fwd", "implicit"),
    (shape_kw(spatial_dims=3, n=2, in_size=(3, 7, 9), c_in=128, c_out=64, k=(1, 1, 1), stride=(1, 1, 1),
              pad=(0, 0, 0), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "fwd", "pointwise"),
    (shape_kw(spatial_dims=3, n=1, in_size=(4, 10, 9), c_in=64, c_out=64, groups=64, k=(1, 3, 3), stride=(1, 2, 2),
              pad=(0, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "fwd", "depthwise"),
    (shape_kw(spatial_dims=3, n=2, in_size=(3, 10, 9), c_in=64, c_out=128, k=(1, 3, 3), stride=(1, 2, 2),
              pad=(0, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "dgrad", "dgrad"),
    # 3-D input gradients on the implicit GEMM (unit depth stride: one dy source per kernel-depth tap,
    # items over N*D dx slices): 3x3x3; H/W stride 2 (four stride phases per depth tap) with depth
    # dilation and (begin, end) depth padding; several k-blocks and a 128-wide N tile; a 192-wide N
    # tile; a depth-1 kernel with depth padding (one source at a depth offset)
    (shape_kw(spatial_dims=3, n=2, in_size=(4, 9, 11), c_in=64, c_out=64, k=(3, 3, 3), stride=(1, 1, 1),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "dgrad", "dgrad"),
    (shape_kw(spatial_dims=3, n=1, in_size=(6, 10, 9), c_in=64, c_out=128, k=(3, 3, 3), stride=(1, 2, 2),
              pad=(2, 1, 1), pad_end=(0, 1, 1), dil=(2, 1, 1), layout="ndhwc", wlayout="odhwi"), "dgrad", "dgrad"),
    (shape_kw(spatial_dims=3, n=1, in_size=(3, 6, 7), c_in=128, c_out=192, k=(2, 2, 3), stride=(1, 1, 1),
              pad=(0, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "dgrad", "dgrad"),
    (shape_kw(spatial_dims=3, n=1, in_size=(3, 8, 6), c_in=192, c_out=64, k=(2, 3, 3), stride=(1, 2, 2),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "dgrad", "dgrad"),
    (shape_kw(spatial_dims=3, n=2, in_size=(3, 7, 6), c_in=64, c_out=64, k=(1, 3, 3), stride=(1, 1, 1),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "dgrad", "dgrad"),
    # depth strides: dx split into depth phases, each met by the kernel-depth taps that divide
    # evenly: 2x2x2 strides (eight phases, an odd depth); depth stride 3; depth stride 2 with depth
    # dilation and (begin, end) depth padding; a depth-1 kernel, whose odd depth phase no tap reaches
    (shape_kw(spatial_dims=3, n=1, in_size=(5, 8, 9), c_in=64, c_out=64, k=(3, 3, 3), stride=(2, 2, 2),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "dgrad", "dgrad"),
    (shape_kw(spatial_dims=3, n=2, in_size=(7, 6, 7), c_in=64, c_out=64, k=(3, 3, 3), stride=(3, 1, 1),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "dgrad", "dgrad"),
    (shape_kw(spatial_dims=3, n=1, in_size=(7, 6, 5), c_in=64, c_out=128, k=(3, 3, 3), stride=(2, 1, 1),
              pad=(2, 1, 1), pad_end=(1, 1, 1), dil=(2, 1, 1), layout="ndhwc", wlayout="odhwi"), "dgrad", "dgrad"),
    (shape_kw(spatial_dims=3, n=2, in_size=(5, 7, 6), c_in=64, c_out=64, k=(1, 3, 3), stride=(2, 1, 1),
              pad=(0, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "dgrad", "dgrad"),
    # small groups (1 < G < C, C_in/G = C_out/G in {2, 4, 8}): TMA halo tiles on CUDA cores; ragged
    # tile rows and columns, strides, dilation, (begin, end) padding, 1-D, OIHW weights, a 1x1 kernel
    (shape_kw(n=2, in_size=(13, 37), c_in=64, c_out=64, groups=16, bias=True), "fwd", "smallgroup"),
    (shape_kw(n=1, in_size=(15, 14), c_in=128, c_out=128, groups=64, stride=(2, 2), bias=True), "fwd", "smallgroup"),
    (shape_kw(n=2, in_size=(10, 9), c_in=128, c_out=128, groups=16, k=(5, 3), pad=(2, 1), dil=(1, 2)), "fwd",
     "smallgroup"),
    (shape_kw(n=1, in_size=(9, 40), c_in=64, c_out=64, groups=32, k=(1, 1), pad=(0, 0)), "fwd", "smallgroup"),
    (shape_kw(n=2, in_size=(11, 12), c_in=64, c_out=64, groups=8, pad=(0, 1), pad_end=(2, 0), bias=True), "fwd",
     "smallgroup"),
    (shape_kw(spatial_dims=1, n=2, in_size=(70,), c_in=64, c_out=64, groups=16, k=(5,), stride=(1,), pad=(2,),
              dil=(1,), layout="nlc", wlayout="oki"), "fwd", "smallgroup"),
    (shape_kw(n=1, in_size=(8, 8), c_in=64, c_out=64, groups=16, wlayout="oihw"), "fwd", "smallgroup"),
    (shape_kw(n=1, in_size=(20, 66), c_in=192, c_out=192, groups=48, stride=(1, 2), pad=(1, 1)), "fwd", "smallgroup"),
    # outputs 56 and 112 wide, partial and whole 32-column tiles (8 channels per group: the generic
    # path; 2 per group: the compile-time 3x3)
    (shape_kw(n=1, in_size=(10, 112), c_in=128, c_out=128, groups=16, bias=True), "fwd", "smallgroup"),
    (shape_kw(n=2, in_size=(9, 56), c_in=64, c_out=64, groups=32, bias=True), "fwd", "smallgroup"),
    # their input gradients: the tiled kernel at stride 1 (transposed, flipped weights), the gather otherwise
    (shape_kw(n=2, in_size=(13, 37), c_in=64, c_out=64, groups=16), "dgrad", "smallgroup_dgrad"),
    (shape_kw(n=1, in_size=(12, 11), c_in=128, c_out=128, groups=16, dil=(2, 2), pad=(2, 2)), "dgrad",
     "smallgroup_dgrad"),
    (shape_kw(n=2, in_size=(9, 10), c_in=64, c_out=64, groups=32, pad=(0, 0)), "dgrad", "smallgroup_dgrad"),
    (shape_kw(n=1, in_size=(8, 8), c_in=64, c_out=64, groups=16, pad=(3, 3)), "dgrad", "smallgroup_dgrad"),
    (shape_kw(n=1, in_size=(9, 9), c_in=64, c_out=64, groups=8, pad=(1, 0), pad_end=(0, 2), wlayout="oihw"),
     "dgrad", "smallgroup_dgrad"),
    (shape_kw(n=2, in_size=(15, 13), c_in=64, c_out=64, groups=16, stride=(2, 2)), "dgrad", "smallgroup_dgrad"),
    (shape_kw(n=1, in_size=(14, 11), c_in=128, c_out=128, groups=16, k=(3, 2), stride=(2, 1), pad=(1, 0)), "dgrad",
     "smallgroup_dgrad"),
    (shape_kw(n=2, in_size=(12, 13), c_in=64, c_out=64, groups=32, stride=(3, 2), wlayout="oihw"), "dgrad",
     "smallgroup_dgrad"),
    (shape_kw(n=1, in_size=(10, 56), c_in=128, c_out=128, groups=16), "dgrad", "smallgroup_dgrad"),
    # grouped dense convolutions on the tensor cores: one implicit GEMM per group (group views of the
    # activations, group offsets into the weight and the output); whole and partial 64-channel k-blocks
    # per group, C_out/G != C_in/G, strides (stride-phase sources / phases), 1x1, tiles wider than a group
    (shape_kw(n=2, in_size=(9, 11), c_in=128, c_out=128, groups=2, bias=True), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(10, 9), c_in=128, c_out=128, groups=4), "fwd", "implicit"),
    (shape_kw(n=2, in_size=(8, 13), c_in=128, c_out=256, groups=8, bias=True), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(13, 12), c_in=192, c_out=96, groups=3, stride=(2, 2), bias=True), "fwd", "implicit"),
    (shape_kw(n=2, in_size=(7, 9), c_in=96, c_out=48, groups=2, k=(1, 1), pad=(0, 0)), "fwd", "implicit"),
    (shape_kw(n=1, in_size=(11, 10), c_in=64, c_out=64, groups=4, dil=(2, 1), pad=(2, 1), pad_end=(0, 1)), "fwd",
     "implicit"),
    (shape_kw(n=2, in_size=(9, 11), c_in=128, c_out=128, groups=2), "dgrad", "dgrad"),
    (shape_kw(n=1, in_size=(12, 10), c_in=128, c_out=256, groups=4, stride=(2, 2)), "dgrad", "dgrad"),
    (shape_kw(n=2, in_size=(10, 9), c_in=96, c_out=192, groups=6, stride=(2, 1), k=(3, 2), pad=(1, 0)), "dgrad",
     "dgrad"),
    (shape_kw(n=1, in_size=(8, 8), c_in=256, c_out=128, groups=2, k=(1, 1), pad=(0, 0)), "dgrad", "dgrad"),
    # generic direct kernels (CUDA cores)
    (shape_kw(spatial_dims=1, n=2, in_size=(32,), c_in=4, c_out=8, k=(3,), stride=(1,), pad=(2,), dil=(2,),
              layout="ncl", wlayout="oik", dtype="f32", bias=True), "fwd", "direct"),
    (shape_kw(n=2, in_size=(11, 9), c_in=6, c_out=9, groups=3, k=(3, 2), stride=(2, 1), pad=(1, 0), dil=(1, 2),
              dtype="f32", bias=True), "fwd", "direct"),
    (shape_kw(n=1, in_size=(9, 8), c_in=16, c_out=8, layout="nchw", wlayout="oihw", stride=(2, 2)), "fwd", "direct"),
    (shape_kw(n=2, in_size=(7, 9), c_in=6, c_out=4, groups=2, layout="nchw", wlayout="oihw", dtype="f32",
              stride=(2, 2)), "dgrad", "direct_dgrad"),
    (shape_kw(n=1, in_size=(10, 6), c_in=16, c_out=16, groups=2, stride=(2, 1)), "dgrad", "direct_dgrad"),
]


def _ids():
    return ["%s-%d" % (fam, i) for i, (_, _, fam) in enumerate(SMALL)]


@pytest.mark.parametrize("case", range(len(SMALL)), ids=_ids())
def test_small_shapes_match_oracle(gb, case):
    kw, op, family = SMALL[case]
    d = lib_desc(gb, kw)
    assert gb.gbconv_select(d, gb.GBCONV_OP_BWD_DATA if op == "dgrad" else gb.GBCONV_OP_FWD) == family
    c = oracle_conv(kw)
    inp = draw(c, kw["dtype"], 100 + case, op=op, bias=kw["bias"])
    if op == "fwd":
        got = run_fwd(gb, kw, inp)
        ref = oracle.conv_fwd(c, inp["x"], inp["w"], inp.get("b"))
        scale = scale_fwd(c, inp["x"], inp["w"], inp.get("b"))
    else:
        got = run_dgrad(gb, kw, inp)
        ref = oracle.conv_dgrad(c, inp["g"], inp["w"])
        scale = scale_dgrad(c, inp["g"], inp["w"])
    assert got.shape == ref.shape
    if kw["dtype"] == "f32":
        check_f32(got, ref, scale)
    else:
        check_bf16(got, ref, scale)


# Host (pinned CPU) tensors through the public calls: batch slices whose copies overlap the kernels
# (sliced here even at these sizes), uneven slices, each call kind.
HOST = [
    (shape_kw(n=5, in_size=(12, 11), c_in=64, c_out=64, bias=True), "fwd"),
    (shape_kw(n=6, in_size=(14, 15), c_in=64, c_out=64, groups=64, stride=(2, 2)), "fwd"),
    (shape_kw(n=3, in_size=(16, 13), c_in=128, c_out=64, stride=(2, 2)), "dgrad"),
    (shape_kw(n=4, in_size=(13, 10), c_in=128, c_out=256, stride=(2, 2)), "transpose"),
    (shape_kw(n=3, in_size=(9, 8), c_in=6, c_out=4, groups=2, layout="nchw", wlayout="oihw", dtype="f32",
              bias=True), "fwd"),
    (shape_kw(spatial_dims=3, n=2, in_size=(4, 9, 11), c_in=64, c_out=64, k=(3, 3, 3), stride=(1, 1, 1),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "dgrad"),
]


def _pinned(torch, arr_f32, bits=None):
    if bits is not None:
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr_f32, dtype=np.float32))
    return t.pin_memory()


@pytest.mark.parametrize("case", range(len(HOST)), ids=["%s-%d" % (op, i) for i, (_, op) in enumerate(HOST)])
def test_host_buffers_match_oracle(gb, case, monkeypatch):
    monkeypatch.setattr(gb, "HOST_SLICES", 4)  # batches of 3-6 in 4 slices: uneven slices
    kw, op = HOST[case]
    d = lib_desc(gb, kw)
    c = oracle_conv(kw)
    bits = kw["dtype"] == "bf16"
    inp = draw(c, kw["dtype"], 900 + case, op="dgrad" if op != "fwd" else "fwd", bias=kw["bias"])
    w = _pinned(torch, inp["w"], inp.get("w_bits") if bits else None)
    if op == "fwd":
        x = _pinned(torch, inp["x"], inp.get("x_bits") if bits else None)
        b = None if "b" not in inp else _pinned(torch, inp["b"])
        got = gb.conv_fwd(d, x, w, b)
        ref = oracle.conv_fwd(c, inp["x"], inp["w"], inp.get("b"))
        scale = scale_fwd(c, inp["x"], inp["w"], inp.get("b"))
    elif op == "dgrad":
        g = _pinned(torch, inp["g"], inp.get("g_bits") if bits else None)
        got = gb.conv_bwd_data(d, g, w)
        ref = oracle.conv_dgrad(c, inp["g"], inp["w"])
        scale = scale_dgrad(c, inp["g"], inp["w"])
    else:
        g = _pinned(torch, inp["g"], inp.get("g_bits") if bits else None)
        bias = synth.normal(990 + case, (kw["c_in"],), 0.5).astype(np.float32)
        got = gb.conv_transpose(d, g, w, _pinned(torch, bias))
        ref = oracle.conv_transpose(c, inp["g"], inp["w"], bias)
        scale = oracle.conv_transpose(c, np.abs(inp["g"]), np.abs(inp["w"]), np.abs(bias))
    assert not got.is_cuda
    got = to_host_f64(torch, got)
    assert got.shape == ref.shape
    (check_bf16 if bits else check_f32)(got, ref, scale)


# Transposed convolution forward (dgrad + a bias over C_in), one case per dgrad kernel family.
TRANSPOSE = [
    (shape_kw(n=2, in_size=(13, 10), c_in=128, c_out=256, stride=(2, 2)), "dgrad"),
    (shape_kw(n=2, in_size=(14, 15), c_in=64, c_out=64, groups=64, stride=(2, 2)), "depthwise_dgrad"),
    (shape_kw(n=1, in_size=(9, 13), c_in=40, c_out=40, groups=40), "depthwise_dgrad"),
    (shape_kw(n=1, in_size=(37, 70), c_in=128, c_out=128, groups=128, stride=(2, 2)), "depthwise_dgrad"),
    (shape_kw(n=2, in_size=(7, 9), c_in=6, c_out=4, groups=2, layout="nchw", wlayout="oihw", dtype="f32",
              stride=(2, 2)), "direct_dgrad"),
    (shape_kw(n=1, in_size=(10, 6), c_in=16, c_out=16, groups=2, stride=(2, 1)), "direct_dgrad"),
    (shape_kw(n=2, in_size=(11, 9), c_in=64, c_out=64, groups=16), "smallgroup_dgrad"),
    (shape_kw(n=1, in_size=(10, 12), c_in=128, c_out=64, groups=2, stride=(2, 2)), "dgrad"),
    (shape_kw(n=1, in_size=(12, 10), c_in=128, c_out=128, groups=32, stride=(2, 2)), "smallgroup_dgrad"),
    (shape_kw(n=1, in_size=(8, 140), c_in=64, c_out=128, stride=(2, 2)), "dgrad"),
    (shape_kw(spatial_dims=3, n=1, in_size=(4, 8, 7), c_in=64, c_out=128, k=(3, 3, 3), stride=(1, 2, 1),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "dgrad"),
    (shape_kw(spatial_dims=3, n=2, in_size=(5, 6, 8), c_in=128, c_out=64, k=(3, 3, 3), stride=(2, 2, 1),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "dgrad"),
]


@pytest.mark.parametrize("case", range(len(TRANSPOSE)), ids=["%s-%d" % (f, i) for i, (_, f) in enumerate(TRANSPOSE)])
def test_conv_transpose_matches_oracle(gb, case):
    kw, family = TRANSPOSE[case]
    d = lib_desc(gb, kw)
    assert gb.gbconv_select(d, gb.GBCONV_OP_BWD_DATA) == family
    c = oracle_conv(kw)
    inp = draw(c, kw["dtype"], 500 + case, op="dgrad")
    b = synth.normal(600 + case, (c.c_in,)).astype(np.float32)
    bits = kw["dtype"] == "bf16"
    x = to_device(torch, inp["g"], inp.get("g_bits") if bits else None)
    w = to_device(torch, inp["w"], inp.get("w_bits") if bits else None)
    xs, _, _ = gb.desc_shapes(d)
    buf, y = _guarded(xs, torch.bfloat16 if bits else torch.float32)
    gb.conv_transpose(d, x, w, to_device(torch, b), y=y)
    gb.device_status()
    assert _guards_intact(buf), "kernel wrote outside y"
    got = to_host_f64(torch, y)
    ref = oracle.conv_transpose(c, inp["g"], inp["w"], b)
    scale = oracle.conv_transpose(c, np.abs(inp["g"]), np.abs(inp["w"]), np.abs(b))
    assert got.shape == ref.shape
    if kw["dtype"] == "f32":
        check_f32(got, ref, scale)
    else:
        check_bf16(got, ref, scale)


@pytest.mark.parametrize("case", range(len(SMALL)), ids=_ids())
def test_integer_inputs_bit_exact(gb, case):
    kw, op, _ = SMALL[case]
    c = oracle_conv(kw)
    inp = draw(c, kw["dtype"], 300 + case, op=op, bias=kw["bias"], kind="int")
    if op == "fwd":
        got = run_fwd(gb, kw, inp)
        ref = oracle.conv_fwd(c, inp["x"], inp["w"], inp.get("b"))
    else:
        got = run_dgrad(gb, kw, inp)
        ref = oracle.conv_dgrad(c, inp["g"], inp["w"])
    if kw["dtype"] == "bf16":
        ref = bf16_round(ref)
    np.testing.assert_array_equal(got, ref)


def test_dgrad_is_deterministic(gb):
    kw = shape_kw(n=2, in_size=(13, 10), c_in=128, c_out=256, stride=(2, 2))
    c = oracle_conv(kw)
    inp = draw(c, "bf16", 77, op="dgrad")
    a = run_dgrad(gb, kw, inp)
    b = run_dgrad(gb, kw, inp)
    assert np.array_equal(a, b)


def test_pack_weight_then_fast_path(gb):
    # OIHW weight packed on the device to OHWI gives the same forward result
    kw = shape_kw(n=2, in_size=(9, 11), c_in=64, c_out=64)
    c_oihw = oracle_conv(dict(kw, wlayout="oihw"))
    inp = draw(c_oihw, "bf16", 91)
    d = lib_desc(gb, dict(kw, wlayout="oihw"))
    w_oihw = to_device(torch, inp["w"], inp["w_bits"])
    w_ohwi = gb.pack_weight(d, w_oihw)
    np.testing.assert_array_equal(to_host_f64(torch, w_ohwi),
                                  inp["w"].transpose(0, 2, 3, 1).astype(np.float64))
    got = run_fwd(gb, kw, dict(x=inp["x"], x_bits=inp["x_bits"], w=inp["w"].transpose(0, 2, 3, 1).copy(),
                               w_bits=inp["w_bits"].transpose(0, 2, 3, 1).copy()))
    ref = oracle.conv_fwd(c_oihw, inp["x"], inp["w"])
    check_bf16(got, ref, scale_fwd(c_oihw, inp["x"], inp["w"], None))


@pytest.mark.parametrize("kw", [
    shape_kw(spatial_dims=1, n=1, in_size=(9,), c_in=16, c_out=24, k=(5,), stride=(1,), pad=(2,), dil=(1,),
             layout="nlc", wlayout="oik"),
    shape_kw(n=1, in_size=(6, 7), c_in=32, c_out=16, groups=2, k=(3, 2), pad=(1, 0), wlayout="oihw"),
    shape_kw(spatial_dims=3, n=1, in_size=(4, 5, 6), c_in=16, c_out=8, k=(3, 2, 3), stride=(1, 1, 1),
             pad=(1, 0, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="oidhw", dtype="f32"),
], ids=["1d", "2d-grouped", "3d-f32"])
def test_pack_weight_shapes(gb, kw):
    # [C_out, C_in/G, K...] -> [C_out, K..., C_in/G] on the device, 1-D, 2-D and 3-D
    d = lib_desc(gb, kw)
    c = oracle_conv(kw)
    w = synth.integers(93, c.w_shape(), -100, 100).astype(np.float32)
    dt = torch.bfloat16 if kw["dtype"] == "bf16" else torch.float32
    got = gb.pack_weight(d, torch.from_numpy(w).to("cuda").to(dt))
    torch.cuda.synchronize()
    nd = w.ndim
    np.testing.assert_array_equal(to_host_f64(torch, got), np.moveaxis(w, 1, nd - 1).astype(np.float64))


# ------------------------------------------------------------ full-size workloads

def _run_workload(gb, wl, inp):
    kw = dict(wl.__dict__)
    if wl.op == "wgrad":
        return run_wgrad(gb, kw, inp, want_db=wl.bias)
    if wl.op == "fwd":
        return run_fwd(gb, kw, inp), None
    return run_dgrad(gb, kw, inp), None


def _oracle_workload(c, wl, inp, absolute=False):
    """The oracle's whole result for the workload (on the host's cores), or with ``absolute`` the
    per-element scale (the same sums over absolute values, |bias| included)."""
    f = np.abs if absolute else (lambda v: v)
    if wl.op == "wgrad":
        return oracle_whole(c, "wgrad", f(inp["x"]), f(inp["g"]))
    if wl.op == "fwd":
        b = inp.get("b")
        return oracle_whole(c, "fwd", f(inp["x"]), f(inp["w"]), None if b is None else f(b))
    return oracle_whole(c, "dgrad", f(inp["g"]), f(inp["w"]))


@pytest.mark.parametrize("wl", WORKLOADS + EXTRA_WORKLOADS, ids=[w.name for w in WORKLOADS + EXTRA_WORKLOADS])
def test_workload_full_size(gb, wl):
    # every output element of the workload, in the launch configuration the benchmark times, against
    # the whole oracle result: the normwise bar and the per-element bound
    c = oracle_conv(wl)
    inp = make_inputs(wl)
    got, db = _run_workload(gb, wl, inp)
    ref = _oracle_workload(c, wl, inp)
    scale = _oracle_workload(c, wl, inp, absolute=True)
    assert got.shape == ref.shape
    if wl.dtype == "f32":
        check_f32(got, ref, scale)
    else:
        check_bf16(got, ref, scale)
    if db is not None and wl.bias:
        check_bf16(db, oracle.conv_bgrad(c, inp["g"]), oracle.conv_bgrad(c, np.abs(inp["g"])))


def _integer_inputs(wl):
    """Integer-valued inputs of the workload's shapes (activations and output gradients in [-3, 3],
    weights in [-2, 2], bias in [-4, 4]): every bf16 product and every fp32 partial sum is exact."""
    base = 6000 + wl.index
    out = {}
    shapes = {"fwd": (("x", wl.x_shape), ("w", wl.w_shape)), "dgrad": (("g", wl.g_shape), ("w", wl.w_shape)),
              "wgrad": (("x", wl.x_shape), ("g", wl.g_shape))}[wl.op]
    for i, (name, shape) in enumerate(shapes):
        lo, hi = (-2, 2) if name == "w" else (-3, 3)
        out[name + "_bits"], out[name] = synth.as_bf16(synth.integers(base * 16 + i, shape, lo, hi))
    if wl.bias and wl.op == "fwd":
        out["b"] = synth.integers(base * 16 + 7, (wl.c_out,), -4, 4).astype(np.float32)
    return out


BF16_WORKLOADS = [w for w in WORKLOADS + EXTRA_WORKLOADS if w.dtype == "bf16"]


@pytest.mark.parametrize("wl", BF16_WORKLOADS, ids=[w.name for w in BF16_WORKLOADS])
def test_workload_full_size_integer_bit_exact(gb, wl):
    # the full-size launch configurations (wide tiles, several persistent rounds, every stride phase,
    # chunked weight-gradient sums) on integer inputs: the largest sum stays below 2^24, so fp32 holds
    # every partial sum exactly and the output must equal the oracle rounded once to bf16, bit for bit
    c = oracle_conv(wl)
    inp = _integer_inputs(wl)
    got, db = _run_workload(gb, wl, inp)
    ref = _oracle_workload(c, wl, inp)
    scale = _oracle_workload(c, wl, inp, absolute=True)
    assert float(scale.max()) < 2.0 ** 24
    np.testing.assert_array_equal(got, bf16_round(ref))
    if db is not None and wl.bias:
        np.testing.assert_array_equal(db, oracle.conv_bgrad(c, inp["g"]))


# ---------------------------------------------------------------- weight gradient

def draw_wgrad(c, dtype, seed, kind="normal"):
    """Seeded x and dy for a weight-gradient case (float32 values, and bf16 bits for bf16)."""
    out = {}
    for i, (name, shape) in enumerate([("x", c.x_shape()), ("g", c.y_shape())]):
        v = synth.integers(seed * 16 + i, shape, -3, 3) if kind == "int" else synth.normal(seed * 16 + i, shape, 1.0)
        if dtype == "bf16":
            out[name + "_bits"], out[name] = synth.as_bf16(v)
        else:
            out[name] = v.astype(np.float32)
    return out


def run_wgrad(gb, kw, inp, want_db=True):
    d = lib_desc(gb, kw)
    bits = kw["dtype"] == "bf16"
    x = to_device(torch, inp["x"], inp.get("x_bits") if bits else None)
    g = to_device(torch, inp["g"], inp.get("g_bits") if bits else None)
    _, ws, _ = gb.desc_shapes(d)
    buf, dw = _guarded(ws, torch.bfloat16 if bits else torch.float32)
    dbuf, db = _guarded((kw["c_out"],), torch.float32)
    need = gb.gbconv_bwd_filter_workspace(d)
    # the workspace starts as garbage: every partial the reduction reads must have been written
    wsp = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    gb.conv_bwd_filter(d, x, g, dw=dw, db=db if want_db else None, workspace=wsp)
    gb.device_status()
    assert _guards_intact(buf), "kernel wrote outside dw"
    assert _guards_intact(dbuf), "kernel wrote outside db"
    return to_host_f64(torch, dw), to_host_f64(torch, db)


# (shape, expected kernel family)
WGRAD = [
    # generic CUDA-core path: fp32 NCL conv1d (the conv1d workload's shape), grouped / strided / dilated
    # NCHW fp32, NHWC fp32 with OIHW weights, depthwise bf16, NCHW bf16
    (shape_kw(spatial_dims=1, n=2, in_size=(32,), c_in=4, c_out=8, k=(3,), stride=(1,), pad=(2,), dil=(2,),
              layout="ncl", wlayout="oik", dtype="f32"), "direct_wgrad"),
    (shape_kw(n=2, in_size=(11, 9), c_in=6, c_out=9, groups=3, k=(3, 2), stride=(2, 1), pad=(1, 0), dil=(1, 2),
              layout="nchw", wlayout="oihw", dtype="f32"), "direct_wgrad"),
    (shape_kw(n=3, in_size=(10, 12), c_in=16, c_out=8, wlayout="oihw", dtype="f32", stride=(2, 2)), "direct_wgrad"),
    (shape_kw(n=2, in_size=(14, 15), c_in=64, c_out=64, groups=64, stride=(2, 2)), "direct_wgrad"),
    (shape_kw(n=1, in_size=(9, 8), c_in=16, c_out=8, layout="nchw", wlayout="oihw", stride=(2, 2)), "direct_wgrad"),
    # NHWC bf16 that the tensor-core path declines: a 5-wide kernel, five kernel rows in one stride phase
    (shape_kw(n=1, in_size=(13, 12), c_in=16, c_out=24, k=(5, 5), pad=(2, 2), dil=(1, 2)), "direct_wgrad"),
    (shape_kw(n=1, in_size=(15, 14), c_in=16, c_out=24, k=(5, 3), pad=(4, 1), dil=(2, 1), stride=(2, 1)),
     "direct_wgrad"),
    # tensor-core path at H/W strides: one unit per stride phase, x through a strided view.  1x1 s2;
    # 3x3 s2 with odd extents; 7x7 s2 (four phases of up to four kernel rows, input-channel tail);
    # (2, 1) strides; stride 3 (nine one-tap phases); dilation 2 at stride 2 (every kernel row in one
    # phase); (begin, end) padding at stride 2; 3-D at H/W stride 2
    (shape_kw(n=2, in_size=(15, 14), c_in=32, c_out=48, k=(1, 1), pad=(0, 0), stride=(2, 2)), "wgrad"),
    (shape_kw(n=2, in_size=(15, 14), c_in=64, c_out=128, k=(3, 3), pad=(1, 1), stride=(2, 2)), "wgrad"),
    # two output blocks per unit (x loaded once for both), the second block 32 channels wide, two input blocks
    (shape_kw(n=3, in_size=(30, 29), c_in=128, c_out=96, k=(3, 3), pad=(1, 1), stride=(2, 2)), "wgrad"),
    (shape_kw(n=1, in_size=(21, 20), c_in=24, c_out=64, k=(7, 7), pad=(3, 3), stride=(2, 2)), "wgrad"),
    (shape_kw(n=2, in_size=(12, 11), c_in=64, c_out=64, k=(3, 3), pad=(1, 1), stride=(2, 1)), "wgrad"),
    (shape_kw(n=2, in_size=(13, 14), c_in=64, c_out=64, k=(3, 3), pad=(1, 1), stride=(3, 3)), "wgrad"),
    (shape_kw(n=2, in_size=(16, 15), c_in=64, c_out=64, k=(3, 3), pad=(2, 2), dil=(2, 2), stride=(2, 2)), "wgrad"),
    (shape_kw(n=2, in_size=(14, 13), c_in=64, c_out=64, k=(3, 3), pad=(1, 0), pad_end=(0, 1), stride=(2, 2)),
     "wgrad"),
    # tensor-core path: 3x3 over several chunks; channel tails and four block pairs; 2x2 without
    # padding; 1x1 (one kernel row: the second M atom unused); 3x1; dilation 2; conv1d NLC; 16 channels
    (shape_kw(n=4, in_size=(20, 21), c_in=64, c_out=64, k=(3, 3), pad=(1, 1)), "wgrad"),
    (shape_kw(n=2, in_size=(16, 17), c_in=128, c_out=96, k=(3, 3), pad=(1, 1)), "wgrad"),
    (shape_kw(n=3, in_size=(11, 10), c_in=64, c_out=128, k=(2, 2), pad=(0, 0)), "wgrad"),
    (shape_kw(n=2, in_size=(9, 13), c_in=256, c_out=64, k=(1, 1), pad=(0, 0)), "wgrad"),
    (shape_kw(n=2, in_size=(12, 9), c_in=64, c_out=64, k=(3, 1), pad=(1, 0)), "wgrad"),
    (shape_kw(n=2, in_size=(14, 15), c_in=64, c_out=64, k=(3, 3), pad=(2, 2), dil=(2, 2)), "wgrad"),
    (shape_kw(spatial_dims=1, n=3, in_size=(37,), c_in=32, c_out=64, k=(3,), stride=(1,), pad=(2,), dil=(2,),
              layout="nlc", wlayout="oki"), "wgrad"),
    (shape_kw(n=2, in_size=(7, 8), c_in=16, c_out=8, k=(3, 3), pad=(1, 1)), "wgrad"),
    # (begin, end) padding on both weight-gradient paths
    (shape_kw(n=2, in_size=(11, 12), c_in=64, c_out=64, pad=(0, 1), pad_end=(2, 0)), "wgrad"),
    (shape_kw(n=2, in_size=(9, 10), c_in=6, c_out=9, groups=3, stride=(2, 1), pad=(1, 0), pad_end=(0, 1),
              layout="nchw", wlayout="oihw", dtype="f32"), "direct_wgrad"),
    # 3-D: the generic path (fp32 NCDHW with groups), and the tensor-core path (an H/W stride too), one
    # kernel-depth tap per unit over (batch, depth) slices: depth strides (with depth dilation and
    # (begin, end) depth padding); 3x3x3; depth dilation with (begin, end) depth padding and 128
    # output channels; a depth-2 kernel over six block pairs; a depth-1 kernel with depth padding;
    # 16 input channels; and a depth-1 kernel over N*D images
    (shape_kw(spatial_dims=3, n=2, in_size=(5, 6, 7), c_in=4, c_out=6, groups=2, k=(3, 2, 3), stride=(2, 1, 2),
              pad=(1, 0, 1), dil=(1, 2, 1), layout="ncdhw", wlayout="oidhw", dtype="f32"), "direct_wgrad"),
    (shape_kw(spatial_dims=3, n=1, in_size=(5, 6, 7), c_in=64, c_out=64, k=(3, 3, 3), stride=(1, 2, 2),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "wgrad"),
    (shape_kw(spatial_dims=3, n=1, in_size=(5, 6, 7), c_in=64, c_out=64, k=(3, 3, 3), stride=(2, 1, 1),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "wgrad"),
    (shape_kw(spatial_dims=3, n=2, in_size=(7, 6, 5), c_in=64, c_out=64, k=(3, 3, 3), stride=(2, 1, 1),
              pad=(2, 1, 1), pad_end=(1, 1, 1), dil=(2, 1, 1), layout="ndhwc", wlayout="odhwi"), "wgrad"),
    (shape_kw(spatial_dims=3, n=1, in_size=(4, 6, 5), c_in=16, c_out=8, k=(3, 3, 3), stride=(1, 1, 1),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "wgrad"),
    (shape_kw(spatial_dims=3, n=2, in_size=(4, 9, 11), c_in=64, c_out=64, k=(3, 3, 3), stride=(1, 1, 1),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "wgrad"),
    (shape_kw(spatial_dims=3, n=1, in_size=(6, 10, 9), c_in=64, c_out=128, k=(3, 3, 3), stride=(1, 1, 1),
              pad=(2, 1, 1), pad_end=(0, 1, 1), dil=(2, 1, 1), layout="ndhwc", wlayout="odhwi"), "wgrad"),
    (shape_kw(spatial_dims=3, n=1, in_size=(3, 6, 7), c_in=128, c_out=192, k=(2, 2, 3), stride=(1, 1, 1),
              pad=(0, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "wgrad"),
    (shape_kw(spatial_dims=3, n=2, in_size=(3, 7, 6), c_in=64, c_out=64, k=(1, 3, 3), stride=(1, 1, 1),
              pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "wgrad"),
    (shape_kw(spatial_dims=3, n=2, in_size=(3, 9, 11), c_in=64, c_out=64, k=(1, 3, 3), stride=(1, 1, 1),
              pad=(0, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi"), "wgrad"),
    # more block pairs than SMs: CTAs take several units in turn (the accumulators are handed over)
    (shape_kw(n=1, in_size=(6, 6), c_in=1024, c_out=1024, k=(3, 3), pad=(1, 1)), "wgrad"),
]


def _wgrad_ids():
    return ["%s-%d" % (fam, i) for i, (_, fam) in enumerate(WGRAD)]


@pytest.mark.parametrize("case", range(len(WGRAD)), ids=_wgrad_ids())
def test_wgrad_matches_oracle(gb, case):
    kw, family = WGRAD[case]
    d = lib_desc(gb, kw)
    assert gb.gbconv_select(d, gb.GBCONV_OP_BWD_FILTER) == family
    c = oracle_conv(kw)
    inp = draw_wgrad(c, kw["dtype"], 700 + case)
    dw, db = run_wgrad(gb, kw, inp)
    ref = oracle.conv_wgrad(c, inp["x"], inp["g"])
    scale = oracle.conv_wgrad(c, np.abs(inp["x"]), np.abs(inp["g"]))
    assert dw.shape == ref.shape
    if kw["dtype"] == "f32":
        check_f32(dw, ref, scale)
    else:
        check_bf16(dw, ref, scale)
    # the bias gradient is always float32
    check_f32(db, oracle.conv_bgrad(c, inp["g"]), oracle.conv_bgrad(c, np.abs(inp["g"])))


@pytest.mark.parametrize("case", range(len(WGRAD)), ids=_wgrad_ids())
def test_wgrad_integer_inputs_bit_exact(gb, case):
    kw, _ = WGRAD[case]
    c = oracle_conv(kw)
    inp = draw_wgrad(c, kw["dtype"], 800 + case, kind="int")
    dw, db = run_wgrad(gb, kw, inp)
    ref = oracle.conv_wgrad(c, inp["x"], inp["g"])
    if kw["dtype"] == "bf16":
        ref = bf16_round(ref)
    np.testing.assert_array_equal(dw, ref)
    np.testing.assert_array_equal(db, oracle.conv_bgrad(c, inp["g"]))


def test_wgrad_is_deterministic_and_db_optional(gb):
    kw, _ = WGRAD[7]
    c = oracle_conv(kw)
    inp = draw_wgrad(c, "bf16", 900)
    dw1, db1 = run_wgrad(gb, kw, inp)
    dw2, db2 = run_wgrad(gb, kw, inp)
    dw3, db3 = run_wgrad(gb, kw, inp, want_db=False)
    assert np.array_equal(dw1, dw2) and np.array_equal(db1, db2)
    assert np.array_equal(dw1, dw3)
    assert np.all(db3 == 7.0)  # not asked for: untouched


def test_wgrad_tc_chunks_longer_than_one_load(gb):
    # 8 images of 120x120: 64-row-wide boxes hold one block of 4 rows per load, and the row blocks
    # outnumber the chunks, so CTAs sweep several segments; checked on every dW element
    kw = shape_kw(n=8, in_size=(120, 120), c_in=64, c_out=64, k=(3, 3), pad=(1, 1))
    d = lib_desc(gb, kw)
    assert gb.gbconv_select(d, gb.GBCONV_OP_BWD_FILTER) == "wgrad"
    plan = dict(f.split("=") for f in gb.gbconv_describe(d, gb.GBCONV_OP_BWD_FILTER).split()[1:])
    assert int(plan["seg_blocks"]) == 1 and int(plan["chunks"]) < 8 * 30
    c = oracle_conv(kw)
    inp = draw_wgrad(c, "bf16", 950)
    dw, db = run_wgrad(gb, kw, inp)
    ref = oracle_whole(c, "wgrad", inp["x"], inp["g"])
    scale = oracle_whole(c, "wgrad", np.abs(inp["x"]), np.abs(inp["g"]))
    check_bf16(dw, ref, scale)
    check_f32(db, oracle.conv_bgrad(c, inp["g"]), oracle.conv_bgrad(c, np.abs(inp["g"])))
