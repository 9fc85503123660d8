"""Host-side checks of the C ABI that need no GPU.

The library is built here (nvcc cross-compiles for sm_103a), loaded through
ctypes, and checked for: every function include/gbconv.h declares is
exported; output sizes agree with the oracle; invalid shapes and arguments are
rejected before anything is launched; the kernel family chosen per workload.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from synth.workloads import BY_NAME, EXTRA_WORKLOADS, WORKLOADS
from tests.helpers import lib_desc, oracle_conv, shape_kw

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gb():
    import __graft_entry__
    __graft_entry__.build()
    import convolution_conv_fwd_gb300 as gb
    return gb


def declared_functions():
    text = open(os.path.join(ROOT, "include", "gbconv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gbconv_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_function_is_exported(gb):
    names = declared_functions()
    assert len(names) >= 8
    for name in names:
        assert hasattr(gb._lib, name), name
    assert set(names) == set(gb.EXPORTS)


@pytest.mark.parametrize("kw", [
    shape_kw(),
    shape_kw(in_size=(112, 112), c_in=256, c_out=256, groups=256, stride=(2, 2)),
    shape_kw(in_size=(63, 64), stride=(2, 2), k=(3, 3), pad=(1, 1)),
    shape_kw(in_size=(10, 7), k=(4, 2), stride=(3, 2), pad=(2, 0), dil=(3, 2)),
    shape_kw(spatial_dims=1, in_size=(32,), k=(3,), stride=(1,), pad=(2,), dil=(2,), layout="ncl", wlayout="oik",
             dtype="f32"),
    shape_kw(spatial_dims=1, in_size=(17,), k=(4,), stride=(3,), pad=(1,), dil=(2,)),
])
def test_out_shape_matches_oracle(gb, kw):
    d = lib_desc(gb, kw)
    c = oracle_conv(kw)
    oh, ow = gb.gbconv_out_shape(d)
    if kw["spatial_dims"] == 1:
        assert (oh, ow) == (c.out_hw()[1], 1)
    else:
        assert (oh, ow) == c.out_hw()


@pytest.mark.parametrize("bad", [
    dict(n=0), dict(c_in=0), dict(c_out=0), dict(groups=0), dict(groups=5), dict(stride=(0, 1)),
    dict(dil=(1, 0)), dict(k=(11, 3)), dict(in_size=(0, 8)), dict(pad=(-1, 0)),
])
def test_degenerate_shapes_rejected(gb, bad):
    kw = shape_kw(c_in=12, c_out=12, groups=2)
    kw.update(bad)
    d = lib_desc(gb, kw)
    with pytest.raises(gb.GbconvError) as e:
        gb.gbconv_out_shape(d)
    assert e.value.status == gb.GBCONV_EINVAL
    # the enqueuing entry points reject the same shape before touching the device
    assert gb.gbconv_fwd(d, 16, 16, None, 16, 0) == gb.GBCONV_EINVAL
    assert gb.gbconv_bwd_data(d, 16, 16, 16, 0) == gb.GBCONV_EINVAL
    assert not oracle.check(oracle_conv(kw))  # the oracle rejects the same shapes


def test_enum_fields_and_null_pointers_rejected(gb):
    d = lib_desc(gb, shape_kw())
    assert gb.gbconv_fwd(d, 0, 16, None, 16, 0) == gb.GBCONV_EINVAL
    assert gb.gbconv_fwd(d, 16, 0, None, 16, 0) == gb.GBCONV_EINVAL
    assert gb.gbconv_fwd(d, 16, 16, None, 0, 0) == gb.GBCONV_EINVAL
    assert gb.gbconv_bwd_data(d, 0, 16, 16, 0) == gb.GBCONV_EINVAL
    assert gb.gbconv_pack_weight(d, 0, 16, 0) == gb.GBCONV_EINVAL
    for field, value in (("spatial_dims", 4), ("spatial_dims", 0), ("layout", 7), ("wlayout", -1), ("dtype", 5)):
        d2 = lib_desc(gb, shape_kw())
        setattr(d2, field, value)
        assert gb.gbconv_fwd(d2, 16, 16, None, 16, 0) == gb.GBCONV_EINVAL


def test_index_overflow_is_unsupported(gb):
    d = lib_desc(gb, shape_kw(n=4096, in_size=(1024, 1024), c_in=64, c_out=64))
    assert gb.gbconv_fwd(d, 16, 16, None, 16, 0) == gb.GBCONV_EUNSUPPORTED
    with pytest.raises(gb.GbconvError) as e:
        gb.gbconv_out_shape(d)
    assert e.value.status == gb.GBCONV_EUNSUPPORTED


def test_status_strings(gb):
    for s in range(5):
        assert gb.status_string(s)
    assert gb.status_string(99) == "unknown status"


EXPECTED_FAMILY = {
    "conv1d_ncl_f32": {"direct"},
    "pointwise_1x1_nhwc_bf16": {"pointwise"},
    "dense3x3_nhwc_bf16": {"implicit"},
    "depthwise3x3_s2_nhwc_bf16": {"depthwise"},
    "dgrad3x3_s2_nhwc_bf16": {"dgrad"},
    "depthwise3x3_s2_dgrad_nhwc_bf16": {"depthwise_dgrad"},
    "dense3x3_s2_nhwc_bf16": {"implicit"},
    "wgrad3x3_nhwc_bf16": {"wgrad", "direct_wgrad"},
    "dense3x3x3_ndhwc_bf16": {"implicit"},
    "dgrad3x3x3_ndhwc_bf16": {"dgrad"},
    "wgrad3x3x3_ndhwc_bf16": {"wgrad"},
    "wgrad3x3_s2_nhwc_bf16": {"wgrad"},
    "smallgroup3x3_g64_nhwc_bf16": {"smallgroup"},
    "smallgroup3x3_g64_dgrad_nhwc_bf16": {"smallgroup_dgrad"},
    "grouped3x3_g2_nhwc_bf16": {"implicit"},
}

OPS = {"fwd": 0, "dgrad": 1, "wgrad": 2}


@pytest.mark.parametrize("wl", WORKLOADS + EXTRA_WORKLOADS, ids=[w.name for w in WORKLOADS + EXTRA_WORKLOADS])
def test_workload_kernel_family(gb, wl):
    d = lib_desc(gb, wl)
    assert gb.gbconv_select(d, OPS[wl.op]) in EXPECTED_FAMILY[wl.name]


def test_generic_families_for_other_layouts(gb):
    assert gb.gbconv_select(lib_desc(gb, shape_kw(layout="nchw", wlayout="oihw")), 0) == "direct"
    assert gb.gbconv_select(lib_desc(gb, shape_kw(dtype="f32")), 0) == "direct"
    assert gb.gbconv_select(lib_desc(gb, shape_kw(groups=2)), 1) == "direct_dgrad"
    # strided forwards read stride-phase views of x: the implicit GEMM (up to 9 phases, 32 taps)
    assert gb.gbconv_select(lib_desc(gb, shape_kw(stride=(2, 2))), 0) == "implicit"
    assert gb.gbconv_select(lib_desc(gb, shape_kw(stride=(2, 2), k=(7, 7), pad=(3, 3))), 0) == "direct"
    assert gb.gbconv_select(lib_desc(gb, shape_kw(stride=(2, 2), c_in=32, c_out=32)), 1) == "dgrad"
    assert gb.gbconv_select(lib_desc(gb, shape_kw(stride=(2, 2))), 1) == "dgrad"
    # channel counts that are not a multiple of 8 break the 16-byte TMA row pitch
    assert gb.gbconv_select(lib_desc(gb, shape_kw(c_in=12, c_out=12)), 1) == "direct_dgrad"
    assert gb.gbconv_select(lib_desc(gb, shape_kw(c_in=12, c_out=12)), 0) == "direct"
    # a strided 1x1 forward reads a strided TMA view: the implicit GEMM with one tap
    assert gb.gbconv_select(lib_desc(gb, shape_kw(k=(1, 1), pad=(0, 0), stride=(2, 2))), 0) == "implicit"
    assert gb.gbconv_select(lib_desc(gb, shape_kw(k=(1, 1), pad=(1, 1), stride=(2, 2))), 0) == "implicit"
    # depthwise dgrad (G = C_in = C_out, C a multiple of 8) has its own gather kernel
    assert gb.gbconv_select(lib_desc(gb, shape_kw(c_in=32, c_out=32, groups=32, stride=(2, 2))), 1) == "depthwise_dgrad"
    assert gb.gbconv_select(lib_desc(gb, shape_kw(c_in=12, c_out=12, groups=12)), 1) == "direct_dgrad"


def _plan(gb, kw_or_wl, op=0):
    text = gb.gbconv_describe(lib_desc(gb, kw_or_wl), op)
    fields = dict(f.split("=", 1) for f in text.split()[2:])
    return text.split()[0], text.split()[1], fields


def test_describe_dense_plans(gb):
    # dense 3x3 at C_out = 64: 64-wide N tiles, two 128-row sub-tiles per item on a virtual grid of
    # 56 x (56 + 2) positions per image, every (k-block, tap) weight tile resident
    fam, op, f = _plan(gb, BY_NAME["dense3x3_nhwc_bf16"])
    assert (fam, op) == ("implicit_gemm", "fwd")
    assert f["bn"] == "64" and f["nsub"] == "2" and f["taps"] == "9" and f["weights"] == "resident"
    assert int(f["items"]) == 32 * -(-56 * 58 // 256)
    assert int(f["smem"]) <= 227 * 1024
    # 1x2 kernel at dilation 3: the virtual grid pitch is OW + 3
    _, _, f = _plan(gb, shape_kw(n=1, in_size=(9, 30), c_in=64, c_out=16, k=(1, 2), pad=(0, 1), dil=(1, 3)))
    assert f["taps"] == "2" and int(f["items"]) == -(-9 * (29 + 3) // 256)
    # C_out = 192: one 192-wide tile, one sub-tile per item; C_in = 96: two k-blocks
    _, _, f = _plan(gb, shape_kw(n=2, in_size=(10, 9), c_in=96, c_out=192, k=(3, 2), pad=(1, 0)))
    assert f["bn"] == "192" and f["nsub"] == "1" and f["kb"] == "2"
    # weights too large to stay resident stream through a ring
    _, _, f = _plan(gb, shape_kw(c_in=256, c_out=128))
    assert f["weights"] == "streamed" and int(f["b_stages"]) >= 3


def test_describe_phases_sources_and_families(gb):
    _, op, f = _plan(gb, BY_NAME["dense3x3_s2_nhwc_bf16"])
    assert op == "fwd" and f["sources"] == "4" and f["taps"] == "9"
    _, op, f = _plan(gb, BY_NAME["dgrad3x3_s2_nhwc_bf16"], 1)
    assert op == "dgrad" and f["phases"] == "4" and f["taps"] == "4" and f["weights"] == "streamed"
    assert gb.gbconv_describe(lib_desc(gb, BY_NAME["depthwise3x3_s2_nhwc_bf16"]), 0) == "depthwise"
    assert gb.gbconv_describe(lib_desc(gb, BY_NAME["conv1d_ncl_f32"]), 0) == "direct"
    d = lib_desc(gb, shape_kw())
    buf = ctypes.create_string_buffer(8)
    assert gb._lib.gbconv_describe(ctypes.byref(d), 0, buf, 8) == gb.GBCONV_OK
    assert buf.value == b"implici"  # truncated to the buffer, NUL-terminated
    assert gb._lib.gbconv_describe(ctypes.byref(d), 7, buf, 8) == gb.GBCONV_EINVAL
    assert gb._lib.gbconv_describe(ctypes.byref(d), 0, None, 8) == gb.GBCONV_EINVAL
    assert gb._lib.gbconv_describe(ctypes.byref(d), 0, buf, 0) == gb.GBCONV_EINVAL


def test_bwd_filter_workspace_and_argument_checks(gb):
    d = lib_desc(gb, shape_kw(n=2, in_size=(9, 7), c_in=16, c_out=8))
    need = gb.gbconv_bwd_filter_workspace(d)
    assert need > 0 and need % 256 == 0
    # every family the weight gradient can take, for shapes the forward accepts
    assert gb.gbconv_select(d, gb.GBCONV_OP_BWD_FILTER) in ("wgrad", "direct_wgrad")
    assert gb.gbconv_select(lib_desc(gb, shape_kw(layout="nchw", wlayout="oihw", dtype="f32")), 2) == "direct_wgrad"
    assert gb.gbconv_select(lib_desc(gb, shape_kw(groups=2)), 2) == "direct_wgrad"
    assert gb.gbconv_describe(lib_desc(gb, shape_kw(groups=2)), 2) == "direct_wgrad"
    # argument errors come back before anything touches a device
    fake = 1 << 20  # never dereferenced: the calls below fail their checks first
    assert gb.gbconv_bwd_filter(d, None, fake, fake, None, fake, need, None) == gb.GBCONV_EINVAL
    assert gb.gbconv_bwd_filter(d, fake, None, fake, None, fake, need, None) == gb.GBCONV_EINVAL
    assert gb.gbconv_bwd_filter(d, fake, fake, None, None, fake, need, None) == gb.GBCONV_EINVAL
    assert gb.gbconv_bwd_filter(d, fake, fake, fake, None, fake, need - 256, None) == gb.GBCONV_EINVAL
    assert gb.gbconv_bwd_filter(d, fake, fake, fake, None, None, need, None) == gb.GBCONV_EINVAL
    assert gb.gbconv_bwd_filter(d, fake, fake, fake, None, fake + 4, need, None) == gb.GBCONV_EINVAL
    bad = lib_desc(gb, shape_kw(k=(40, 3)))
    b = ctypes.c_int64(0)
    assert gb._lib.gbconv_bwd_filter_workspace(ctypes.byref(bad), ctypes.byref(b)) == gb.GBCONV_EINVAL
    assert gb._lib.gbconv_bwd_filter_workspace(ctypes.byref(d), None) == gb.GBCONV_EINVAL
    k = ctypes.c_int32(-1)
    assert gb._lib.gbconv_select(ctypes.byref(d), 3, ctypes.byref(k)) == gb.GBCONV_EINVAL


def test_host_staging_bytes_and_argument_checks(gb):
    """The host-buffer calls' staging buffer holds the weight, the bias, the whole source batch and the
    whole result batch, each rounded up to 256 bytes; argument errors come back before any CUDA call."""
    kw = shape_kw(n=2, in_size=(9, 7), c_in=16, c_out=8)
    d = lib_desc(gb, kw)
    c = oracle_conv(kw)
    r256 = lambda b: (b + 255) // 256 * 256
    nbytes = lambda shape: 2 * int(np.prod(shape))
    x_b, y_b, w_b = nbytes(c.x_shape()), nbytes(c.y_shape()), nbytes(c.w_shape())
    assert gb.gbconv_host_staging_bytes(d, gb.GBCONV_OP_FWD) == r256(w_b) + r256(x_b) + r256(y_b)
    assert gb.gbconv_host_staging_bytes(d, gb.GBCONV_OP_FWD, True) == r256(w_b) + r256(4 * 8) + r256(x_b) + r256(y_b)
    assert gb.gbconv_host_staging_bytes(d, gb.GBCONV_OP_BWD_DATA) == r256(w_b) + r256(y_b) + r256(x_b)
    assert gb.gbconv_host_staging_bytes(d, gb.GBCONV_OP_BWD_DATA, True) == (r256(w_b) + r256(4 * 16) + r256(y_b) +
                                                                           r256(x_b))
    b = ctypes.c_int64(0)
    assert gb._lib.gbconv_host_staging_bytes(ctypes.byref(d), gb.GBCONV_OP_BWD_FILTER, 0,
                                             ctypes.byref(b)) == gb.GBCONV_EINVAL
    assert gb._lib.gbconv_host_staging_bytes(ctypes.byref(d), gb.GBCONV_OP_FWD, 0, None) == gb.GBCONV_EINVAL
    bad = lib_desc(gb, shape_kw(k=(40, 3)))
    assert gb._lib.gbconv_host_staging_bytes(ctypes.byref(bad), gb.GBCONV_OP_FWD, 0, ctypes.byref(b)) == gb.GBCONV_EINVAL
    need = gb.gbconv_host_staging_bytes(d, gb.GBCONV_OP_FWD)
    fake = 1 << 20  # never dereferenced: the calls below fail their checks first
    assert gb.gbconv_fwd_host(d, None, fake, None, fake, fake, need, 0, None) == gb.GBCONV_EINVAL
    assert gb.gbconv_fwd_host(d, fake, None, None, fake, fake, need, 0, None) == gb.GBCONV_EINVAL
    assert gb.gbconv_fwd_host(d, fake, fake, None, None, fake, need, 0, None) == gb.GBCONV_EINVAL
    assert gb.gbconv_fwd_host(d, fake, fake, None, fake, None, need, 0, None) == gb.GBCONV_EINVAL
    assert gb.gbconv_fwd_host(d, fake, fake, None, fake, fake, need - 1, 0, None) == gb.GBCONV_EINVAL
    assert gb.gbconv_fwd_host(d, fake, fake, None, fake, fake + 16, need, 0, None) == gb.GBCONV_EINVAL
    # with a bias the staging buffer must also hold it
    assert gb.gbconv_fwd_host(d, fake, fake, fake, fake, fake, need, 0, None) == gb.GBCONV_EINVAL
    need_dg = gb.gbconv_host_staging_bytes(d, gb.GBCONV_OP_BWD_DATA)
    assert gb.gbconv_bwd_data_host(d, fake, fake, fake, fake, need_dg - 256, 0, None) == gb.GBCONV_EINVAL
    assert gb.gbconv_conv_transpose_host(d, fake, fake, fake, fake, fake, need_dg, 0, None) == gb.GBCONV_EINVAL
    assert gb.gbconv_fwd_host(bad, fake, fake, None, fake, fake, need, 0, None) == gb.GBCONV_EINVAL


def test_describe_weight_gradient_stride_phases(gb):
    # a unit per (chunk, block pair, stride phase); each phase the unit-stride sum over its own taps
    _, _, f = _plan(gb, shape_kw(n=32, in_size=(56, 56), c_in=64, c_out=64), op=2)
    assert f["phases"] == "1" and f["groups"] == "2" and f["n"] == "192" and f["pitch"] == "58"
    assert f["out_blocks"] == "1"  # one 64-channel output block
    # 3x3 stride 2: phases {1} x {1}, {1} x {0, 2}, {0, 2} x {1}, {0, 2} x {0, 2}; the pitch is OW + 1
    _, _, f = _plan(gb, shape_kw(n=32, in_size=(56, 56), c_in=128, c_out=128, stride=(2, 2)), op=2)
    assert f["phases"] == "4" and f["groups"] == "1" and f["n"] == "128" and f["pitch"] == "29"
    # two output blocks per unit (x loaded once for both): 2 input blocks x 1 output-block pair x 4 phases
    assert f["out_blocks"] == "2"
    assert int(f["units"]) == 2 * 4 * int(f["chunks"]) and int(f["units"]) <= 152
    # 7x7 stride 2: four kernel rows and columns in the (0, 0) phase -> two groups, N = 256
    _, _, f = _plan(gb, shape_kw(n=8, in_size=(112, 112), c_in=64, c_out=64, k=(7, 7), pad=(3, 3), stride=(2, 2)), op=2)
    assert f["phases"] == "4" and f["groups"] == "2" and f["n"] == "256"
    # 1x1 stride 2: one phase, one tap
    _, _, f = _plan(gb, shape_kw(n=4, in_size=(28, 28), c_in=64, c_out=64, k=(1, 1), pad=(0, 0), stride=(2, 2)), op=2)
    assert f["phases"] == "1" and f["groups"] == "1" and f["n"] == "64"
    # 3x3 stride 3: nine one-tap phases; 2x2 stride 4: a phase per tap, twelve phases empty
    _, _, f = _plan(gb, shape_kw(n=4, in_size=(30, 30), c_in=64, c_out=64, stride=(3, 3)), op=2)
    assert f["phases"] == "9" and f["n"] == "64"
    _, _, f = _plan(gb, shape_kw(n=4, in_size=(32, 32), c_in=64, c_out=64, k=(2, 2), pad=(0, 0), stride=(4, 4)), op=2)
    assert f["phases"] == "4"
    # dilation 2 at stride 2: every kernel row in one phase, consecutive phase rows
    _, _, f = _plan(gb, shape_kw(n=4, in_size=(30, 30), c_in=64, c_out=64, pad=(2, 2), dil=(2, 2), stride=(2, 2)), op=2)
    assert f["phases"] == "1" and f["groups"] == "2" and f["n"] == "192"
    # five kernel rows in one phase, or a stride above 4: the generic kernel
    assert gb.gbconv_select(lib_desc(gb, shape_kw(k=(5, 3), pad=(4, 1), dil=(2, 1), stride=(2, 1),
                                                  c_in=64, c_out=64)), 2) == "direct_wgrad"
    assert gb.gbconv_select(lib_desc(gb, shape_kw(in_size=(30, 30), stride=(5, 5), c_in=64, c_out=64)), 2) == "direct_wgrad"


def test_begin_end_padding_shapes_and_families(gb):
    # out = (in + begin + end - eff) // stride + 1 per axis, as the oracle computes it
    cases = [shape_kw(in_size=(7, 8), k=(3, 3), stride=(2, 2), pad=(0, 1), pad_end=(1, 0)),
             shape_kw(in_size=(6, 9), k=(2, 3), pad=(1, 0), pad_end=(0, 2)),
             shape_kw(spatial_dims=1, in_size=(13,), k=(4,), stride=(3,), pad=(2,), pad_end=(0,), dil=(2,),
                      layout="nlc", wlayout="oki")]
    for kw in cases:
        c = oracle_conv(kw)
        oh, ow = c.out_hw()
        want = (ow, 1) if kw["spatial_dims"] == 1 else (oh, ow)
        assert gb.gbconv_out_shape(lib_desc(gb, kw)) == want
    # a zero-initialised descriptor pads symmetrically: pad_end is read only in (begin, end) mode
    d = lib_desc(gb, shape_kw(in_size=(8, 8), pad=(1, 1)))
    d.pad_end[0], d.pad_end[1] = 5, 5
    assert gb.gbconv_out_shape(d) == (8, 8)
    d.pad_mode = gb.GBCONV_PAD_BEGIN_END
    assert gb.gbconv_out_shape(d) == (12, 12)
    for bad_mode in (2, -1):
        d.pad_mode = bad_mode
        with pytest.raises(gb.GbconvError):
            gb.gbconv_out_shape(d)
    with pytest.raises(gb.GbconvError):
        gb.gbconv_out_shape(lib_desc(gb, shape_kw(pad=(1, 1), pad_end=(-1, 0))))
    with pytest.raises(gb.GbconvError):  # padded input shorter than the kernel
        gb.gbconv_out_shape(lib_desc(gb, shape_kw(in_size=(2, 8), k=(5, 3), pad=(1, 1), pad_end=(1, 1))))
    # families: the 1x1 GEMM and the tiled depthwise kernels take symmetric padding only
    assert gb.gbconv_select(lib_desc(gb, shape_kw(k=(1, 1), pad=(0, 0), pad_end=(1, 1), c_out=64)), 0) == "implicit"
    assert gb.gbconv_select(lib_desc(gb, shape_kw(c_in=64, c_out=64, groups=64, stride=(2, 2), pad=(0, 0),
                                                 pad_end=(1, 1))), 0) == "depthwise"
    assert gb.gbconv_select(lib_desc(gb, shape_kw(stride=(2, 2), pad=(0, 0), pad_end=(1, 1))), 1) == "dgrad"


def s3(**kw):
    """A 3-D shape_kw: triples for every per-axis field."""
    d = dict(spatial_dims=3, in_size=(4, 6, 5), k=(3, 3, 3), stride=(1, 1, 1), pad=(1, 1, 1), dil=(1, 1, 1),
             layout="ndhwc", wlayout="odhwi")
    d.update(kw)
    return shape_kw(**d)


def test_conv3d_shapes_and_families(gb):
    cases = [s3(), s3(in_size=(5, 7, 6), k=(2, 3, 1), stride=(2, 1, 3), pad=(0, 1, 0), dil=(1, 2, 1)),
             s3(in_size=(6, 5, 5), pad=(1, 0, 1), pad_end=(0, 2, 1), stride=(2, 2, 1))]
    for kw in cases:
        assert gb.gbconv_out_shape(lib_desc(gb, kw)) == oracle_conv(kw).out_hw()
        xs, ws, ys = gb.desc_shapes(lib_desc(gb, kw))
        c = oracle_conv(kw)
        assert (xs, ws, ys) == (c.x_shape(), c.w_shape(), c.y_shape())
    # a real depth kernel: the forward and the input gradient on the implicit GEMM with one activation
    # source per kernel-depth tap, the weight gradient on the tensor-core kernel one kernel-depth tap
    # per unit; depth 1, unit stride, no depth padding: the 2-D families on N*D images (channels-last only)
    assert gb.gbconv_select(lib_desc(gb, s3(c_in=64, c_out=64)), 0) == "implicit"
    _, _, f = _plan(gb, s3(n=2, in_size=(5, 6, 7), c_in=64, c_out=64, stride=(2, 1, 1)))
    od = (5 + 2 - 3) // 2 + 1
    assert f["sources"] == "3" and f["taps"] == "27" and int(f["items"]) == 2 * od * -(-6 * (7 + 2) // 256)
    assert gb.gbconv_select(lib_desc(gb, s3(c_in=64, c_out=64, stride=(1, 2, 2))), 0) == "direct"  # 12 sources
    assert gb.gbconv_select(lib_desc(gb, s3(c_in=64, c_out=64, layout="ncdhw", wlayout="oidhw")), 0) == "direct"
    assert gb.gbconv_select(lib_desc(gb, s3(c_in=64, c_out=64)), 1) == "dgrad"
    # the gradient: items over N*D dx slices, one dy source per kernel-depth tap, each with its phase's taps
    _, _, f = _plan(gb, s3(n=2, in_size=(5, 6, 7), c_in=64, c_out=64), op=1)
    assert f["phases"] == "1" and f["sources"] == "3" and f["taps"] == "27"
    assert int(f["items"]) == 2 * 5 * -(-6 * (7 + 2) // 256)
    _, _, f = _plan(gb, s3(n=1, in_size=(4, 8, 8), c_in=64, c_out=64, stride=(1, 2, 2)), op=1)
    assert f["phases"] == "4" and f["sources"] == "3" and f["taps"] == "12"
    # a depth stride splits dx into depth phases (2 x 2 x 2 strides: eight), each with the kernel-depth
    # taps that reach it
    _, _, f = _plan(gb, s3(n=1, in_size=(5, 8, 9), c_in=64, c_out=64, stride=(2, 2, 2)), op=1)
    assert f["phases"] == "8" and f["taps"] == "8"
    _, _, f = _plan(gb, s3(n=1, in_size=(7, 6, 7), c_in=64, c_out=64, stride=(3, 1, 1)), op=1)
    assert f["phases"] == "3" and f["sources"] in ("1",) and f["taps"] == "9"
    assert gb.gbconv_select(lib_desc(gb, s3(c_in=64, c_out=64, stride=(2, 1, 1))), 1) == "dgrad"
    assert gb.gbconv_select(lib_desc(gb, s3(c_in=64, c_out=64, layout="ncdhw", wlayout="oidhw")), 1) == "direct_dgrad"
    assert gb.gbconv_select(lib_desc(gb, s3(c_in=64, c_out=64)), 2) == "wgrad"
    # the weight gradient: one unit per (chunk, block pair, kernel-depth tap), about one unit per SM
    _, _, f = _plan(gb, s3(n=2, in_size=(16, 56, 56), c_in=64, c_out=64), op=2)
    assert f["depth_taps"] == "3" and int(f["units"]) == 3 * int(f["chunks"]) and int(f["units"]) <= 152
    assert gb.gbconv_select(lib_desc(gb, s3(c_in=64, c_out=64, stride=(2, 1, 1))), 2) == "wgrad"
    assert gb.gbconv_select(lib_desc(gb, s3(c_in=64, c_out=64, stride=(1, 2, 2))), 2) == "wgrad"
    assert gb.gbconv_select(lib_desc(gb, s3(c_in=64, c_out=64, layout="ncdhw", wlayout="oidhw")), 2) == "direct_wgrad"
    flat = dict(k=(1, 3, 3), pad=(0, 1, 1), c_in=64, c_out=64)
    assert gb.gbconv_select(lib_desc(gb, s3(**flat)), 0) == "implicit"
    assert gb.gbconv_select(lib_desc(gb, s3(**flat)), 1) == "dgrad"
    assert gb.gbconv_select(lib_desc(gb, s3(**flat)), 2) == "wgrad"
    assert gb.gbconv_select(lib_desc(gb, s3(**dict(flat, layout="ncdhw", wlayout="oidhw"))), 0) == "direct"
    assert gb.gbconv_select(lib_desc(gb, s3(k=(1, 1, 1), pad=(0, 0, 0), c_in=64, c_out=64)), 0) == "pointwise"
    assert gb.gbconv_select(lib_desc(gb, s3(k=(1, 3, 3), pad=(0, 1, 1), c_in=32, c_out=32, groups=32)), 0) == "depthwise"
    # depth padding with a depth-1 kernel: not a repeated 2-D convolution, one depth source at offset -1
    assert gb.gbconv_select(lib_desc(gb, s3(k=(1, 3, 3), pad=(1, 1, 1), c_in=64, c_out=64)), 0) == "implicit"
    # folded: the implicit GEMM's items count N*D images
    _, _, f = _plan(gb, s3(n=2, in_size=(3, 9, 7), **flat))
    assert int(f["items"]) == 2 * 3 * -(-9 * (7 + 2) // 256)


def test_tensors_on_different_devices_are_refused(gb):
    # the C ABI takes device pointers on the current device: one call, one device
    import types
    torch = pytest.importorskip("torch")
    a = types.SimpleNamespace(device=torch.device("cuda", 0))
    b = types.SimpleNamespace(device=torch.device("cuda", 1))
    assert gb._one_device(x=a, w=a, bias=None) == torch.device("cuda", 0)
    with pytest.raises(ValueError, match="one device"):
        gb._one_device(x=a, w=a, y=b)


@pytest.mark.parametrize("kw,fam_fwd,fam_dgrad", [
    # the small-group regime: 1 < G < C with C_in/G = C_out/G in {2, 4, 8} and whole 64-channel chunks
    (shape_kw(in_size=(16, 16), c_in=128, c_out=128, groups=32), "smallgroup", "smallgroup_dgrad"),
    (shape_kw(in_size=(16, 16), c_in=128, c_out=128, groups=16, stride=(2, 2)), "smallgroup", "smallgroup_dgrad"),
    (shape_kw(in_size=(16, 16), c_in=128, c_out=128, groups=64), "smallgroup", "smallgroup_dgrad"),
    # outside it: 16 channels per group and C_out/G != C_in/G (multiples of 8) are grouped implicit GEMMs
    # on the tensor cores; 4 -> 8 channels per group, channels not in whole 64-channel chunks, and fp32
    # take the generic kernels
    (shape_kw(in_size=(16, 16), c_in=128, c_out=128, groups=8), "implicit", "dgrad"),
    (shape_kw(in_size=(16, 16), c_in=256, c_out=512, groups=16), "implicit", "dgrad"),
    (shape_kw(in_size=(16, 16), c_in=256, c_out=512, groups=32), "direct", "direct_dgrad"),
    (shape_kw(in_size=(16, 16), c_in=128, c_out=256, groups=32), "direct", "direct_dgrad"),
    (shape_kw(in_size=(16, 16), c_in=96, c_out=96, groups=24), "direct", "direct_dgrad"),
    (shape_kw(in_size=(16, 16), c_in=128, c_out=128, groups=32, dtype="f32"), "direct", "direct_dgrad"),
])
def test_small_group_regime_selection(gb, kw, fam_fwd, fam_dgrad):
    d = lib_desc(gb, kw)
    assert gb.gbconv_select(d, 0) == fam_fwd
    assert gb.gbconv_select(d, 1) == fam_dgrad


def test_gpu_parity_cases_select_their_families(gb):
    # every GPU parity case asserts the kernel family it exercises; the choice is made on the host,
    # so a plan that no longer fits (and would silently fall back) is caught here without a GPU
    pytest.importorskip("torch")
    from tests import test_gpu_parity as t
    for kw, op, fam in t.SMALL:
        assert gb.gbconv_select(lib_desc(gb, kw), 1 if op == "dgrad" else 0) == fam, (kw, op)
    for kw, fam in t.TRANSPOSE:
        assert gb.gbconv_select(lib_desc(gb, kw), 1) == fam, kw
    for kw, fam in t.WGRAD:
        assert gb.gbconv_select(lib_desc(gb, kw), 2) == fam, kw
