"""The weight gradient for callers that cannot allocate device memory.

gbconv_bwd_filter_noalloc serves callers that have no way to hand the library a workspace (code
running inside an allocator's callbacks, a plugin that only receives its tensors, an application
that reserves all device memory up front): its partial sums live in a fixed array the library
declares in device global memory.  These tests call it through the C ABI and check, on two calls in
a row per shape, that it gives what gbconv_bwd_filter gives with a caller-owned workspace, within
the parity bars the other GPU tests use (and, since both run the same kernels in the same order,
bit for bit).  A shape whose workspace exceeds the array is refused before anything is launched.

The file sorts last, so a run that stops at its first failure has run every other test already.
"""
import numpy as np
import pytest

import synth
from tests.helpers import check_bf16, check_f32, lib_desc, oracle_conv, shape_kw, to_device, to_host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import convolution_conv_fwd_gb300 as gb
    return gb


# (shape, expected weight-gradient family)
SHAPES = [
    # tensor-core partial sums over ~100 chunks: about half the static array
    (shape_kw(n=8, in_size=(56, 56), c_in=64, c_out=64, k=(3, 3), pad=(1, 1)), "wgrad"),
    # the generic CUDA-core path: fp32, NCHW, grouped, strided, dilated
    (shape_kw(n=3, in_size=(17, 15), c_in=12, c_out=18, groups=3, k=(3, 2), stride=(2, 1), pad=(1, 0), dil=(1, 2),
              layout="nchw", wlayout="oihw", dtype="f32"), "direct_wgrad"),
]


def _inputs(kw, seed):
    c = oracle_conv(kw)
    bits = kw["dtype"] == "bf16"
    out = {}
    for i, (name, shape) in enumerate((("x", c.x_shape()), ("g", c.y_shape()))):
        v = synth.normal(seed * 16 + i, shape, 1.0)
        if bits:
            b, f = synth.as_bf16(v)
            out[name] = to_device(torch, f, b)
        else:
            out[name] = to_device(torch, v.astype(np.float32))
    return out


def _run(gb, kw, inp, noalloc):
    d = lib_desc(gb, kw)
    dt = torch.bfloat16 if kw["dtype"] == "bf16" else torch.float32
    _, ws_shape, _ = gb.desc_shapes(d)
    dw = torch.full(ws_shape, 7.0, dtype=dt, device="cuda")
    db = torch.full((kw["c_out"],), 7.0, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    if noalloc:
        st = gb.gbconv_bwd_filter_noalloc(d, inp["x"].data_ptr(), inp["g"].data_ptr(), dw.data_ptr(), db.data_ptr(),
                                          stream)
    else:
        need = gb.gbconv_bwd_filter_workspace(d)
        wsp = torch.empty((max(need, 1),), dtype=torch.uint8, device="cuda")
        st = gb.gbconv_bwd_filter(d, inp["x"].data_ptr(), inp["g"].data_ptr(), dw.data_ptr(), db.data_ptr(),
                                  wsp.data_ptr(), wsp.numel(), stream)
    assert st == gb.GBCONV_OK, gb.status_string(st)
    assert gb.gbconv_device_status(stream) == gb.GBCONV_OK
    return to_host_f64(torch, dw), to_host_f64(torch, db)


def _same(kw, got, ref):
    """got within the parity bar of ref (the other tests' bars), and bitwise equal."""
    for g, r in zip(got, ref):
        scale = np.abs(r)
        if kw["dtype"] == "bf16":
            check_bf16(g, r, scale)
        else:
            check_f32(g, r, scale)
        assert np.array_equal(g, r)


def test_noalloc_matches_workspace_call_twice_in_a_row(gb):
    refs, inps = [], []
    for i, (kw, family) in enumerate(SHAPES):
        assert gb.gbconv_select(lib_desc(gb, kw), gb.GBCONV_OP_BWD_FILTER) == family
        assert gb.gbconv_bwd_filter_workspace(lib_desc(gb, kw)) <= gb.NOALLOC_WORKSPACE_BYTES
        inp = _inputs(kw, 4100 + i)
        ref = _run(gb, kw, inp, noalloc=False)
        assert np.isfinite(ref[0]).all() and np.isfinite(ref[1]).all()
        for _ in range(2):  # two calls in a row; the second starts from the first one's leftovers
            _same(kw, _run(gb, kw, inp, noalloc=True), ref)
        refs.append(ref)
        inps.append(inp)
    # the first shape again, after the other shape has overwritten part of the array
    _same(SHAPES[0][0], _run(gb, SHAPES[0][0], inps[0], noalloc=True), refs[0])


def test_noalloc_refuses_shapes_beyond_its_array(gb):
    # fp32 NCHW 3x3, C 256 -> 256 on 128x128: the generic path needs 64 chunks of 590k partial sums
    kw = shape_kw(n=1, in_size=(128, 128), c_in=256, c_out=256, layout="nchw", wlayout="oihw", dtype="f32")
    d = lib_desc(gb, kw)
    assert gb.gbconv_bwd_filter_workspace(d) > gb.NOALLOC_WORKSPACE_BYTES
    inp = _inputs(kw, 4200)
    _, ws_shape, _ = gb.desc_shapes(d)
    dw = torch.zeros(ws_shape, dtype=torch.float32, device="cuda")
    before = gb.gbconv_kernels_launched()
    st = gb.gbconv_bwd_filter_noalloc(d, inp["x"].data_ptr(), inp["g"].data_ptr(), dw.data_ptr(), None,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == gb.GBCONV_EUNSUPPORTED
    assert gb.gbconv_kernels_launched() == before
