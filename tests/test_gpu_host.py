"""The host-buffer entry points (gbconv_fwd_host, gbconv_bwd_data_host, gbconv_conv_transpose_host).

They move the batch through a device staging buffer in slices of consecutive images, with the copies
in and out on the library's own streams overlapping the kernels, and return once the host result is
complete.  Checked here against the oracle: the library's own choice of slices on a batch large
enough to be cut, more slices asked for than there are images (clamped), one slice, and the
bounded-wait failure path reported by the call itself.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import check_bf16, draw, lib_desc, oracle_conv, scale_dgrad, scale_fwd, shape_kw, to_host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import convolution_conv_fwd_gb300 as gb
    return gb


def _pinned(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).pin_memory()


def _staging(gb, d, op, bias):
    n = gb.gbconv_host_staging_bytes(d, op, bias)
    return torch.empty((n,), dtype=torch.uint8, device="cuda"), n


CASES = [
    # depthwise, 12 images of 56x56x128: a 9.6 MB result, which the library cuts into 4 slices
    (shape_kw(n=12, in_size=(56, 56), c_in=128, c_out=128, groups=128, bias=True), "fwd", 0),
    # dense 3x3 with bias, more slices asked for than there are images
    (shape_kw(n=3, in_size=(20, 18), c_in=64, c_out=64, bias=True), "fwd", 16),
    # strided input gradient (four stride phases), five images in three uneven slices
    (shape_kw(n=5, in_size=(18, 20), c_in=128, c_out=256, stride=(2, 2)), "dgrad", 3),
    # transposed convolution (input gradient plus a bias over C_in), one slice
    (shape_kw(n=2, in_size=(14, 15), c_in=64, c_out=64, groups=64, stride=(2, 2)), "transpose", 1),
]


@pytest.mark.parametrize("kw,op,slices", CASES, ids=["%s-s%d-%d" % (c[1], c[2], i) for i, c in enumerate(CASES)])
def test_host_entry_points_match_oracle(gb, kw, op, slices):
    d = lib_desc(gb, kw)
    c = oracle_conv(kw)
    inp = draw(c, "bf16", 4700 + slices, op="fwd" if op == "fwd" else "dgrad", bias=kw["bias"])
    w = _pinned(inp["w_bits"])
    xs, _, ys = gb.desc_shapes(d)
    stream = torch.cuda.current_stream().cuda_stream
    if op == "fwd":
        x = _pinned(inp["x_bits"])
        b = torch.from_numpy(inp["b"].astype(np.float32)).pin_memory() if "b" in inp else None
        y = torch.full(ys, 7.0, dtype=torch.bfloat16).pin_memory()
        stg, n = _staging(gb, d, gb.GBCONV_OP_FWD, b is not None)
        st = gb.gbconv_fwd_host(d, x.data_ptr(), w.data_ptr(), None if b is None else b.data_ptr(), y.data_ptr(),
                                stg.data_ptr(), n, slices, stream)
        ref = oracle.conv_fwd(c, inp["x"], inp["w"], inp.get("b"))
        scale = scale_fwd(c, inp["x"], inp["w"], inp.get("b"))
    elif op == "dgrad":
        g = _pinned(inp["g_bits"])
        y = torch.full(xs, 7.0, dtype=torch.bfloat16).pin_memory()
        stg, n = _staging(gb, d, gb.GBCONV_OP_BWD_DATA, False)
        st = gb.gbconv_bwd_data_host(d, g.data_ptr(), w.data_ptr(), y.data_ptr(), stg.data_ptr(), n, slices, stream)
        ref = oracle.conv_dgrad(c, inp["g"], inp["w"])
        scale = scale_dgrad(c, inp["g"], inp["w"])
    else:
        g = _pinned(inp["g_bits"])
        bias = synth.normal(4790, (kw["c_in"],), 0.5).astype(np.float32)
        y = torch.full(xs, 7.0, dtype=torch.bfloat16).pin_memory()
        stg, n = _staging(gb, d, gb.GBCONV_OP_BWD_DATA, True)
        bt = _keep(bias)
        st = gb.gbconv_conv_transpose_host(d, g.data_ptr(), w.data_ptr(), bt.data_ptr(), y.data_ptr(), stg.data_ptr(),
                                           n, slices, stream)
        ref = oracle.conv_transpose(c, inp["g"], inp["w"], bias)
        scale = oracle.conv_transpose(c, np.abs(inp["g"]), np.abs(inp["w"]), np.abs(bias))
    assert st == gb.GBCONV_OK
    # the call is synchronous: the host result is complete without any further synchronisation
    check_bf16(to_host_f64(torch, y), ref, scale)


_kept = []


def _keep(arr):
    """A pinned host copy of arr that outlives the call."""
    t = torch.from_numpy(np.ascontiguousarray(arr)).pin_memory()
    _kept.append(t)
    return t


def test_host_call_reports_an_expired_wait(gb):
    """A wait bound far below one work item's time: the host call itself returns GBCONV_ETIMEOUT (and
    clears the record), and the next call, at the normal bound, is correct."""
    kw = shape_kw(n=4, in_size=(56, 56), c_in=256, c_out=64, bias=True)  # long reductions, as in the device test
    d = lib_desc(gb, kw)
    assert gb.gbconv_select(d, gb.GBCONV_OP_FWD) == "implicit"
    c = oracle_conv(kw)
    inp = draw(c, "bf16", 4795, op="fwd", bias=True)
    x, w = _pinned(inp["x_bits"]), _pinned(inp["w_bits"])
    b = _keep(inp["b"].astype(np.float32))
    _, _, ys = gb.desc_shapes(d)
    y = torch.full(ys, 7.0, dtype=torch.bfloat16).pin_memory()
    stg, n = _staging(gb, d, gb.GBCONV_OP_FWD, True)
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        return gb.gbconv_fwd_host(d, x.data_ptr(), w.data_ptr(), b.data_ptr(), y.data_ptr(), stg.data_ptr(), n, 1,
                                  stream)

    assert gb.gbconv_device_status(stream) == gb.GBCONV_OK
    prev = gb.gbconv_set_wait_limit_ns(1000)  # 1 us
    try:
        assert call() == gb.GBCONV_ETIMEOUT
    finally:
        gb.gbconv_set_wait_limit_ns(prev)
    assert gb.gbconv_device_status(stream) == gb.GBCONV_OK  # the call cleared the record
    y.fill_(7.0)
    assert call() == gb.GBCONV_OK
    check_bf16(to_host_f64(torch, y), oracle.conv_fwd(c, inp["x"], inp["w"], inp["b"]),
               scale_fwd(c, inp["x"], inp["w"], inp["b"]))


def test_async_calls_in_flight_together(gb):
    """The public async calls: every case above enqueued at once, each with its own staging buffer
    and completion event, then waited on; each result against the oracle.  The copies of the calls
    share the library's two copy streams, in call order."""
    pending = []
    for i, (kw, op, _) in enumerate(CASES):
        d = lib_desc(gb, kw)
        c = oracle_conv(kw)
        inp = draw(c, "bf16", 4800 + i, op="fwd" if op == "fwd" else "dgrad", bias=kw["bias"])
        w = _pinned(inp["w_bits"])
        if op == "fwd":
            b = _keep(inp["b"].astype(np.float32)) if "b" in inp else None
            call = gb.conv_fwd_async(d, _pinned(inp["x_bits"]), w, b)
            ref = oracle.conv_fwd(c, inp["x"], inp["w"], inp.get("b"))
            scale = scale_fwd(c, inp["x"], inp["w"], inp.get("b"))
        elif op == "dgrad":
            call = gb.conv_bwd_data_async(d, _pinned(inp["g_bits"]), w)
            ref = oracle.conv_dgrad(c, inp["g"], inp["w"])
            scale = scale_dgrad(c, inp["g"], inp["w"])
        else:
            bias = synth.normal(4890 + i, (kw["c_in"],), 0.5).astype(np.float32)
            call = gb.conv_transpose_async(d, _pinned(inp["g_bits"]), w, _keep(bias))
            ref = oracle.conv_transpose(c, inp["g"], inp["w"], bias)
            scale = oracle.conv_transpose(c, np.abs(inp["g"]), np.abs(inp["w"]), np.abs(bias))
        pending.append((call, ref, scale))
    for call, ref, scale in pending:
        got = call.wait()
        assert call.done() and not got.is_cuda
        check_bf16(to_host_f64(torch, got), ref, scale)
    assert gb.gbconv_device_status(torch.cuda.current_stream().cuda_stream) == gb.GBCONV_OK


def test_pageable_buffers_given_output_and_3d(gb):
    """Host tensors that are not page-locked (the copies then do not overlap, but the results are the
    same), a caller-given result tensor, and a 3-D shape, through the public calls."""
    kw = shape_kw(spatial_dims=3, n=3, in_size=(4, 9, 11), c_in=64, c_out=64, k=(3, 3, 3), stride=(1, 1, 1),
                  pad=(1, 1, 1), dil=(1, 1, 1), layout="ndhwc", wlayout="odhwi", bias=True)
    d = lib_desc(gb, kw)
    c = oracle_conv(kw)
    inp = draw(c, "bf16", 4900, op="fwd", bias=True)
    x = torch.from_numpy(np.ascontiguousarray(inp["x_bits"]).view(np.int16)).view(torch.bfloat16)  # pageable
    w = torch.from_numpy(np.ascontiguousarray(inp["w_bits"]).view(np.int16)).view(torch.bfloat16)
    b = torch.from_numpy(inp["b"].astype(np.float32))
    _, _, ys = gb.desc_shapes(d)
    y = torch.full(ys, 7.0, dtype=torch.bfloat16)  # pageable, given by the caller
    assert not x.is_pinned() and not y.is_pinned()
    ref = oracle.conv_fwd(c, inp["x"], inp["w"], inp["b"])
    scale = scale_fwd(c, inp["x"], inp["w"], inp["b"])
    got = gb.conv_fwd(d, x, w, b, y)
    assert got is y
    check_bf16(to_host_f64(torch, y), ref, scale)
    y.fill_(7.0)
    call = gb.conv_fwd_async(d, x, w, b, y)
    assert call.wait() is y
    check_bf16(to_host_f64(torch, y), ref, scale)
    # its input gradient through the synchronous host call, four slices of three images
    g = draw(c, "bf16", 4901, op="dgrad")
    dy = torch.from_numpy(np.ascontiguousarray(g["g_bits"]).view(np.int16)).view(torch.bfloat16)
    xs, _, _ = gb.desc_shapes(d)
    dx = torch.empty(xs, dtype=torch.bfloat16)
    stg, n = _staging(gb, d, gb.GBCONV_OP_BWD_DATA, False)
    w2 = torch.from_numpy(np.ascontiguousarray(g["w_bits"]).view(np.int16)).view(torch.bfloat16)
    assert gb.gbconv_bwd_data_host(d, dy.data_ptr(), w2.data_ptr(), dx.data_ptr(), stg.data_ptr(), n, 4,
                                   torch.cuda.current_stream().cuda_stream) == gb.GBCONV_OK
    check_bf16(to_host_f64(torch, dx), oracle.conv_dgrad(c, g["g"], g["w"]), scale_dgrad(c, g["g"], g["w"]))


def test_host_call_errors_raise(gb):
    """Argument errors of the host calls come back as exceptions before anything is enqueued."""
    kw = shape_kw(n=2, in_size=(9, 7), c_in=64, c_out=64)
    d = lib_desc(gb, kw)
    xs, ws, ys = gb.desc_shapes(d)
    x = torch.zeros(xs, dtype=torch.bfloat16).pin_memory()
    w = torch.zeros(ws, dtype=torch.bfloat16).pin_memory()
    with pytest.raises(ValueError):
        gb.conv_fwd_async(d, torch.zeros((1, 2, 3, 4), dtype=torch.bfloat16), w)  # wrong shape
    with pytest.raises(ValueError):
        gb.conv_fwd_async(d, x, w, y=torch.zeros((1,), dtype=torch.bfloat16))  # wrong result shape
    stg, n = _staging(gb, d, gb.GBCONV_OP_FWD, False)
    st = torch.cuda.current_stream().cuda_stream
    y = torch.empty(ys, dtype=torch.bfloat16).pin_memory()
    assert gb.gbconv_fwd_host(d, x.data_ptr(), w.data_ptr(), None, y.data_ptr(), stg.data_ptr(), n - 256, 0,
                              st) == gb.GBCONV_EINVAL
    assert gb.gbconv_fwd_host(d, x.data_ptr(), w.data_ptr(), None, y.data_ptr(), stg.data_ptr() + 128, n, 0,
                              st) == gb.GBCONV_EINVAL
    assert gb.gbconv_device_status(st) == gb.GBCONV_OK
