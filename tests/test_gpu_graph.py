"""CUDA-graph capture of the library's calls.

A serving loop can replay a fixed sequence of kernels as one CUDA graph instead of enqueuing them call
by call.  The C entry points do their host work (validation, planning, tensor-map encoding) at the call
and only enqueue kernels on the stream they are given, so a call made while that stream is being
captured becomes part of the graph, with its pointers fixed.  Each test makes one call outside any
capture (the first call on a device raises the kernels' shared-memory limits, which is not a stream
operation), captures the same call, then replays the graph on new values copied into the same device
buffers and compares every replay with the oracle.
"""
import numpy as np
import pytest

import oracle
from tests.helpers import (check_bf16, check_f32, draw, lib_desc, oracle_conv, scale_dgrad, scale_fwd, shape_kw,
                           to_device, to_host_f64)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import convolution_conv_fwd_gb300 as gb
    return gb


# (shape, op, family the call must run on)
CASES = [
    (shape_kw(n=2, in_size=(20, 18), c_in=64, c_out=64, bias=True), "fwd", "implicit"),
    (shape_kw(n=2, in_size=(18, 22), c_in=128, c_out=256, stride=(2, 2)), "dgrad", "dgrad"),
    (shape_kw(n=2, in_size=(12, 10), c_in=64, c_out=128, k=(1, 1), pad=(0, 0), bias=True), "fwd", "pointwise"),
    (shape_kw(n=2, in_size=(22, 19), c_in=128, c_out=128, groups=128, stride=(2, 2)), "fwd", "depthwise"),
    (shape_kw(n=2, in_size=(22, 19), c_in=128, c_out=128, groups=128, stride=(2, 2)), "dgrad", "depthwise_dgrad"),
    (shape_kw(n=2, in_size=(14, 40), c_in=128, c_out=128, groups=32, bias=True), "fwd", "smallgroup"),
]


def _call(gb, d, op, src, w, b, out, stream):
    if op == "dgrad":
        return gb.gbconv_bwd_data(d, src.data_ptr(), w.data_ptr(), out.data_ptr(), stream)
    return gb.gbconv_fwd(d, src.data_ptr(), w.data_ptr(), None if b is None else b.data_ptr(), out.data_ptr(), stream)


@pytest.mark.parametrize("kw,op,family", CASES, ids=[f"{c[2]}-{c[1]}" for c in CASES])
def test_captured_call_replays_correctly(gb, kw, op, family):
    d = lib_desc(gb, kw)
    assert gb.gbconv_select(d, gb.GBCONV_OP_BWD_DATA if op == "dgrad" else gb.GBCONV_OP_FWD) == family
    c = oracle_conv(kw)
    key = "g" if op == "dgrad" else "x"
    inp = draw(c, "bf16", 4400, op=op, bias=kw["bias"])
    src = to_device(torch, inp[key], inp[key + "_bits"])
    w = to_device(torch, inp["w"], inp["w_bits"])
    b = to_device(torch, inp["b"]) if "b" in inp else None
    xs, _, ys = gb.desc_shapes(d)
    out = torch.empty(xs if op == "dgrad" else ys, dtype=torch.bfloat16, device="cuda")
    assert _call(gb, d, op, src, w, b, out, torch.cuda.current_stream().cuda_stream) == gb.GBCONV_OK
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    before = gb.gbconv_kernels_launched()
    with torch.cuda.graph(graph):
        st = _call(gb, d, op, src, w, b, out, torch.cuda.current_stream().cuda_stream)
    assert st == gb.GBCONV_OK
    assert gb.gbconv_kernels_launched() == before + 1  # one kernel per forward / input-gradient call
    for seed in (4401, 4402):
        new = draw(c, "bf16", seed, op=op, bias=kw["bias"])
        src.copy_(to_device(torch, new[key], new[key + "_bits"]))
        w.copy_(to_device(torch, new["w"], new["w_bits"]))
        if b is not None:
            b.copy_(to_device(torch, new["b"]))
        out.fill_(7.0)
        graph.replay()
        torch.cuda.synchronize()
        assert gb.gbconv_device_status(torch.cuda.current_stream().cuda_stream) == gb.GBCONV_OK
        got = to_host_f64(torch, out)
        if op == "dgrad":
            check_bf16(got, oracle.conv_dgrad(c, new["g"], new["w"]), scale_dgrad(c, new["g"], new["w"]))
        else:
            check_bf16(got, oracle.conv_fwd(c, new["x"], new["w"], new.get("b")),
                       scale_fwd(c, new["x"], new["w"], new.get("b")))


def test_captured_weight_gradient_replays_correctly(gb):
    """The weight gradient is two or three kernels per call (partial sums, bias partial sums, the
    ordered reduction) through a caller-owned workspace: all of them go into the graph."""
    kw = shape_kw(n=3, in_size=(20, 17), c_in=64, c_out=128)
    d = lib_desc(gb, kw)
    assert gb.gbconv_select(d, gb.GBCONV_OP_BWD_FILTER) == "wgrad"
    c = oracle_conv(kw)
    import synth
    vals = lambda seed: {name: synth.as_bf16(synth.normal(seed * 16 + i, shape, 1.0))
                         for i, (name, shape) in enumerate((("x", c.x_shape()), ("g", c.y_shape())))}
    first = vals(4410)
    x = to_device(torch, first["x"][1], first["x"][0])
    g = to_device(torch, first["g"][1], first["g"][0])
    _, ws_shape, _ = gb.desc_shapes(d)
    dw = torch.empty(ws_shape, dtype=torch.bfloat16, device="cuda")
    db = torch.empty((kw["c_out"],), dtype=torch.float32, device="cuda")
    wsp = torch.empty((gb.gbconv_bwd_filter_workspace(d),), dtype=torch.uint8, device="cuda")

    def call():
        return gb.gbconv_bwd_filter(d, x.data_ptr(), g.data_ptr(), dw.data_ptr(), db.data_ptr(), wsp.data_ptr(),
                                    wsp.numel(), torch.cuda.current_stream().cuda_stream)

    assert call() == gb.GBCONV_OK
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        assert call() == gb.GBCONV_OK
    for seed in (4411, 4412):
        new = vals(seed)
        x.copy_(to_device(torch, new["x"][1], new["x"][0]))
        g.copy_(to_device(torch, new["g"][1], new["g"][0]))
        dw.fill_(7.0)
        db.fill_(7.0)
        graph.replay()
        torch.cuda.synchronize()
        assert gb.gbconv_device_status(torch.cuda.current_stream().cuda_stream) == gb.GBCONV_OK
        xf, gf = new["x"][1], new["g"][1]
        check_bf16(to_host_f64(torch, dw), oracle.conv_wgrad(c, xf, gf), oracle.conv_wgrad(c, np.abs(xf), np.abs(gf)))
        check_f32(to_host_f64(torch, db), oracle.conv_bgrad(c, gf), oracle.conv_bgrad(c, np.abs(gf)))
