"""Calls on several streams at once.

The entry points keep no per-call state on the device besides the caller's buffers (the weight
gradient's scratch is the caller's workspace), so calls enqueued on different streams may run at the
same time.  Here five kinds of call (tensor-core forward and input gradient, depthwise, small-group,
and two weight gradients with their own workspaces) go onto four streams, interleaved and repeated
with nothing synchronised in between; every result is then compared with the oracle.
"""
import numpy as np
import pytest

import oracle
import synth
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


FWD_DGRAD = [
    (shape_kw(n=4, in_size=(20, 22), c_in=64, c_out=64, bias=True), "fwd", "implicit"),
    (shape_kw(n=3, in_size=(18, 20), c_in=128, c_out=256, stride=(2, 2)), "dgrad", "dgrad"),
    (shape_kw(n=3, in_size=(22, 19), c_in=128, c_out=128, groups=128, stride=(2, 2)), "fwd", "depthwise"),
    (shape_kw(n=2, in_size=(14, 40), c_in=128, c_out=128, groups=32, bias=True), "fwd", "smallgroup"),
]
WGRAD = [
    shape_kw(n=3, in_size=(20, 17), c_in=64, c_out=128),
    shape_kw(n=2, in_size=(16, 18), c_in=64, c_out=64, stride=(2, 2)),
]


def test_calls_on_four_streams_at_once(gb):
    streams = [torch.cuda.Stream() for _ in range(4)]
    jobs = []  # (stream index, launch callable, check callable)
    for i, (kw, op, family) in enumerate(FWD_DGRAD):
        d = lib_desc(gb, kw)
        assert gb.gbconv_select(d, gb.GBCONV_OP_BWD_DATA if op == "dgrad" else gb.GBCONV_OP_FWD) == family
        c = oracle_conv(kw)
        inp = draw(c, "bf16", 4500 + i, op=op, bias=kw["bias"])
        key = "g" if op == "dgrad" else "x"
        src = to_device(torch, inp[key], inp[key + "_bits"])
        w = to_device(torch, inp["w"], inp["w_bits"])
        b = to_device(torch, inp["b"]) if "b" in inp else None
        xs, _, ys = gb.desc_shapes(d)
        out = torch.full(xs if op == "dgrad" else ys, 7.0, dtype=torch.bfloat16, device="cuda")

        def launch(s, d=d, op=op, src=src, w=w, b=b, out=out):
            if op == "dgrad":
                return gb.gbconv_bwd_data(d, src.data_ptr(), w.data_ptr(), out.data_ptr(), s.cuda_stream)
            return gb.gbconv_fwd(d, src.data_ptr(), w.data_ptr(), None if b is None else b.data_ptr(),
                                 out.data_ptr(), s.cuda_stream)

        def check(c=c, op=op, inp=inp, out=out):
            got = to_host_f64(torch, out)
            if op == "dgrad":
                check_bf16(got, oracle.conv_dgrad(c, inp["g"], inp["w"]), scale_dgrad(c, inp["g"], inp["w"]))
            else:
                check_bf16(got, oracle.conv_fwd(c, inp["x"], inp["w"], inp.get("b")),
                           scale_fwd(c, inp["x"], inp["w"], inp.get("b")))
        jobs.append((i % 4, launch, check))
    for i, kw in enumerate(WGRAD):
        d = lib_desc(gb, kw)
        assert gb.gbconv_select(d, gb.GBCONV_OP_BWD_FILTER) == "wgrad"
        c = oracle_conv(kw)
        v = {name: synth.as_bf16(synth.normal(4600 + i * 16 + j, shape, 1.0))
             for j, (name, shape) in enumerate((("x", c.x_shape()), ("g", c.y_shape())))}
        x = to_device(torch, v["x"][1], v["x"][0])
        g = to_device(torch, v["g"][1], v["g"][0])
        _, ws_shape, _ = gb.desc_shapes(d)
        dw = torch.full(ws_shape, 7.0, dtype=torch.bfloat16, device="cuda")
        db = torch.full((kw["c_out"],), 7.0, dtype=torch.float32, device="cuda")
        wsp = torch.empty((gb.gbconv_bwd_filter_workspace(d),), dtype=torch.uint8, device="cuda")

        def launch(s, d=d, x=x, g=g, dw=dw, db=db, wsp=wsp):
            return gb.gbconv_bwd_filter(d, x.data_ptr(), g.data_ptr(), dw.data_ptr(), db.data_ptr(), wsp.data_ptr(),
                                        wsp.numel(), s.cuda_stream)

        def check(c=c, v=v, dw=dw, db=db):
            xf, gf = v["x"][1], v["g"][1]
            check_bf16(to_host_f64(torch, dw), oracle.conv_wgrad(c, xf, gf),
                       oracle.conv_wgrad(c, np.abs(xf), np.abs(gf)))
            check_f32(to_host_f64(torch, db), oracle.conv_bgrad(c, gf), oracle.conv_bgrad(c, np.abs(gf)))
        jobs.append(((i + 2) % 4, launch, check))
    torch.cuda.synchronize()
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for _ in range(3):  # each call three times, all streams running together
        for si, launch, _ in jobs:
            assert launch(streams[si]) == gb.GBCONV_OK
    for s in streams:
        assert gb.gbconv_device_status(s.cuda_stream) == gb.GBCONV_OK
    torch.cuda.synchronize()
    for _, _, check in jobs:
        check()
