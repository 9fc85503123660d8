"""The bounded-wait failure path of the tensor-core kernels, exercised on purpose without a fault.

Every barrier wait in the library's kernels is bounded; a wait that runs out makes the kernel record
GBCONV_ETIMEOUT, let its other roles stop, wait (by time only) for the copies and tensor-core
operations it already issued, free its tensor memory and return.  Here the bound is set far below
one work item's time, so the implicit-GEMM kernel's waits run out; the call must report the timeout
through gbconv_device_status, and the next call on the same stream, at the normal bound, must give
the right result.  Nothing faults, traps or spins without a bound.
"""
import numpy as np
import pytest

import oracle
from tests.helpers import check_bf16, draw, lib_desc, oracle_conv, scale_dgrad, scale_fwd, shape_kw, to_device, to_host_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import convolution_conv_fwd_gb300 as gb
    return gb


@pytest.mark.parametrize("op", ["fwd", "dgrad"])
def test_expired_wait_reports_timeout_and_the_next_call_is_correct(gb, op):
    # Long reductions (a 256- or 1024-channel k loop per tap): one work item's MMAs take well over
    # 10 us, so the epilogue's first wait, for the item's accumulator, outlasts the bound however
    # quickly the operands arrive (an L2-warm halo can land within a microsecond).
    kw = shape_kw(n=4, in_size=(56, 56), c_in=256, c_out=64, bias=(op == "fwd"))
    if op == "dgrad":
        kw = shape_kw(n=4, in_size=(48, 48), c_in=128, c_out=1024, stride=(2, 2))
    d = lib_desc(gb, kw)
    assert gb.gbconv_select(d, gb.GBCONV_OP_FWD if op == "fwd" else gb.GBCONV_OP_BWD_DATA) == (
        "implicit" if op == "fwd" else "dgrad")
    c = oracle_conv(kw)
    inp = draw(c, "bf16", 4300 + (op == "dgrad"), op=op, bias=kw["bias"])
    src = to_device(torch, inp["g" if op == "dgrad" else "x"], inp["g_bits" if op == "dgrad" else "x_bits"])
    w = to_device(torch, inp["w"], inp["w_bits"])
    b = to_device(torch, inp["b"]) if "b" in inp else None
    xs, _, ys = gb.desc_shapes(d)
    out = torch.empty(xs if op == "dgrad" else ys, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        if op == "fwd":
            return gb.gbconv_fwd(d, src.data_ptr(), w.data_ptr(), None if b is None else b.data_ptr(),
                                 out.data_ptr(), stream)
        return gb.gbconv_bwd_data(d, src.data_ptr(), w.data_ptr(), out.data_ptr(), stream)

    assert gb.gbconv_device_status(stream) == gb.GBCONV_OK  # nothing pending from earlier tests
    prev = gb.gbconv_set_wait_limit_ns(1000)  # 1 us
    try:
        assert call() == gb.GBCONV_OK  # the launch itself succeeds
        assert gb.gbconv_device_status(stream) == gb.GBCONV_ETIMEOUT
    finally:
        gb.gbconv_set_wait_limit_ns(prev)
    assert gb.gbconv_device_status(stream) == gb.GBCONV_OK  # the record was cleared
    # the same stream, the normal bound: a complete, correct result
    out.fill_(7.0)
    assert call() == gb.GBCONV_OK
    assert gb.gbconv_device_status(stream) == gb.GBCONV_OK
    got = to_host_f64(torch, out)
    if op == "fwd":
        check_bf16(got, oracle.conv_fwd(c, inp["x"], inp["w"], inp["b"]), scale_fwd(c, inp["x"], inp["w"], inp["b"]))
    else:
        check_bf16(got, oracle.conv_dgrad(c, inp["g"], inp["w"]), scale_dgrad(c, inp["g"], inp["w"]))
