"""Largest shapes: tensors just under the library's 32-bit element-index limit (2^31 - 1 elements).

Each kernel family runs once with its largest tensor at about 2.13e9 elements (4.3 GB in bf16), so any
32-bit index product that could overflow does so here.  Inputs are integer-valued (activations in
[-3, 3], weights in [-2, 2]; a seeded block tiled over the tensor): every product and partial sum is
exact in fp32, so the sampled outputs must equal the oracle rounded once to bf16, bit for bit.  The
samples are the last elements of the output, every edge and corner class and a seeded random spread;
the oracle computes them one by one (a whole oracle pass at this size would take hours).
"""
import numpy as np
import pytest

import oracle
import synth
from tests.helpers import bf16_round, lib_desc, oracle_conv, shape_kw

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if torch.cuda.get_device_properties(0).total_memory < (40 << 30):
        pytest.skip("needs about 20 GB of device memory")
    import convolution_conv_fwd_gb300 as gb
    return gb


def _tiled_ints(seed, shape, lo, hi, block=(1, 16, 16)):
    """Integer values of `shape` (N, H, W, C): a seeded (1, 16, 16, C) block tiled over the tensor."""
    bshape = tuple(block) + (shape[-1],)
    b = synth.integers(seed, bshape, lo, hi).astype(np.float32)
    reps = tuple(-(-s // t) for s, t in zip(shape[:-1], block)) + (1,)
    return np.ascontiguousarray(np.tile(b, reps)[: shape[0], : shape[1], : shape[2]])


def _bf16_dev(a):
    """Device bf16 tensor with exactly the values of `a` (small integers are exact in bf16)."""
    return torch.from_numpy(a).to("cuda").to(torch.bfloat16)


def _samples(shape4, seed, count=1500):
    """(n, c, h, w) indices of an NCHW-ordered output: the last elements of the NHWC tensor, every
    corner / edge class, and a seeded random spread."""
    n, c, h, w = shape4
    rng = synth.uniform01(seed, count * 4).reshape(count, 4)
    idx = [np.floor(rng[:, i] * m).astype(np.int64) for i, m in enumerate((n, c, h, w))]
    rows = list(zip(*idx))
    for k in range(1, 257):  # the last 256 NHWC elements: channels fastest
        flat = n * h * w * c - k
        cc, rest = flat % c, flat // c
        ww, rest = rest % w, rest // w
        hh, nn = rest % h, rest // h
        rows.append((nn, cc, hh, ww))
    for hh in (0, h // 2, h - 1):
        for ww in (0, w // 2, w - 1):
            for cc in (0, c - 1):
                rows.append((n - 1, cc, hh, ww))
                rows.append((0, cc, hh, ww))
    return np.array(rows, dtype=np.int64)


def _gather_nhwc(t, idx):
    """t[n, h, w, c] at the (n, c, h, w) rows of idx, as float64 on the host."""
    i = torch.from_numpy(idx).to(t.device)
    return t[i[:, 0], i[:, 2], i[:, 3], i[:, 1]].float().cpu().numpy().astype(np.float64)


CASES = {
    "depthwise": (shape_kw(n=127, in_size=(512, 512), c_in=64, c_out=64, groups=64), "fwd"),
    # wide images run on column strips of the implicit GEMM
    "implicit": (shape_kw(n=127, in_size=(512, 512), c_in=64, c_out=64, bias=True), "fwd"),
    "smallgroup": (shape_kw(n=63, in_size=(512, 512), c_in=128, c_out=128, groups=32), "fwd"),
    "pointwise": (shape_kw(n=127, in_size=(512, 512), c_in=64, c_out=64, k=(1, 1), pad=(0, 0)), "fwd"),
    "dgrad": (shape_kw(n=127, in_size=(512, 512), c_in=64, c_out=64, stride=(2, 2)), "dgrad"),
}


@pytest.mark.parametrize("family", list(CASES))
def test_largest_tensors_fwd_dgrad(gb, family):
    kw, op = CASES[family]
    d = lib_desc(gb, kw)
    assert gb.gbconv_select(d, 1 if op == "dgrad" else 0) == family
    c = oracle_conv(kw)
    xs, ws, ys = gb.desc_shapes(d)
    src_shape, dst_shape = (ys, xs) if op == "dgrad" else (xs, ys)
    assert max(int(np.prod(src_shape)), int(np.prod(dst_shape))) >= 2 ** 31 - 2 ** 25  # really near the limit
    src = _tiled_ints(31 + len(family), src_shape, -3, 3)
    w = synth.integers(41 + len(family), ws, -2, 2).astype(np.float32)
    b = synth.integers(51, (kw["c_out"],), -4, 4).astype(np.float32) if kw["bias"] else None
    src_d, w_d = _bf16_dev(src), _bf16_dev(w)
    out = torch.empty(dst_shape, dtype=torch.bfloat16, device="cuda")
    if op == "dgrad":
        gb.conv_bwd_data(d, src_d, w_d, dx=out)
    else:
        gb.conv_fwd(d, src_d, w_d, None if b is None else torch.from_numpy(b).cuda(), y=out)
    gb.device_status()
    del src_d
    n_, h_, w_, ch = dst_shape
    idx = _samples((n_, ch, h_, w_), 61 + len(family))
    got = _gather_nhwc(out, idx)
    if op == "dgrad":
        ref = oracle.conv_dgrad_points(c, src, w, idx)
    else:
        ref = oracle.conv_fwd_points(c, src, w, b, idx)
    np.testing.assert_array_equal(got, bf16_round(ref))
    del out
    torch.cuda.empty_cache()


SPARSE = (0, 146, 292)


def test_largest_tensors_wgrad(gb):
    # weight gradient over 293 images of 1016 x 112 x 64: x and dy at 2.13e9 elements each (the tensor-core
    # weight gradient keeps an image row in one box: at most about 112 columns)
    kw = shape_kw(n=293, in_size=(1016, 112), c_in=64, c_out=64)
    d = lib_desc(gb, kw)
    assert gb.gbconv_select(d, 2) == "wgrad"
    c = oracle_conv(kw)
    xs, ws, ys = gb.desc_shapes(d)
    # x in [-1, 1] and dy in [-1, 1]: |dW| <= 293 * 1016 * 112 = 3.3e7 would pass 2^24, so dy is zero
    # outside three images (the first, a middle one, the last: sums of at most 3.4e5 exact products)
    x = _tiled_ints(71, xs, -1, 1)
    g = np.zeros(ys, dtype=np.float32)
    for i, nn in enumerate(SPARSE):
        g[nn] = _tiled_ints(72 + i, (1,) + ys[1:], -1, 1)[0]
    x_d, g_d = _bf16_dev(x), _bf16_dev(g)
    dw, db = gb.conv_bwd_filter(d, x_d, g_d, want_db=True)
    gb.device_status()
    got = dw.float().cpu().numpy().astype(np.float64)
    # every weight element is a sum over the three images: the oracle on those images alone
    sub = oracle.Conv(**{**c.__dict__, "n": len(SPARSE)})
    ref = oracle.conv_wgrad(sub, x[list(SPARSE)], g[list(SPARSE)])
    np.testing.assert_array_equal(got, bf16_round(ref))
    np.testing.assert_array_equal(db.cpu().numpy().astype(np.float64), oracle.conv_bgrad(sub, g[list(SPARSE)]))
