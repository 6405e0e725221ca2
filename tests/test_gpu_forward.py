"""Forward convolution on the GPU (conv_bwd_data_run_forward, the operator whose
adjoint the library's backward-data path computes) against the oracle's
forward correlation, element by element, and the adjoint identity checked on
the GPU's own outputs:
    <conv(x, w), dy> = <x, dgrad(dy, w)>   with dy = conv(x, w) as the GPU wrote it,
so that the left side is a sum of squares (a signal far above the rounding
bound) and a wrong tap, flip or index on either GPU path shows up as an O(1)
mismatch.  Tolerance of the forward parity (ref = oracle, S = sum of |x*w|
over the window): |err| <= 2^-8 |ref| + 1e-4 S, as for dgrad."""
import zlib

import numpy as np
import pytest
import torch

import oracle
from conv2d_backward_implicit_bwd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conv2d_backward_implicit_bwd_gb300 import build as cbuild
    cbuild.build()
    from conv2d_backward_implicit_bwd_gb300 import binding
    return binding


def _mk(name, **kw):
    base = dict(dtype=wl.BF16, layout=wl.NHWC, dist="normal", sigma=0.5, seed=zlib.crc32(name.encode()) % 100000)
    base.update(kw)
    return wl.Case(name=name, **base)


FWD_CASES = [
    _mk("fwd_3x3s1", N=2, C=64, K=64, Hi=9, Wi=9, Y=3, X=3, pad=(1, 1)),
    _mk("fwd_3x3s2_ragged_k", N=3, C=128, K=136, Hi=13, Wi=11, Y=3, X=3, pad=(1, 1), stride=(2, 2)),
    _mk("fwd_dil2", N=2, C=64, K=128, Hi=12, Wi=12, Y=3, X=3, pad=(2, 2), dil=(2, 2)),
    _mk("fwd_groups2", N=2, C=128, K=64, Hi=10, Wi=9, Y=3, X=3, pad=(1, 1), stride=(2, 2), groups=2),
    _mk("fwd_1x2_s1x2_small", N=2, C=256, K=256, Hi=1, Wi=64, Y=1, X=2, stride=(1, 2)),
    _mk("fwd_c_tail", N=2, C=72, K=40, Hi=7, Wi=9, Y=2, X=3, pad=(0, 1), stride=(2, 1)),
    _mk("fwd_5x5s3", N=2, C=64, K=64, Hi=19, Wi=17, Y=5, X=5, pad=(2, 2), stride=(3, 3)),
    _mk("fwd_many_tiles", N=4, C=64, K=256, Hi=20, Wi=20, Y=3, X=3, pad=(1, 1)),
    _mk("fwd_deep_c", N=1, C=512, K=64, Hi=6, Wi=7, Y=2, X=2, pad=(1, 0), stride=(1, 2)),
]


def _geom(c):
    return oracle.geom(c.N, c.C, c.K, c.Hi, c.Wi, c.Y, c.X, c.pad, c.stride, c.dil, c.groups)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _inputs(c, g):
    dy_s, w_s, dx_s = oracle.shapes(g, oracle.LAYOUT_NHWC)
    x, w = wl.draw(c, dx_s, w_s)
    return x, w, dy_s


@pytest.mark.parametrize("c", FWD_CASES, ids=lambda c: c.name)
def test_forward_matches_oracle(B, c):
    g = _geom(c)
    x, w, dy_s = _inputs(c, g)
    plan = B.Plan.from_case(c)
    y = torch.full(dy_s, float("nan"), dtype=torch.bfloat16, device="cuda")
    plan.run_forward(_dev(x), _dev(w), y)
    st, det = plan.status()
    assert st == B.OK, (B.status_string(st), hex(det))
    got = _f64(y)
    assert np.all(np.isfinite(got)), "unwritten (NaN) outputs"
    ref = oracle.conv_fwd(g, oracle.LAYOUT_NHWC, x, w)
    ab = oracle.conv_fwd(g, oracle.LAYOUT_NHWC, np.abs(oracle.widen(x)), np.abs(oracle.widen(w)))
    bound = oracle.tolerance(ref, ab, wl.BF16)
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"max excess {float(np.max(err - bound)):.3e}"


@pytest.mark.parametrize("c", FWD_CASES, ids=lambda c: c.name)
def test_adjoint_identity_on_gpu(B, c):
    g = _geom(c)
    x, w, dy_s = _inputs(c, g)
    plan = B.Plan.from_case(c)
    xd, wd = _dev(x), _dev(w)
    y = torch.empty(dy_s, dtype=torch.bfloat16, device="cuda")
    plan.run_forward(xd, wd, y)
    dx = torch.empty(x.shape, dtype=torch.bfloat16, device="cuda")
    plan.run(y, wd, dx)  # dy := the forward output
    st, det = plan.status()
    assert st == B.OK, (B.status_string(st), hex(det))
    yv, dxv, xv = _f64(y), _f64(dx), oracle.widen(x)
    lhs = float(np.sum(yv * yv))
    rhs = float(np.sum(xv * dxv))
    scale = float(np.sum(np.abs(xv) * np.abs(dxv)))
    assert lhs > 0.0
    assert abs(lhs - rhs) <= 2.0 ** -6 * scale, (lhs, rhs, scale)


def test_forward_unsupported_and_argument_errors(B):
    f32 = B.Plan(1, 64, 64, 8, 8, 3, 3, (1, 1), dtype="f32")
    assert f32.run_forward_ptr(4096, 8192, 1 << 20) == B.ERR_UNSUPPORTED
    narrow = B.Plan(1, 64, 64, 8, 8, 3, 3, (1, 1), groups=2, layout="nhwc", dtype="bf16")  # C/G = 32
    assert narrow.run_forward_ptr(4096, 8192, 1 << 20) == B.ERR_UNSUPPORTED
    big_stride = B.Plan(1, 64, 64, 40, 40, 3, 3, (1, 1), stride=(9, 9), layout="nhwc", dtype="bf16")
    assert big_stride.run_forward_ptr(4096, 8192, 1 << 20) == B.ERR_UNSUPPORTED
    ok = B.Plan(1, 64, 64, 8, 8, 3, 3, (1, 1), layout="nhwc", dtype="bf16")
    assert ok.run_forward_ptr(0, 8192, 1 << 20) == B.ERR_INVALID_ARG
    x = torch.zeros(1 * 8 * 8 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(64 * 9 * 64, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(1 * 8 * 8 * 64, dtype=torch.bfloat16, device="cuda")
    assert ok.run_forward_ptr(x.data_ptr() + 2, w.data_ptr(), y.data_ptr()) == B.ERR_MISALIGNED
    assert ok.run_forward_ptr(x.data_ptr(), w.data_ptr(), x.data_ptr() + 16) == B.ERR_INVALID_ARG  # y overlaps x
