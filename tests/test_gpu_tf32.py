"""GPU parity of the fp32 tensor-core path (tcgen05 kind::tf32, each operand
split as hi + lo, three products per k step) against the fp64 oracle, with the
fp32 tolerance |err| <= 1e-5 * sum |dy*w| per element -- the bound plain TF32
(10-bit operands) would miss by two orders of magnitude, so these cases also
show that the split carries the low bits.

Small cases force the path (CONVBWD_DEBUG_PATH=tf32) and cover several m and
n tiles with ragged tails, K/G not a multiple of the 32-channel k step, groups,
uncovered pixels (the kernel's own fill), an empty-class 1x1 stride-2 problem
and NCHW/GKCYX problems (dy and dx transposed around the NHWC kernel, the
filter split reading GKCYX directly).  The fp32 workloads above the size
threshold take the path by themselves and are checked element by element,
also through the pipelined host entry point."""
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
    base = dict(dtype=wl.F32, layout=wl.NHWC, dist="uniform", seed=zlib.crc32(name.encode()) % 100000)
    base.update(kw)
    return wl.Case(name=name, **base)


def _geom(c):
    return oracle.geom(c.N, c.C, c.K, c.Hi, c.Wi, c.Y, c.X, c.pad, c.stride, c.dil, c.groups)


def _lay(c):
    return oracle.LAYOUT_NCHW if c.layout == wl.NCHW else oracle.LAYOUT_NHWC


def inputs(c):
    g = _geom(c)
    dy_s, w_s, _ = oracle.shapes(g, _lay(c))
    dy, w = wl.draw(c, dy_s, w_s)
    return g, dy, w


def run_gpu(B, c, dy, w):
    plan = B.Plan.from_case(c)
    _, _, dx_s = plan.shapes()
    dx = torch.full(dx_s, float("nan"), dtype=torch.float32, device="cuda")
    plan.run(torch.from_numpy(dy).cuda(), torch.from_numpy(w).cuda(), dx)
    st, det = plan.status()
    assert st == B.OK, (B.status_string(st), hex(det))
    return dx.cpu().numpy().astype(np.float64), plan


def check_full(c, got, g, dy, w, n_range=None):
    ref, ab = oracle.dgrad(g, _lay(c), dy, w, n_range=n_range)
    if n_range is not None:
        sl = slice(*n_range)
        got, ref, ab = got[sl], ref[sl], ab[sl]
    assert np.all(np.isfinite(got)), "unwritten (NaN) outputs"
    bound = oracle.tolerance(ref, ab, c.dtype)
    err = np.abs(got - ref)
    worst = float(np.max(err - bound))
    assert worst <= 0.0, f"max excess {worst:.3e}; max err {err.max():.3e}"
    # the three-term split keeps the error far inside the fp32 bound (plain
    # TF32 operands would sit near 1e-3 * sum |dy*w|)
    rel = float(np.max(err / np.maximum(ab, 1e-300)))
    assert rel < 4e-6, rel
    return rel


FORCED = [
    _mk("tf32_3x3s2_two_n_tiles", N=2, C=256, K=256, Hi=17, Wi=15, Y=3, X=3, pad=(1, 1), stride=(2, 2)),
    _mk("tf32_ragged_k_tail", N=3, C=72, K=44, Hi=11, Wi=13, Y=5, X=3, pad=(2, 1), stride=(2, 3), dil=(1, 2)),
    _mk("tf32_groups2", N=2, C=192, K=128, Hi=10, Wi=10, Y=3, X=3, pad=(1, 1), groups=2),
    _mk("tf32_fill_d2", N=2, C=128, K=64, Hi=12, Wi=12, Y=3, X=3, pad=(1, 1), stride=(2, 2), dil=(2, 2)),
    _mk("tf32_1x1_s2", N=4, C=64, K=128, Hi=14, Wi=14, Y=1, X=1, stride=(2, 2)),
    _mk("tf32_many_m_tiles", N=4, C=32, K=96, Hi=33, Wi=31, Y=3, X=3, pad=(1, 1)),
    _mk("tf32_nchw", N=2, C=64, K=96, Hi=9, Wi=11, Y=3, X=3, pad=(1, 1), stride=(2, 2), layout=wl.NCHW),
    _mk("tf32_nchw_groups4", N=2, C=128, K=128, Hi=7, Wi=7, Y=3, X=3, pad=(1, 1), groups=4, layout=wl.NCHW),
    # 5x5 filter, stride 5: 25 residue classes, so two launches of at most 16 classes each
    _mk("tf32_25_classes", N=2, C=64, K=36, Hi=23, Wi=21, Y=5, X=5, pad=(2, 2), stride=(5, 5)),
    # 4 channels per group: one 128-wide n-tile with 124 zero columns
    _mk("tf32_narrow_cg4", N=2, C=4, K=64, Hi=13, Wi=12, Y=3, X=3, pad=(1, 1), stride=(2, 2)),
]


@pytest.mark.parametrize("c", FORCED, ids=lambda c: c.name)
def test_forced_tf32_matches_oracle(B, monkeypatch, c):
    monkeypatch.setenv("CONVBWD_DEBUG_PATH", "tf32")
    g, dy, w = inputs(c)
    got, plan = run_gpu(B, c, dy, w)
    path, launches = plan.path()
    assert path == "tf32", plan.path()
    # filter split + one kernel per 16 classes (+ the tile zeroing of each launch
    # whose last round is cut into k-block ranges), and two transposes around
    # them for NCHW
    kernels = (plan.num_subgemms() + 15) // 16
    assert launches - (2 if c.layout == wl.NCHW else 0) in range(1 + kernels, 2 + 2 * kernels), plan.path()
    check_full(c, got, g, dy, w)


@pytest.mark.parametrize("split", ["1", "0"])
@pytest.mark.parametrize("idx", [0, 1, 3, 5])
def test_tail_split_schedule(B, monkeypatch, idx, split):
    """Tiles of the last round cut into k-block ranges over every SM (fp32
    atomic adds into a zeroed dx region) against whole tiles only."""
    c = FORCED[idx]
    monkeypatch.setenv("CONVBWD_DEBUG_PATH", "tf32")
    monkeypatch.setenv("CONVBWD_DEBUG_STREAMK", split)
    g, dy, w = inputs(c)
    got, plan = run_gpu(B, c, dy, w)
    # these problems hold fewer tiles than SMs: every tile is in the last round,
    # so the split adds the zeroing launch to the filter split and the kernel
    assert plan.path() == ("tf32", 3 if split == "1" else 2), plan.path()
    check_full(c, got, g, dy, w)


def test_tf32_matches_cuda_core_path(B, monkeypatch):
    """The same problem on the tensor cores and on the CUDA cores: both within
    the fp32 bound of the oracle and within twice that bound of each other."""
    c = FORCED[0]
    g, dy, w = inputs(c)
    monkeypatch.setenv("CONVBWD_DEBUG_PATH", "tf32")
    tc, _ = run_gpu(B, c, dy, w)
    monkeypatch.setenv("CONVBWD_DEBUG_PATH", "simt")
    simt, plan = run_gpu(B, c, dy, w)
    assert plan.path()[0] == "simt"
    ref, ab = oracle.dgrad(g, _lay(c), dy, w)
    assert np.all(np.abs(tc - simt) <= 2 * oracle.tolerance(ref, ab, c.dtype))


LARGE = [c for c in wl.CASES if c.tags[0] == "fp32_large"]


@pytest.mark.parametrize("c", LARGE, ids=lambda c: c.name)
def test_large_fp32_workloads(B, c):
    g, dy, w = inputs(c)
    got, plan = run_gpu(B, c, dy, w)
    assert plan.path()[0] == "tf32", plan.path()
    check_full(c, got, g, dy, w)  # every element


def test_run_host_pipelined_tf32(B):
    """run_host over batch chunks: each chunk plan splits the filter into the
    parent's buffers (same stream, in turn) before its kernel."""
    c = wl.case("fp32_nhwc_32x28x28x512")
    g, dy, w = inputs(c)
    plan = B.Plan.from_case(c)
    assert plan.path()[0] == "tf32"
    dy_s, w_s, dx_s = plan.shapes()
    dy_h = torch.from_numpy(dy).reshape(dy_s).pin_memory()
    w_h = torch.from_numpy(w).reshape(w_s).pin_memory()
    dx_h = torch.full(dx_s, float("nan"), dtype=torch.float32).pin_memory()
    dy_d = torch.empty(dy_s, dtype=torch.float32, device="cuda")
    w_d = torch.empty(w_s, dtype=torch.float32, device="cuda")
    dx_d = torch.full(dx_s, float("nan"), dtype=torch.float32, device="cuda")
    plan.run_host(dy_h, w_h, dx_h, dy_d, w_d, dx_d)
    st, det = plan.status()
    assert st == B.OK, (B.status_string(st), hex(det))
    got = dx_h.numpy().astype(np.float64)
    assert np.all(np.isfinite(got)), "unwritten (NaN) outputs"
    check_full(c, got, g, dy, w)


def test_tf32_alignment_rule(B, monkeypatch):
    monkeypatch.setenv("CONVBWD_DEBUG_PATH", "tf32")
    c = FORCED[4]
    plan = B.Plan.from_case(c)
    assert plan.path()[0] == "tf32"
    dy_s, w_s, dx_s = plan.shapes()
    dy = torch.zeros(dy_s, dtype=torch.float32, device="cuda")
    w = torch.zeros(w_s, dtype=torch.float32, device="cuda")
    dx = torch.zeros(int(np.prod(dx_s)) + 4, dtype=torch.float32, device="cuda")
    assert plan.run_ptr(dy.data_ptr(), w.data_ptr(), dx.data_ptr() + 4) == B.ERR_MISALIGNED
    torch.cuda.synchronize()


def test_split_filter_unavailable_falls_back_to_cuda_cores(B, monkeypatch):
    """When the plan cannot hold the split filter it runs on the CUDA cores,
    rescheduled for that kernel's 64-row tiles (several per class here, so a
    tile count left at the tensor-core kernel's 128 rows would leave rows of
    dx unwritten)."""
    monkeypatch.setenv("CONVBWD_DEBUG_PATH", "tf32")
    monkeypatch.setenv("CONVBWD_DEBUG_NO_WSPLIT", "1")
    c = _mk("tf32_no_split_filter", N=4, C=96, K=80, Hi=17, Wi=19, Y=3, X=3, pad=(1, 1), stride=(2, 2))
    g, dy, w = inputs(c)
    got, plan = run_gpu(B, c, dy, w)
    assert plan.path()[0] == "simt", plan.path()
    assert plan.tile()[:2] == (64, 64), plan.tile()
    check_full(c, got, g, dy, w)
