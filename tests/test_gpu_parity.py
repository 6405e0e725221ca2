"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Tolerances per element (ref = oracle value, S = sum over taps of |dy*w|):
  fp32 output: |err| <= 1e-5 * S
  bf16 output: |err| <= 2^-8 * |ref| + 1e-4 * S
Inputs come from the seeded generators shared with the oracle (byte-identical
bf16/fp32 values).  dx is pre-filled with NaN so that a pixel the library
forgets to write shows up as a failure.  Every output element is compared with
the oracle, the five benchmark workloads included (at the plan and launch
configuration the benchmark times).
"""
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


def _geom(c):
    return oracle.geom(c.N, c.C, c.K, c.Hi, c.Wi, c.Y, c.X, c.pad, c.stride, c.dil, c.groups)


def _lay(c):
    return oracle.LAYOUT_NCHW if c.layout == wl.NCHW else oracle.LAYOUT_NHWC


def to_dev(a, dtype):
    if dtype == wl.BF16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_dgrad(B, c, dy, w, stream=None, prefill=float("nan")):
    plan = B.Plan.from_case(c)
    _, _, dx_s = plan.shapes()
    tdt = torch.bfloat16 if c.dtype == wl.BF16 else torch.float32
    dyd, wd = to_dev(dy, c.dtype), to_dev(w, c.dtype)
    dx = torch.full(dx_s, prefill, dtype=tdt, device="cuda")
    plan.run(dyd, wd, dx, stream)
    st, det = plan.status(stream)
    assert st == B.OK, (B.status_string(st), hex(det))
    return dx.float().cpu().numpy().astype(np.float64), plan


def inputs(c):
    g = _geom(c)
    dy_s, w_s, _ = oracle.shapes(g, _lay(c))
    dy, w = wl.draw(c, dy_s, w_s)
    return g, dy, w


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
    return float(np.max(err / np.maximum(bound, 1e-300)))


SMALL = [c for c in wl.CASES if c.tags[0] == "fp32_small"]


@pytest.mark.parametrize("c", SMALL, ids=lambda c: c.name)
def test_small_configs_full(B, c):
    g, dy, w = inputs(c)
    got, plan = gpu_dgrad(B, c, dy, w)
    assert plan.path()[0] == "simt"
    check_full(c, got, g, dy, w)


LARGE = ["bf16_16x1x512x2048", "bf16_resnext_64x56x56x256", "bf16_32x28x28x512", "bf16_32x14x14_1024",
         "bf16_32x57x57x128"]


@pytest.mark.parametrize("name", LARGE)
def test_large_configs(B, name):
    """The whole dx of each bf16 benchmark workload against the oracle's."""
    c = wl.case(name)
    g, dy, w = inputs(c)
    got, plan = gpu_dgrad(B, c, dy, w)
    assert plan.path()[0] == ("grouped" if name == "bf16_resnext_64x56x56x256" else "tcgen05")
    check_full(c, got, g, dy, w)


def _mk(name, **kw):
    base = dict(dtype=wl.BF16, layout=wl.NHWC, dist="normal", sigma=0.5, seed=zlib.crc32(name.encode()) % 100000)
    base.update(kw)
    return wl.Case(name=name, **base)


# Tensor-core path: several tiles, ragged M / N / K tails, groups, classes whose
# taps all fall outside dy, uncovered rows/columns, asymmetric geometry.
TC_CASES = [
    _mk("tc_ragged_3x3s2", N=3, C=192, K=136, Hi=13, Wi=11, Y=3, X=3, pad=(1, 1), stride=(2, 2)),
    _mk("tc_1x1s2", N=2, C=256, K=64, Hi=9, Wi=17, Y=1, X=1, stride=(2, 2)),
    _mk("tc_groups2", N=2, C=128, K=128, Hi=10, Wi=10, Y=3, X=3, pad=(1, 1), groups=2),
    _mk("tc_groups4_kg72", N=2, C=256, K=288, Hi=7, Wi=8, Y=3, X=2, pad=(1, 0), stride=(2, 1), groups=4),
    _mk("tc_asym", N=4, C=320, K=96, Hi=7, Wi=9, Y=5, X=3, pad=(2, 1), stride=(3, 2), dil=(1, 2)),
    _mk("tc_filter_gt_input", N=2, C=64, K=64, Hi=3, Wi=3, Y=5, X=5, pad=(2, 2)),
    _mk("tc_stride4_uncovered", N=2, C=128, K=64, Hi=15, Wi=14, Y=3, X=3, pad=(1, 1), stride=(4, 4)),
    _mk("tc_m1", N=1, C=512, K=512, Hi=1, Wi=1, Y=1, X=1),
    _mk("tc_1x2_s1x2_small", N=2, C=256, K=256, Hi=1, Wi=64, Y=1, X=2, stride=(1, 2)),
    _mk("tc_dil2_s2", N=2, C=128, K=128, Hi=12, Wi=12, Y=3, X=3, pad=(1, 1), stride=(2, 2), dil=(2, 2)),
    _mk("tc_mixed", N=2, C=200, K=40, Hi=11, Wi=6, Y=2, X=4, pad=(0, 3), stride=(3, 1), dil=(2, 3)),
    _mk("tc_bn256_ragged", N=3, C=264, K=64, Hi=6, Wi=7, Y=3, X=3, pad=(1, 1), stride=(1, 1)),
    _mk("tc_deep_k", N=1, C=64, K=1024, Hi=5, Wi=6, Y=2, X=2, pad=(1, 1), stride=(2, 2)),
    _mk("tc_25_classes", N=1, C=64, K=64, Hi=20, Wi=20, Y=5, X=5, pad=(2, 2), stride=(5, 5)),
    _mk("tc_groups2_kg96", N=2, C=128, K=192, Hi=9, Wi=9, Y=3, X=3, pad=(1, 1), stride=(2, 2), groups=2),
]


@pytest.mark.parametrize("c", TC_CASES, ids=lambda c: c.name)
def test_tensor_core_path_full(B, c):
    g, dy, w = inputs(c)
    got, plan = gpu_dgrad(B, c, dy, w)
    assert plan.path()[0] == "tcgen05", plan.path()
    check_full(c, got, g, dy, w)


# Class pairs on the 1-SM kernel (C/G <= 128): two classes with the same rows
# and tap counts share a 128 x 256 tile (one A load, N = 256 MMAs, the upper
# 128 columns being the second class's channels and dx pixels): the 5x5
# stride-3 geometry (two pairs of 4-tap classes, two of 2-tap classes, one
# class alone), a 2x2 stride-2 filter with ragged C and K (columns past C/G and
# k past K zero), groups, and a pair mixed with unpaired classes in one launch;
# each also with pairing off (CONVBWD_DEBUG_FUSE=0, 128-wide tiles).
FUSE_CASES = [
    _mk("pair_tiles_5x5_s3", N=2, C=128, K=128, Hi=20, Wi=19, Y=5, X=5, pad=(2, 2), stride=(3, 3)),
    _mk("pair_tiles_2x2_s2_c96_k72", N=3, C=96, K=72, Hi=14, Wi=12, Y=2, X=2, stride=(2, 2)),
    _mk("pair_tiles_groups2", N=2, C=256, K=256, Hi=10, Wi=12, Y=2, X=2, stride=(2, 2), groups=2),
    _mk("pair_tiles_3x3_s3_uneven", N=2, C=64, K=136, Hi=13, Wi=11, Y=3, X=3, pad=(1, 1), stride=(3, 3)),
]


@pytest.mark.parametrize("paired", [True, False])
@pytest.mark.parametrize("c", FUSE_CASES + [wl.case("bf16_32x57x57x128")], ids=lambda c: c.name)
def test_class_pair_tiles(B, monkeypatch, c, paired):
    if not paired:
        monkeypatch.setenv("CONVBWD_DEBUG_FUSE", "0")
    g, dy, w = inputs(c)
    got, plan = gpu_dgrad(B, c, dy, w)
    assert plan.path()[0] == "tcgen05"
    assert plan.tile() == ((128, 256, 1) if paired else (128, 128, 1)), plan.tile()
    check_full(c, got, g, dy, w)


# Narrow-group path (C/G = K/G in {8, 16, 32}): every pixel written by the
# kernel itself, including ones no tap reaches.  Three kernels:
#   band  tcgen05, each band of dy staged once and read by every tap (C % 64 == 0,
#         strides <= 2, <= 32 taps): the default where it applies;
#   mma   warp-level MMA (C/G in {8, 16}, G % 8 == 0);
#   tc    tcgen05 with one im2col load of dy per tap (C % 64 == 0, <= 12 taps).
# CONVBWD_DEBUG_GROUPED selects one where it applies.
GROUPED_CASES = [
    _mk("grp_g32_cg8_3x3s2", N=2, C=256, K=256, Hi=13, Wi=11, Y=3, X=3, pad=(1, 1), stride=(2, 2), groups=32),
    _mk("grp_g32_cg8_s3_uncov", N=1, C=256, K=256, Hi=10, Wi=9, Y=2, X=2, pad=(0, 1), stride=(3, 3), groups=32),
    _mk("grp_g32_cg8_dil2", N=2, C=256, K=256, Hi=9, Wi=12, Y=3, X=3, pad=(2, 2), stride=(2, 2), dil=(2, 2), groups=32),
    _mk("grp_g64_cg8_1x1", N=3, C=512, K=512, Hi=7, Wi=5, Y=1, X=1, stride=(1, 1), groups=64),
    _mk("grp_g32_cg16_2x2s2", N=2, C=512, K=512, Hi=6, Wi=7, Y=2, X=2, pad=(1, 1), stride=(2, 2), groups=32),
    _mk("grp_g32_cg8_wide_row", N=1, C=256, K=256, Hi=3, Wi=37, Y=3, X=3, pad=(1, 1), stride=(2, 2), groups=32),
    _mk("grp_g8_cg8", N=2, C=64, K=64, Hi=9, Wi=10, Y=3, X=3, pad=(1, 1), stride=(2, 2), groups=8),
    _mk("grp_g16_cg16_s4", N=2, C=256, K=256, Hi=11, Wi=9, Y=3, X=3, pad=(1, 1), stride=(4, 4), groups=16),
    _mk("grp_g32_cg8_5x3_s1x2", N=1, C=256, K=256, Hi=8, Wi=13, Y=5, X=3, pad=(2, 1), stride=(1, 2), groups=32),
    _mk("grp_g8_cg8_3x3s2_many_tiles", N=4, C=64, K=64, Hi=30, Wi=29, Y=3, X=3, pad=(1, 1), stride=(2, 2), groups=8),
]
GROUPED_TC_ONLY = [
    # 32 channels per group: the tcgen05 kernels cover it
    _mk("grp_g8_cg32_3x3s2", N=2, C=256, K=256, Hi=11, Wi=12, Y=3, X=3, pad=(1, 1), stride=(2, 2), groups=8),
    # rows of one parity uncovered (stride 2, dilation 2, pad 2): written as zero by the kernel itself
    _mk("grp_g16_cg16_dil2_fill", N=2, C=256, K=256, Hi=13, Wi=10, Y=3, X=3, pad=(2, 2), stride=(2, 2), dil=(2, 2),
        groups=16),
    _mk("grp_g64_cg8_2x2_s2", N=3, C=512, K=512, Hi=9, Wi=8, Y=2, X=2, stride=(2, 2), groups=64),
]
# Banded kernel: several column segments, stride 1 (windows shifted by -1, 0
# and +1 pixel), mixed strides, 32-channel groups at stride 1, a 1x1 stride-2
# filter (classes without taps), a 4x4 and a 5x5 filter (16 and 25 windows,
# 28-column segments), output rows not a multiple of the band, more 64-channel
# blocks than SMs (a second wave of CTAs), and a full-size stride-1 ResNeXt
# layer (many units per CTA: every stage and accumulator buffer reused).
BAND_CASES = [
    _mk("band_cg8_s2_segs", N=2, C=128, K=128, Hi=9, Wi=130, Y=3, X=3, pad=(1, 1), stride=(2, 2), groups=16),
    _mk("band_cg8_s1_segs", N=2, C=64, K=64, Hi=7, Wi=70, Y=3, X=3, pad=(1, 1), stride=(1, 1), groups=8),
    _mk("band_cg16_s2x1", N=3, C=128, K=128, Hi=10, Wi=21, Y=3, X=3, pad=(1, 1), stride=(2, 1), groups=8),
    _mk("band_cg32_s1", N=2, C=256, K=256, Hi=14, Wi=15, Y=3, X=3, pad=(1, 1), stride=(1, 1), groups=8),
    _mk("band_cg8_1x1_s2", N=2, C=256, K=256, Hi=11, Wi=9, Y=1, X=1, stride=(2, 2), groups=32),
    _mk("band_cg8_4x4_s2_p1x2", N=1, C=128, K=128, Hi=9, Wi=11, Y=4, X=4, pad=(1, 2), stride=(2, 2), groups=16),
    _mk("band_cg8_5x5_s1_p2", N=2, C=128, K=128, Hi=9, Wi=40, Y=5, X=5, pad=(2, 2), stride=(1, 1), groups=16),
    _mk("band_cg8_2x3_s2_p0", N=2, C=64, K=64, Hi=13, Wi=17, Y=2, X=3, pad=(0, 0), stride=(2, 2), groups=8),
    _mk("band_cg8_160_blocks", N=1, C=10240, K=10240, Hi=5, Wi=5, Y=3, X=3, pad=(1, 1), stride=(2, 2), groups=1280),
    _mk("band_resnext_s1_32x56x56x256", N=32, C=256, K=256, Hi=56, Wi=56, Y=3, X=3, pad=(1, 1), stride=(1, 1),
        groups=32, sigma=0.05),
    # classes without pixels (one dx row / column: its odd residue is empty, so
    # the class has no store map) and odd sizes (the odd residue has one row /
    # column fewer, clipped by its map; segments starting past its last column)
    _mk("band_cg8_hi1_s2", N=3, C=64, K=64, Hi=1, Wi=20, Y=3, X=3, pad=(1, 1), stride=(2, 2), groups=8),
    _mk("band_cg8_wi1_s2", N=2, C=128, K=128, Hi=9, Wi=1, Y=3, X=3, pad=(1, 1), stride=(2, 2), groups=16),
    _mk("band_cg16_odd_s2", N=2, C=128, K=128, Hi=7, Wi=63, Y=3, X=3, pad=(1, 1), stride=(2, 2), groups=8),
]


def _band_fits(c):
    """The banded kernel's shared-memory and segment rules: two A stages of one
    staged band each (4 output rows plus the row offsets' span, 32 pixels x 128
    bytes per row), per window (distinct row and column offset pair) a B tile
    of classes x max(16, C/G) rows of 128 bytes, 32 KB epilogue staging,
    alignment and barriers within 227 KB; at least 16 output columns per
    32-pixel staged row."""
    def taps(s, p, d, F):
        return [(r, (r + p - f * d) // s) for r in range(s) for f in range(F) if (r + p - f * d) % s == 0]
    ty = taps(c.stride[0], c.pad[0], c.dil[0], c.Y)
    tx = taps(c.stride[1], c.pad[1], c.dil[1], c.X)
    oy, ox = [o for _, o in ty], [o for _, o in tx]
    windows = {(a[1], b[1]) for a in ty for b in tx}
    stage = (4 + max(oy) - min(oy)) * 32 * 128
    btile = c.stride[0] * c.stride[1] * max(16, c.C // c.groups) * 128
    smem = 1024 + 2 * stage + len(windows) * btile + 32768 + 256
    return smem <= 227 * 1024 and 32 - (max(ox) - min(ox)) >= 16 and 4 + max(oy) - min(oy) <= 64


def _grouped_eligible(c, kernel):
    cg, taps = c.C // c.groups, c.Y * c.X
    if kernel == "band":
        return cg in (8, 16, 32) and c.C % 64 == 0 and max(c.stride) <= 2 and taps <= 32 and _band_fits(c)
    if kernel == "tc":
        return cg in (8, 16, 32) and c.C % 64 == 0 and taps <= 12
    return cg in (8, 16) and c.groups % 8 == 0


def _expected_kernel(c, kernel):
    if _grouped_eligible(c, kernel):
        return kernel
    for k in ("band", "mma", "tc"):
        if _grouped_eligible(c, k):
            return k
    raise AssertionError("no narrow-group kernel applies")


def _run_grouped(B, monkeypatch, c, kernel):
    monkeypatch.setenv("CONVBWD_DEBUG_GROUPED", kernel)
    g, dy, w = inputs(c)
    got, plan = gpu_dgrad(B, c, dy, w)
    assert plan.path() == ("grouped", 1)
    k = _expected_kernel(c, kernel)
    assert plan.grouped_kernel() == k, (plan.grouped_kernel(), k)
    assert plan.tile() == ((0, 0, 1) if k == "mma" else (128, 64, 1)), plan.tile()
    assert plan.a_operand() == {"band": "band", "tc": "im2col", "mma": "gather"}[k]
    check_full(c, got, g, dy, w)


@pytest.mark.parametrize("kernel", ["band", "tc", "mma"])
@pytest.mark.parametrize("c", GROUPED_CASES, ids=lambda c: c.name)
def test_grouped_path_full(B, monkeypatch, c, kernel):
    _run_grouped(B, monkeypatch, c, kernel)


@pytest.mark.parametrize("kernel", ["band", "tc"])
@pytest.mark.parametrize("c", GROUPED_TC_ONLY, ids=lambda c: c.name)
def test_grouped_tensor_core_shapes(B, monkeypatch, c, kernel):
    _run_grouped(B, monkeypatch, c, kernel)


@pytest.mark.parametrize("c", BAND_CASES, ids=lambda c: c.name)
def test_grouped_band_kernel(B, monkeypatch, c):
    _run_grouped(B, monkeypatch, c, "band")


@pytest.mark.parametrize("kernel", ["tc", "mma"])
def test_grouped_layer_on_other_kernels(B, monkeypatch, kernel):
    """The benchmark's grouped layer (whole dx) on the two non-default kernels."""
    _run_grouped(B, monkeypatch, wl.case("bf16_resnext"), kernel)


# CUDA-core path: fp32 in both layouts, bf16 fallbacks (small channel
# counts, NCHW bf16), and random tiny geometries.
def _ok(c):
    return (c.Hi + 2 * c.pad[0] - c.dil[0] * (c.Y - 1) - 1 >= 0 and
            c.Wi + 2 * c.pad[1] - c.dil[1] * (c.X - 1) - 1 >= 0)


SIMT_CASES = (wl.random_tiny_cases(40, seed=31, accept=_ok) +
              wl.random_tiny_cases(20, seed=32, layout=wl.NHWC, accept=_ok) +
              wl.random_tiny_cases(20, seed=33, dtype=wl.BF16, layout=wl.NHWC, accept=_ok) +
              wl.random_tiny_cases(10, seed=34, dtype=wl.BF16, layout=wl.NCHW, accept=_ok) + [
                  _mk("simt_bf16_cg24", N=2, C=48, K=32, Hi=9, Wi=9, Y=3, X=3, pad=(1, 1), stride=(2, 2), groups=2),
                  _mk("simt_f32_nhwc", N=2, C=96, K=80, Hi=8, Wi=7, Y=3, X=3, pad=(1, 1), stride=(2, 2),
                      dtype=wl.F32, dist="uniform"),
                  _mk("simt_f32_wide", N=1, C=130, K=70, Hi=6, Wi=5, Y=2, X=3, pad=(1, 1), stride=(1, 2),
                      dtype=wl.F32, layout=wl.NCHW, dist="uniform"),
                  # 3/4 of dx uncovered: the fill kernel writes 2.45 MB of zeros before the GEMM
                  _mk("simt_f32_fill_56", N=4, C=64, K=64, Hi=56, Wi=57, Y=3, X=3, pad=(1, 1), stride=(2, 2),
                      dil=(2, 2), dtype=wl.F32, layout=wl.NHWC, dist="uniform"),
              ])


@pytest.mark.parametrize("c", SIMT_CASES, ids=lambda c: c.name + "_" + c.dtype + "_" + c.layout)
def test_cuda_core_path_full(B, c):
    g, dy, w = inputs(c)
    got, plan = gpu_dgrad(B, c, dy, w)
    check_full(c, got, g, dy, w)


# bf16 NCHW/GKCYX problems whose NHWC/KYXC twin runs on a tensor-core path:
# dy and w are transposed into plan-owned scratch, dx transposed back.
NCHW_TC_CASES = [
    _mk("nchw_bf16_tc", N=2, C=256, K=128, Hi=9, Wi=11, Y=3, X=3, pad=(1, 1), stride=(2, 2), layout=wl.NCHW),
    _mk("nchw_bf16_pair", N=2, C=512, K=256, Hi=7, Wi=8, Y=3, X=3, pad=(1, 1), layout=wl.NCHW),
    _mk("nchw_bf16_grouped", N=2, C=256, K=256, Hi=9, Wi=10, Y=3, X=3, pad=(1, 1), stride=(2, 2), groups=32,
        layout=wl.NCHW),
    _mk("nchw_bf16_fill", N=2, C=128, K=128, Hi=12, Wi=12, Y=3, X=3, pad=(1, 1), stride=(2, 2), dil=(2, 2),
        layout=wl.NCHW),
    _mk("nchw_bf16_ragged", N=3, C=200, K=40, Hi=11, Wi=6, Y=2, X=4, pad=(0, 3), stride=(3, 1), dil=(2, 3),
        layout=wl.NCHW),
    _mk("nchw_bf16_odd_hw", N=1, C=64, K=72, Hi=13, Wi=67, Y=1, X=3, pad=(0, 1), stride=(1, 2), layout=wl.NCHW),
]


@pytest.mark.parametrize("c", NCHW_TC_CASES, ids=lambda c: c.name)
def test_nchw_bf16_through_transposes(B, c):
    g, dy, w = inputs(c)
    for _ in range(2):  # the second run reuses the scratch
        got, plan = gpu_dgrad(B, c, dy, w)
        name, launches = plan.path()
        assert name in ("tcgen05", "grouped"), plan.path()
        assert launches >= 4, plan.path()  # two transposes in, the kernels, one transpose out
        check_full(c, got, g, dy, w)


def test_forced_simt_matches_tensor_core_path(B, monkeypatch):
    """The tensor-core kernel and the CUDA-core kernel agree on a bf16 case
    (both compared with the oracle too)."""
    c = TC_CASES[0]
    g, dy, w = inputs(c)
    tc, _ = gpu_dgrad(B, c, dy, w)
    monkeypatch.setenv("CONVBWD_DEBUG_PATH", "simt")
    simt, plan = gpu_dgrad(B, c, dy, w)
    assert plan.path()[0] == "simt"
    check_full(c, simt, g, dy, w)
    check_full(c, tc, g, dy, w)


@pytest.mark.parametrize("idx", [0, 4, 8, 10])
def test_cp_async_producer_variant(B, monkeypatch, idx):
    """The cp.async A producer (used where a 64-channel block may cross a
    group boundary, or im2col corners fall outside their range) on shapes
    that normally take the TMA im2col producer."""
    c = TC_CASES[idx]
    g, dy, w = inputs(c)
    monkeypatch.setenv("CONVBWD_DEBUG_NOIM2COL", "1")
    got, plan = gpu_dgrad(B, c, dy, w)
    assert plan.path()[0] == "tcgen05"
    check_full(c, got, g, dy, w)


SK_CASES = [
    _mk("sk_1x2_s1x2_small", N=2, C=256, K=256, Hi=1, Wi=64, Y=1, X=2, stride=(1, 2)),
    _mk("sk_one_tile_deep_k", N=1, C=256, K=2048, Hi=16, Wi=16, Y=1, X=1),          # 32 units over many pairs
    _mk("sk_multiclass", N=2, C=512, K=192, Hi=13, Wi=11, Y=3, X=3, pad=(1, 1), stride=(2, 2)),
    _mk("sk_ragged_n", N=3, C=264, K=64, Hi=6, Wi=7, Y=3, X=3, pad=(1, 1)),
    _mk("sk_dil2_fill", N=4, C=256, K=256, Hi=12, Wi=12, Y=3, X=3, pad=(1, 1), stride=(2, 2), dil=(2, 2)),
]


@pytest.mark.parametrize("forced", ["1", "0"])
@pytest.mark.parametrize("c", SK_CASES, ids=lambda c: c.name)
def test_stream_k_and_whole_tiles(B, monkeypatch, c, forced):
    """The 2-SM kernel with stream-K (units split across SM pairs, partial
    tiles added by the owning pair) and with whole tiles; each run twice so
    the second launch's flags carry a new epoch."""
    g, dy, w = inputs(c)
    monkeypatch.setenv("CONVBWD_DEBUG_STREAMK", forced)
    plan = B.Plan.from_case(c)
    assert plan.path()[0] == "tcgen05"
    dy_s, w_s, dx_s = plan.shapes()
    dyd, wd = to_dev(dy, c.dtype), to_dev(w, c.dtype)
    for _ in range(2):
        dx = torch.full(dx_s, float("nan"), dtype=torch.bfloat16, device="cuda")
        plan.run(dyd, wd, dx)
        st, det = plan.status()
        assert st == B.OK, (B.status_string(st), hex(det))
        check_full(c, dx.float().cpu().numpy().astype(np.float64), g, dy, w)


# 2-SM kernel variants: 512-wide pair tiles (two N=256 MMAs per k slice, one
# accumulator buffer), 256-wide pair tiles, pair tiles for C/G = 128..255, and
# pair tiles whose last 256-row block holds fewer than 129 rows (the second
# CTA of the pair then has no valid rows).
W512 = {"CONVBWD_DEBUG_BN": "512"}
W256 = {"CONVBWD_DEBUG_BN": "256"}
PAIR = {"CONVBWD_DEBUG_2SM": "1"}
PAIR_CASES = [
    (_mk("w512_ragged_n", N=3, C=768, K=192, Hi=9, Wi=7, Y=3, X=3, pad=(1, 1), stride=(2, 2)), W512),
    (_mk("w512_1x2_s1x2", N=2, C=1024, K=512, Hi=1, Wi=64, Y=1, X=2, stride=(1, 2)), W512),
    (_mk("w512_ragged_m", N=4, C=512, K=128, Hi=17, Wi=15, Y=3, X=3, pad=(1, 1)), W512),
    (_mk("w512_groups2", N=2, C=1024, K=256, Hi=8, Wi=9, Y=3, X=3, pad=(1, 1), groups=2), W512),
    (_mk("w512_tail8", N=2, C=520, K=64, Hi=7, Wi=7, Y=3, X=3, pad=(1, 1), stride=(2, 2), dil=(2, 2)), W512),
    (_mk("pair_cg128", N=2, C=128, K=128, Hi=12, Wi=12, Y=3, X=3, pad=(1, 1), stride=(2, 2), dil=(2, 2)), PAIR),
    (_mk("pair_cg200", N=2, C=200, K=40, Hi=11, Wi=6, Y=2, X=4, pad=(0, 3), stride=(3, 1), dil=(2, 3)), PAIR),
    (_mk("pair_5x5s3", N=2, C=128, K=128, Hi=19, Wi=17, Y=5, X=5, pad=(2, 2), stride=(3, 3)), PAIR),
    (_mk("pair_1x2_s1x2", N=4, C=512, K=256, Hi=1, Wi=128, Y=1, X=2, stride=(1, 2)), W256),
    (_mk("pair_odd_blocks", N=3, C=256, K=96, Hi=13, Wi=11, Y=3, X=3, pad=(1, 1), stride=(2, 2)), W256),
    (_mk("pair_kg_tail", N=2, C=384, K=160, Hi=9, Wi=10, Y=3, X=3, pad=(1, 1)), W256),
    (_mk("pair_groups2", N=2, C=512, K=256, Hi=8, Wi=9, Y=3, X=3, pad=(1, 1), stride=(1, 2), groups=2), W256),
    (_mk("pair_dil2_fill", N=4, C=256, K=256, Hi=12, Wi=12, Y=3, X=3, pad=(1, 1), stride=(2, 2), dil=(2, 2)), W256),
    (_mk("w512_short_last_block", N=3, C=1024, K=128, Hi=11, Wi=9, Y=3, X=3, pad=(1, 1), stride=(2, 2)), W512),
    (_mk("w512_one_block", N=1, C=512, K=64, Hi=8, Wi=8, Y=1, X=1), W512),
    # 144 tiles on 76 pairs: the accumulator released by 256-column halves
    # between a pair's tiles, with C/G = 1000 leaving the last tile's upper
    # half partly past C/G
    (_mk("w512_two_tiles_per_pair", N=8, C=1000, K=64, Hi=48, Wi=48, Y=1, X=1), W512),
]


@pytest.mark.parametrize("c,env", PAIR_CASES, ids=[c.name for c, _ in PAIR_CASES])
def test_pair_tile_variants(B, monkeypatch, c, env):
    g, dy, w = inputs(c)
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    for _ in range(2):  # the second run reuses the plan
        got, plan = gpu_dgrad(B, c, dy, w)
        assert plan.path()[0] == "tcgen05"
        tm, tn, sms = plan.tile()
        assert sms == 2 and tm == 256, plan.tile()  # SM pairs, 256-row tiles
        if "CONVBWD_DEBUG_BN" in env:
            assert tn == int(env["CONVBWD_DEBUG_BN"]), plan.tile()
        check_full(c, got, g, dy, w)


# C/G >= 256 layers where the planner's makespan estimate picks 1-SM 128 x 128
# tiles (at most 64 k-blocks per tile): 1-SM tiles by default, SM pairs under
# CONVBWD_DEBUG_2SM=1; both against the oracle.  Ragged M and N tails, several
# classes, a 64-k-block tile, a layer whose 1-SM tiles take two rounds (208
# tiles of four classes), a shallow 1x1 layer of 784 one-k-block tiles, and the
# 1x1 stride-2 benchmark layer.
ONE_SM_CASES = [
    _mk("one_round_1x1s2", N=4, C=512, K=384, Hi=14, Wi=14, Y=1, X=1, stride=(2, 2)),
    _mk("one_round_3x3_cg320", N=2, C=320, K=96, Hi=9, Wi=9, Y=3, X=3, pad=(1, 1)),
    _mk("one_round_3x3s2_classes", N=3, C=256, K=200, Hi=11, Wi=13, Y=3, X=3, pad=(1, 1), stride=(2, 2)),
    _mk("one_round_64_kblocks", N=1, C=384, K=4096, Hi=10, Wi=10, Y=1, X=1, stride=(2, 2)),
    _mk("two_rounds_3x3s2_32x14x14_512", N=32, C=512, K=512, Hi=14, Wi=14, Y=3, X=3, pad=(1, 1), stride=(2, 2)),
    _mk("shallow_1x1_16x56x56_c256_k64", N=16, C=256, K=64, Hi=56, Wi=56, Y=1, X=1),
    wl.case("bf16_32x14x14_1024"),
]


@pytest.mark.parametrize("pairs", [False, True])
@pytest.mark.parametrize("c", ONE_SM_CASES, ids=lambda c: c.name)
def test_one_sm_tile_layers(B, monkeypatch, c, pairs):
    if pairs:
        monkeypatch.setenv("CONVBWD_DEBUG_2SM", "1")
    g, dy, w = inputs(c)
    got, plan = gpu_dgrad(B, c, dy, w)
    assert plan.path()[0] == "tcgen05"
    if pairs:
        assert plan.tile()[2] == 2, plan.tile()
    else:
        assert plan.tile() == (128, 128, 1), plan.tile()
    check_full(c, got, g, dy, w)


# The plain-matrix specialisation of the SM-pair kernel (A = dy as the matrix
# {N*Ho*Wo, K}, 2-D tiled loads): the 1x2 stride-(1,2) layer, 1x1 stride-2
# layers, ragged M and N tails, 512- and 256-wide tiles, and the two benchmark
# workloads it applies to (whole dx).
PLAIN_CASES = [
    _mk("plain_1x2_s1x2", N=2, C=256, K=256, Hi=1, Wi=64, Y=1, X=2, stride=(1, 2)),
    _mk("plain_1x2_s1x2_w512", N=3, C=1024, K=192, Hi=1, Wi=90, Y=1, X=2, stride=(1, 2)),
    _mk("plain_1x1_s2_ragged", N=3, C=384, K=200, Hi=13, Wi=13, Y=1, X=1, stride=(2, 2)),
    _mk("plain_1x1_s1", N=2, C=512, K=128, Hi=9, Wi=7, Y=1, X=1),
    wl.case("bf16_16x1x512x2048"),
    wl.case("bf16_32x14x14_1024"),
]


@pytest.mark.parametrize("c", PLAIN_CASES, ids=lambda c: c.name)
def test_plain_matrix_specialisation(B, monkeypatch, c):
    monkeypatch.setenv("CONVBWD_DEBUG_A", "plain")
    g, dy, w = inputs(c)
    got, plan = gpu_dgrad(B, c, dy, w)
    assert plan.a_operand() == "plain" and plan.tile()[2] == 2, (plan.a_operand(), plan.tile())
    check_full(c, got, g, dy, w)


# Split-K with a reduce-scatter on the SM-pair kernel: S pairs per tile, each
# over 1/S of the k-blocks, exchanging fp32 partials so that each stores 1/S
# of the columns.  Ragged M (a 256-row block whose second CTA has no rows),
# ragged N (columns past C/G inside the last slice), 256- and 512-wide tiles,
# several classes and the dilated stress layer at full size; each plan runs
# twice (the second launch's flags carry a new epoch).
SPLIT_CASES = [
    (_mk("split2_deep", N=2, C=512, K=512, Hi=9, Wi=9, Y=3, X=3, pad=(1, 1), stride=(2, 2), dil=(2, 2)), 2),
    (_mk("split3_ragged_m", N=1, C=512, K=320, Hi=11, Wi=10, Y=3, X=3, pad=(1, 1), stride=(2, 2), dil=(2, 2)), 3),
    (_mk("split3_ragged_n", N=2, C=384, K=256, Hi=8, Wi=9, Y=3, X=3, pad=(1, 1)), 3),
    (_mk("split4_cg256", N=2, C=256, K=512, Hi=7, Wi=7, Y=3, X=3, pad=(1, 1), stride=(2, 2)), 4),
    # classes with 1 and 2 taps, rows of one residue uncovered (stride 3, 2 taps)
    (_mk("split2_multiclass_fill", N=2, C=512, K=256, Hi=13, Wi=11, Y=2, X=3, pad=(0, 1), stride=(3, 2)), 2),
    (wl.case("bf16_32x28x28x512"), 3),
]


@pytest.mark.parametrize("c,S", SPLIT_CASES, ids=[c.name + f"_S{S}" for c, S in SPLIT_CASES])
def test_split_k_reduce_scatter(B, monkeypatch, c, S):
    monkeypatch.setenv("CONVBWD_DEBUG_SPLITK", str(S))
    g, dy, w = inputs(c)
    plan = B.Plan.from_case(c)
    assert plan.path()[0] == "tcgen05" and plan.k_splits() == S, (plan.path(), plan.k_splits())
    dy_s, w_s, dx_s = plan.shapes()
    dyd, wd = to_dev(dy, c.dtype), to_dev(w, c.dtype)
    for _ in range(2):
        dx = torch.full(dx_s, float("nan"), dtype=torch.bfloat16, device="cuda")
        plan.run(dyd, wd, dx)
        st, det = plan.status()
        assert st == B.OK, (B.status_string(st), hex(det))
        check_full(c, dx.float().cpu().numpy().astype(np.float64), g, dy, w)


def test_deterministic_and_stream_ordered(B):
    c = TC_CASES[4]
    g, dy, w = inputs(c)
    s = torch.cuda.Stream()
    a, _ = gpu_dgrad(B, c, dy, w, stream=s)
    b, _ = gpu_dgrad(B, c, dy, w)
    np.testing.assert_array_equal(a, b)


def test_run_host_end_to_end(B):
    c = TC_CASES[0]
    g, dy, w = inputs(c)
    plan = B.Plan.from_case(c)
    dy_s, w_s, dx_s = plan.shapes()
    dy_h = torch.from_numpy(dy.view(np.int16)).view(torch.bfloat16).pin_memory()
    w_h = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).pin_memory()
    dx_h = torch.empty(dx_s, dtype=torch.bfloat16).pin_memory()
    dy_d = torch.empty(dy_s, dtype=torch.bfloat16, device="cuda")
    w_d = torch.empty(w_s, dtype=torch.bfloat16, device="cuda")
    dx_d = torch.empty(dx_s, dtype=torch.bfloat16, device="cuda")
    plan.run_host(dy_h, w_h, dx_h, dy_d, w_d, dx_d)
    torch.cuda.synchronize()
    check_full(c, dx_h.float().numpy().astype(np.float64), g, dy, w)


HOST_PIPE_CASES = [
    _mk("host_pipe_tail_2sm", N=7, C=512, K=512, Hi=40, Wi=40, Y=3, X=3, pad=(1, 1), sigma=0.05),
    _mk("host_pipe_fill", N=7, C=256, K=256, Hi=64, Wi=64, Y=3, X=3, pad=(1, 1), stride=(2, 2), dil=(2, 2),
        sigma=0.05),
]


@pytest.mark.parametrize("c", HOST_PIPE_CASES, ids=lambda c: c.name)
def test_run_host_pipelined_chunks(B, c):
    """run_host over batch chunks (chunks of 2 images plus a 1-image tail, each
    on its own plan, copies on the plan's copy streams): every image is
    computed and copied back, including the tail and the uncovered pixels."""
    g, dy, w = inputs(c)
    plan = B.Plan.from_case(c)
    dy_s, w_s, dx_s = plan.shapes()
    dy_h = torch.from_numpy(dy.view(np.int16)).view(torch.bfloat16).pin_memory()
    w_h = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).pin_memory()
    dx_h = torch.full(dx_s, float("nan"), dtype=torch.bfloat16).pin_memory()
    dy_d = torch.empty(dy_s, dtype=torch.bfloat16, device="cuda")
    w_d = torch.empty(w_s, dtype=torch.bfloat16, device="cuda")
    dx_d = torch.full(dx_s, float("nan"), dtype=torch.bfloat16, device="cuda")
    for _ in range(2):  # the second call reuses the chunk plans, streams and events
        plan.run_host(dy_h, w_h, dx_h, dy_d, w_d, dx_d)
        st, det = plan.status()
        assert st == B.OK, (B.status_string(st), hex(det))
        got = dx_h.float().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), "unwritten (NaN) outputs"
        check_full(c, got, g, dy, w)  # every chunk, the tail chunk's image included
        dx_h.fill_(float("nan"))


def test_overlap_and_alignment_errors(B):
    c = TC_CASES[1]
    plan = B.Plan.from_case(c)
    dy_s, w_s, dx_s = plan.shapes()
    buf = torch.zeros(int(np.prod(dx_s)) + int(np.prod(dy_s)) + 64, dtype=torch.bfloat16, device="cuda")
    base = buf.data_ptr()
    # dx overlapping dy
    assert plan.run_ptr(base, base + 4096, base + 2) == B.ERR_INVALID_ARG
    w = torch.zeros(w_s, dtype=torch.bfloat16, device="cuda")
    dxo = torch.zeros(int(np.prod(dx_s)) + 8, dtype=torch.bfloat16, device="cuda")
    # bf16 tensor-core path needs 16-byte aligned tensors
    dyt = torch.zeros(dy_s, dtype=torch.bfloat16, device="cuda")
    assert plan.run_ptr(dyt.data_ptr(), w.data_ptr(), dxo.data_ptr() + 2) == B.ERR_MISALIGNED
    torch.cuda.synchronize()


def test_bounded_wait_gives_up_and_context_survives(B):
    """A kernel waiting on a barrier that nothing arrives on gives up after its
    budget (~1 ms of SM clocks), records a timeout, and the device keeps
    working afterwards."""
    assert B.selftest_wait_timeout(2_000_000) == B.ERR_DEVICE_TIMEOUT
    c = TC_CASES[5]
    g, dy, w = inputs(c)
    got, _ = gpu_dgrad(B, c, dy, w)
    check_full(c, got, g, dy, w)


def test_per_kernel_timing(B):
    # tensor-core path: one launch (uncovered pixels are zeroed inside it)
    c = wl.case("bf16_32x28x28x512")
    plan = B.Plan.from_case(c)
    dy_s, w_s, dx_s = plan.shapes()
    dy = torch.zeros(dy_s, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(w_s, dtype=torch.bfloat16, device="cuda")
    dx = torch.empty(dx_s, dtype=torch.bfloat16, device="cuda")
    plan.set_timing(True)
    plan.run(dy, w, dx)
    f, m = plan.last_timing()
    assert f == 0 and m > 0
    # CUDA-core path with uncovered pixels: fill kernel + sub-GEMM kernel
    p2 = B.Plan(2, 16, 16, 15, 15, 1, 1, stride=(2, 2))
    assert p2.path() == ("simt", 2)
    dy_s, w_s, dx_s = p2.shapes()
    p2.set_timing(True)
    p2.run(torch.zeros(dy_s, device="cuda"), torch.zeros(w_s, device="cuda"), torch.empty(dx_s, device="cuda"))
    f, m = p2.last_timing()
    assert f > 0 and m > 0
