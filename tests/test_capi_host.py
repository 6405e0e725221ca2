"""Host-side tests of the C ABI (no GPU): the library loads and exports every
declared symbol, and the planner's decomposition (residue classes, gemmIds,
coverage, useful work) agrees with brute-force enumeration of the forward
windows.  The brute force here is written from the forward index relation
hi = ho*sh - ph + y*dh, independently of the planner's closed forms."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

from conv2d_backward_implicit_bwd_gb300 import build as cbuild
from conv2d_backward_implicit_bwd_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    cbuild.build()
    from conv2d_backward_implicit_bwd_gb300 import binding
    return binding


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(conv_bwd_[a-z0-9_]+)\s*\(", txt,
                                re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(B):
    names = declared_functions()
    assert len(names) >= 15
    lib = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(B.EXPORTED) <= set(names)


def brute(c):
    """Per dim: which dx indices some tap reaches, and the useful tap count."""
    def dim(In, Out, F, s, d, p):
        hit = np.zeros(In, dtype=bool)
        useful = 0
        for o in range(Out):
            for f in range(F):
                i = o * s - p + f * d
                if 0 <= i < In:
                    hit[i] = True
                    useful += 1
        return hit, useful
    Ho = (c.Hi + 2 * c.pad[0] - c.dil[0] * (c.Y - 1) - 1) // c.stride[0] + 1
    Wo = (c.Wi + 2 * c.pad[1] - c.dil[1] * (c.X - 1) - 1) // c.stride[1] + 1
    rh, uh = dim(c.Hi, Ho, c.Y, c.stride[0], c.dil[0], c.pad[0])
    rw, uw = dim(c.Wi, Wo, c.X, c.stride[1], c.dil[1], c.pad[1])
    return Ho, Wo, rh, rw, uh, uw


def _ok(c):
    return (c.Hi + 2 * c.pad[0] - c.dil[0] * (c.Y - 1) - 1 >= 0 and
            c.Wi + 2 * c.pad[1] - c.dil[1] * (c.X - 1) - 1 >= 0)


PLAN_CASES = wl.CASES + wl.random_tiny_cases(150, seed=21, accept=_ok)


@pytest.mark.parametrize("c", PLAN_CASES, ids=lambda c: c.name)
def test_planner_against_brute_force(B, c):
    p = B.Plan.from_case(c)
    Ho, Wo, rh, rw, uh, uw = brute(c)
    assert (p.Ho, p.Wo) == (Ho, Wo)
    rows, cols = p.coverage()
    # a sub-GEMM writes exactly the rows/columns some tap reaches (classes are
    # not trimmed, so a written row may still receive only zeros: it is then
    # reached by a tap whose dy row is out of range -- never the case for a
    # row that no tap reaches at all)
    np.testing.assert_array_equal(rows, rh | _class_rows(c, 0))
    np.testing.assert_array_equal(cols, rw | _class_rows(c, 1))
    n = p.num_subgemms()
    infos = [p.subgemm(i) for i in range(n)]
    # consecutive gemmIds, distinct classes
    assert len({(s["ty"], s["tx"]) for s in infos}) == n
    # every written pixel is written by exactly one class: sum of M = N*rows*cols
    assert sum(s["M"] for s in infos) == c.N * int(rows.sum()) * int(cols.sum())
    g = math.gcd(c.stride[0], c.dil[0])
    YT = c.stride[0] // g
    g2 = math.gcd(c.stride[1], c.dil[1])
    XT = c.stride[1] // g2
    assert n <= YT * XT
    # the class's taps are y = ty + YT*j: all of them, and together every tap once
    assert sum(s["taps_y"] * s["taps_x"] for s in infos) <= c.Y * c.X
    for s in infos:
        assert s["taps_y"] == len(range(s["ty"], c.Y, YT))
        assert s["taps_x"] == len(range(s["tx"], c.X, XT))
        assert s["N"] == c.C // c.groups
        assert s["K"] == (c.K // c.groups) * s["taps_y"] * s["taps_x"]
    flop, nbytes = p.work()
    assert flop == 2.0 * c.N * c.K * (c.C // c.groups) * uh * uw
    es = 2 if c.dtype == wl.BF16 else 4
    assert nbytes == es * (c.N * c.K * Ho * Wo + c.K * (c.C // c.groups) * c.Y * c.X + c.N * c.C * c.Hi * c.Wi)


def _class_rows(c, dim):
    """Rows (dim 0) / columns (dim 1) of every residue class that has >= 1 tap,
    enumerated from hi = ht*s + t*d - p directly."""
    In, F, s, d, p = ((c.Hi, c.Y, c.stride[0], c.dil[0], c.pad[0]) if dim == 0 else
                      (c.Wi, c.X, c.stride[1], c.dil[1], c.pad[1]))
    T = s // math.gcd(s, d)
    out = np.zeros(In, dtype=bool)
    for t in range(min(T, F)):
        for ht in range(-In - p - t * d, In + p + 1):
            i = ht * s + t * d - p
            if 0 <= i < In:
                out[i] = True
    return out


def test_class_table_fp32_2x16x15x15(B):
    p = B.Plan.from_case(wl.case("fp32_2x16x15x15"))
    got = [(s["ty"], s["tx"], s["taps_y"] * s["taps_x"], s["M"]) for s in map(p.subgemm, range(p.num_subgemms()))]
    assert got == [(0, 0, 4, 98), (0, 1, 2, 112), (1, 0, 2, 112), (1, 1, 1, 128)]


def test_class_structure_of_strided_bf16_layers(B):
    a = B.Plan.from_case(wl.case("bf16_32x28x28x512"))   # stride 2, dilation 2: one class, 9 taps, 1/4 of dx written
    assert a.num_subgemms() == 1 and a.subgemm(0)["taps_y"] * a.subgemm(0)["taps_x"] == 9
    rows, cols = a.coverage()
    assert rows.sum() == 14 and cols.sum() == 14
    b = B.Plan.from_case(wl.case("bf16_32x14x14_1024"))   # 1x1 stride 2: one class of four non-empty
    assert b.num_subgemms() == 1 and b.subgemm(0)["M"] == 32 * 7 * 7
    c = B.Plan.from_case(wl.case("bf16_32x57x57x128"))   # 5x5 stride 3: nine classes
    taps = sorted(s["taps_y"] * s["taps_x"] for s in map(c.subgemm, range(c.num_subgemms())))
    assert taps == sorted([4, 4, 2, 4, 4, 2, 2, 2, 1])


def test_paths(B):
    assert B.Plan.from_case(wl.case("bf16_16x1x512x2048")).path()[0] == "tcgen05"
    assert B.Plan.from_case(wl.case("bf16_32x28x28x512")).path()[0] == "tcgen05"
    assert B.Plan.from_case(wl.case("fp32_2x16x15x15")).path()[0] == "simt"
    assert B.Plan.from_case(wl.case("bf16_resnext_64x56x56x256")).path() == ("grouped", 1)  # writes every pixel itself
    # launches per run: the tensor-core kernel zeroes uncovered pixels itself
    assert B.Plan.from_case(wl.case("bf16_16x1x512x2048")).path()[1] == 1
    assert B.Plan.from_case(wl.case("bf16_32x28x28x512")).path()[1] == 1
    # the CUDA-core path launches the fill kernel where some pixel is uncovered
    assert B.Plan(1, 4, 4, 9, 9, 1, 1, stride=(2, 2)).path() == ("simt", 2)


def test_narrow_group_kernel_selection(B, monkeypatch):
    """bf16 NHWC narrow groups: the banded tcgen05 kernel where C % 64 == 0,
    strides <= 2 and its staged band fits (every pixel written by one launch);
    otherwise the warp-MMA kernel (C/G in {8, 16}, G % 8 == 0) or the per-tap
    tcgen05 kernel (C/G = 32, <= 12 taps); the override picks one where it
    applies and falls back to the default order where it does not."""
    def kernel(*a, **kw):
        p = B.Plan(*a, layout="nhwc", dtype="bf16", **kw)
        return p.path(), p.grouped_kernel(), p.a_operand(), p.tile()
    band = (("grouped", 1), "band", "band", (128, 64, 1))
    assert kernel(64, 256, 256, 56, 56, 3, 3, pad=(1, 1), stride=(2, 2), groups=32) == band   # the ResNeXt layer
    assert kernel(2, 256, 256, 56, 56, 3, 3, pad=(1, 1), groups=32) == band                   # stride 1
    assert kernel(2, 512, 512, 9, 9, 3, 3, pad=(1, 1), stride=(2, 1), groups=32) == band      # C/G = 16, strides 2x1
    assert kernel(2, 256, 256, 9, 9, 3, 3, pad=(1, 1), stride=(2, 2), groups=8) == band       # C/G = 32
    # stride 3: warp MMA for C/G = 8, the per-tap tcgen05 kernel for C/G = 32
    assert kernel(2, 256, 256, 10, 9, 2, 2, pad=(0, 1), stride=(3, 3), groups=32)[1:3] == ("mma", "gather")
    assert kernel(2, 256, 256, 10, 9, 3, 3, pad=(1, 1), stride=(3, 3), groups=8)[1:3] == ("tc", "im2col")
    # 5x5 stride 1 (8 staged rows, 25 windows) fits; 7x7 (49 taps) is past the window table: warp MMA
    assert kernel(2, 256, 256, 9, 9, 5, 5, pad=(2, 2), groups=32) == band
    assert kernel(2, 256, 256, 9, 9, 7, 7, pad=(3, 3), groups=32)[1] == "mma"
    # one 64-channel block; C % 64 != 0 with G % 8 != 0 has no narrow-group kernel (CUDA cores)
    assert kernel(2, 64, 64, 9, 9, 3, 3, pad=(1, 1), stride=(2, 2), groups=8) == band
    assert kernel(2, 96, 96, 9, 9, 3, 3, pad=(1, 1), stride=(2, 2), groups=12)[0][0] == "simt"
    # overrides
    monkeypatch.setenv("CONVBWD_DEBUG_GROUPED", "mma")
    assert kernel(2, 256, 256, 9, 9, 3, 3, pad=(1, 1), stride=(2, 2), groups=32)[1:4] == ("mma", "gather", (0, 0, 1))
    assert kernel(2, 256, 256, 9, 9, 3, 3, pad=(1, 1), stride=(2, 2), groups=8)[1] == "band"  # C/G = 32: no mma
    monkeypatch.setenv("CONVBWD_DEBUG_GROUPED", "tc")
    assert kernel(2, 256, 256, 9, 9, 3, 3, pad=(1, 1), stride=(2, 2), groups=32)[1:4] == ("tc", "im2col", (128, 64, 1))
    # not on the narrow-group path
    monkeypatch.delenv("CONVBWD_DEBUG_GROUPED")
    assert B.Plan.from_case(wl.case("bf16_16x1x512x2048")).grouped_kernel() == ""


def test_fp32_tensor_core_path_selection(B, monkeypatch):
    """fp32 NHWC problems above 1e9 useful FLOP take the three-term TF32
    tensor-core path (filter split + one kernel, which zeroes uncovered pixels
    itself); smaller ones, shapes outside its alignment and group rules, and
    NCHW plans without a device stay on the CUDA cores."""
    big = B.Plan.from_case(wl.case("fp32_nhwc_32x28x28x512"))
    assert big.path() == ("tf32", 2) and big.tile() == (128, 128, 1)
    assert B.Plan(2, 64, 64, 14, 14, 3, 3, pad=(1, 1), layout="nhwc").path()[0] == "simt"       # 0.03 GFLOP
    assert B.Plan(8, 254, 256, 28, 28, 3, 3, pad=(1, 1), layout="nhwc").path()[0] == "simt"     # C % 4 != 0
    assert B.Plan(8, 256, 256, 28, 28, 3, 3, pad=(1, 1), groups=16, layout="nhwc").path()[0] == "simt"  # K/G = 16
    assert B.Plan(16, 256, 256, 28, 28, 3, 3, pad=(1, 1), groups=8, layout="nhwc").path()[0] == "tf32"  # K/G = 32
    monkeypatch.setenv("CONVBWD_DEBUG_PATH", "tf32")
    assert B.Plan(2, 64, 64, 14, 14, 3, 3, pad=(1, 1), layout="nhwc").path() == ("tf32", 2)
    monkeypatch.setenv("CONVBWD_DEBUG_PATH", "simt")
    assert B.Plan.from_case(wl.case("fp32_nhwc_32x28x28x512")).path()[0] == "simt"


@pytest.mark.parametrize("kw,status", [
    (dict(N=0), 1), (dict(C=3, groups=2), 1), (dict(Y=40), 1), (dict(stride=(0, 1)), 1),
    (dict(pad=(-1, 0)), 1), (dict(dil=(1, 0)), 1), (dict(stride=(65, 1)), 2), (dict(layout=7), 1),
    (dict(dtype=9), 1),
])
def test_invalid_descriptors(B, kw, status):
    args = dict(N=1, C=4, K=4, Hi=8, Wi=8, Y=3, X=3, pad=(1, 1), stride=(1, 1), dil=(1, 1), groups=1,
                layout="nchw", dtype="f32")
    args.update(kw)
    with pytest.raises(B.ConvBwdError) as e:
        B.Plan(**args)
    assert e.value.status == status


def test_run_argument_errors_without_device(B):
    p = B.Plan(1, 4, 4, 8, 8, 3, 3, (1, 1))
    assert p.run_ptr(0, 0, 0) == B.ERR_INVALID_ARG
    import torch
    if not torch.cuda.is_available():
        # a plan made without a device cannot run
        assert p.run_ptr(4096, 8192, 1 << 20) == B.ERR_CUDA


def test_forward_entry_host_checks(B):
    """conv_bwd_data_run_forward rejects unsupported plans before touching a device."""
    assert B.Plan(1, 64, 64, 8, 8, 3, 3, (1, 1), dtype="f32").run_forward_ptr(4096, 8192, 1 << 20) == B.ERR_UNSUPPORTED
    narrow = B.Plan(1, 64, 64, 8, 8, 3, 3, (1, 1), groups=2, layout="nhwc", dtype="bf16")  # C/G = 32
    assert narrow.run_forward_ptr(4096, 8192, 1 << 20) == B.ERR_UNSUPPORTED
    ok = B.Plan(1, 64, 64, 8, 8, 3, 3, (1, 1), layout="nhwc", dtype="bf16")
    assert ok.run_forward_ptr(0, 8192, 1 << 20) == B.ERR_INVALID_ARG
    import torch
    if not torch.cuda.is_available():
        assert ok.run_forward_ptr(4096, 8192, 1 << 20) == B.ERR_CUDA


def test_status_strings(B):
    for s in range(7):
        assert B.status_string(s).startswith("CONV_BWD_")
    assert B.lib().conv_bwd_data_version() >= 100


def test_few_tile_layers_take_1sm_tiles(B, monkeypatch):
    """C/G >= 256: 1-SM 128 x 128 tiles where the planner's makespan estimate
    (tiles dealt in snake order to the SMs, or the SM pairs, at the measured
    clocks per k-block and per epilogue) favours them and a tile has at most
    64 k-blocks; SM pairs otherwise, or under any SM-pair override.  Planning
    without a device assumes 148 SMs."""
    assert B.Plan.from_case(wl.case("bf16_32x14x14_1024")).tile() == (128, 128, 1)   # 13 x 8 tiles, 32 k-blocks
    assert B.Plan.from_case(wl.case("bf16_16x1x512x2048")).tile()[2] == 2          # 2 x 32 x 16 tiles
    assert B.Plan.from_case(wl.case("bf16_32x28x28x512")).tile()[2] == 2           # 72 k-blocks per tile
    one = dict(layout="nhwc", dtype="bf16", stride=(2, 2))
    assert B.Plan(32, 1024, 4096, 14, 14, 1, 1, **one).tile() == (128, 128, 1)    # 64 k-blocks
    assert B.Plan(32, 1024, 4160, 14, 14, 1, 1, **one).tile()[2] == 2             # 65 k-blocks
    assert B.Plan(46, 1024, 2048, 14, 14, 1, 1, **one).tile() == (128, 128, 1)    # 18 x 8 = 144 tiles
    assert B.Plan(64, 1024, 2048, 14, 14, 1, 1, **one).tile()[2] == 2             # 25 x 8 tiles: two rounds
    # 3x3 stride 2: four classes of 32, 16, 16 and 8 k-blocks; the second
    # round of 1-SM tiles holds only the cheapest class
    assert B.Plan(32, 512, 512, 14, 14, 3, 3, pad=(1, 1), **one).tile() == (128, 128, 1)
    # a 1x1 layer of one k-block per tile runs at its epilogues' pace, where the
    # 1-SM tiles are faster; with 16 k-blocks per tile the pairs' wider tiles win
    plain = dict(layout="nhwc", dtype="bf16")
    assert B.Plan(64, 256, 64, 56, 56, 1, 1, **plain).tile() == (128, 128, 1)
    assert B.Plan(64, 256, 1024, 56, 56, 1, 1, **plain).tile()[2] == 2
    assert B.Plan(32, 256, 256, 28, 28, 3, 3, pad=(1, 1), **plain).tile()[2] == 2   # 36 k-blocks, 2 rounds
    for k, v in (("CONVBWD_DEBUG_2SM", "1"), ("CONVBWD_DEBUG_BN", "256"), ("CONVBWD_DEBUG_A", "plain")):
        monkeypatch.setenv(k, v)
        assert B.Plan.from_case(wl.case("bf16_32x14x14_1024")).tile()[2] == 2, k
        monkeypatch.delenv(k)


@pytest.mark.parametrize("name,eligible", [("bf16_16x1x512x2048", True), ("bf16_32x14x14_1024", True),
                                           ("bf16_32x28x28x512", False), ("bf16_32x57x57x128", False)])
def test_plain_matrix_specialisation_eligibility(B, monkeypatch, name, eligible):
    """The plain-matrix A specialisation applies only where every class has one
    tap and its rows are all of dy's pixels in order (checked here by
    enumerating the classes); it is selected by the override, never by
    default."""
    c = wl.case(name)
    p = B.Plan.from_case(c)
    assert p.a_operand() == "im2col"
    classes = [p.subgemm(i) for i in range(p.num_subgemms())]
    # one tap per class and M = every dy pixel (a class with fewer rows would
    # skip pixels; one tap with M = N*Ho*Wo means row m reads dy pixel m)
    plain = all(k["taps_y"] == 1 and k["taps_x"] == 1 and k["M"] == c.N * p.Ho * p.Wo for k in classes)
    assert plain == eligible
    monkeypatch.setenv("CONVBWD_DEBUG_A", "plain")
    q = B.Plan.from_case(c)
    assert q.a_operand() == ("plain" if eligible else "im2col")
