"""Pins for the CPU oracle (no GPU).

The oracle is the fp64 scatter-loop definition of convolution backward-data
(grad_input of ``torch.aten.convolution_backward``, page "Non-unit stride
input backward different input and dispatches between BOO and Fusilli").
Each test below checks it against something other than itself:

* hand-derived golden values (tests/golden/hand_derived.json);
* the zero-insertion formulation of the BOO IR on the same page
  (``tensor.insert_slice`` with a stride, the ``1 - x`` filter flip, then a
  stride-1 correlation), generalised to pad and dilation;
* the adjoint identity <fwd(x, w), dy> = <x, dgrad(dy, w)> with an
  independent gather-loop forward correlation;
* the closed-form GEMM of 1x1 stride-1 filters (numpy matmul);
* one-hot impulse responses, which fix the direction of the filter flip;
* exact zeros (value and magnitude sum) on pixels that no tap reaches,
  counted by brute-force enumeration of the forward windows;
* torch's own fp64 CPU ``conv_transpose2d`` (a library routine);
* the gather-form point evaluation against the scatter loop.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from conv2d_backward_implicit_bwd_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_derived.json")


def _geom(c):
    return oracle.geom(c.N, c.C, c.K, c.Hi, c.Wi, c.Y, c.X, c.pad, c.stride, c.dil, c.groups)


def _valid(c):
    try:
        _geom(c)
        return True
    except ValueError:
        return False


def _layout(c):
    return oracle.LAYOUT_NCHW if c.layout == wl.NCHW else oracle.LAYOUT_NHWC


def _inputs(c):
    g = _geom(c)
    dy_s, w_s, _ = oracle.shapes(g, _layout(c))
    dy, w = wl.draw(c, dy_s, w_s)
    return g, dy, w


TINY = wl.random_tiny_cases(120, seed=11, accept=_valid)
TINY_NHWC = wl.random_tiny_cases(40, seed=12, layout=wl.NHWC, accept=_valid)


def test_golden_hand_derived():
    data = json.load(open(GOLDEN))
    for case in data["cases"]:
        gd = case["geom"]
        g = oracle.geom(gd["N"], gd["C"], gd["K"], gd["Hi"], gd["Wi"], gd["Y"], gd["X"],
                        tuple(gd["pad"]), tuple(gd["stride"]), tuple(gd["dil"]), gd["groups"])
        dy_s, w_s, dx_s = oracle.shapes(g, oracle.LAYOUT_NCHW)
        dy = np.array(case["dy"], dtype=np.float64).reshape(dy_s)
        w = np.array(case["w"], dtype=np.float64).reshape(w_s)
        dx, _ = oracle.dgrad(g, oracle.LAYOUT_NCHW, dy, w)
        np.testing.assert_array_equal(dx.reshape(-1), np.array(case["dx"], dtype=np.float64),
                                      err_msg=case["name"])


@pytest.mark.parametrize("c", TINY + TINY_NHWC, ids=lambda c: c.name + c.layout)
def test_zero_insertion_formulation(c):
    g, dy, w = _inputs(c)
    lay = _layout(c)
    dx, _ = oracle.dgrad(g, lay, dy, w)
    dz = oracle.dgrad_zero_insert(g, lay, dy, w)
    scale = max(1.0, np.abs(dx).max())
    assert np.abs(dx - dz).max() <= 1e-12 * scale


@pytest.mark.parametrize("c", TINY[:60] + TINY_NHWC[:20], ids=lambda c: c.name + c.layout)
def test_adjoint_identity(c):
    g, dy, w = _inputs(c)
    lay = _layout(c)
    _, _, dx_s = oracle.shapes(g, lay)
    rng = np.random.Generator(np.random.PCG64(c.seed + 1))
    x = rng.uniform(-1, 1, dx_s)
    lhs = float(np.sum(oracle.conv_fwd(g, lay, x, w) * oracle.widen(dy)))
    dx, _ = oracle.dgrad(g, lay, dy, w)
    rhs = float(np.sum(x * dx))
    mag = float(np.sum(np.abs(x) * np.abs(dx))) + 1e-30
    assert abs(lhs - rhs) <= 1e-12 * max(mag, 1.0)


@pytest.mark.parametrize("pad", [0, 1, 2])
@pytest.mark.parametrize("layout", [oracle.LAYOUT_NCHW, oracle.LAYOUT_NHWC])
def test_closed_form_gemm_1x1_stride1(pad, layout):
    N, C, K, H, W = 2, 5, 7, 4, 6
    g = oracle.geom(N, C, K, H, W, 1, 1, (pad, pad), (1, 1), (1, 1), 1)
    dy_s, w_s, _ = oracle.shapes(g, layout)
    rng = np.random.Generator(np.random.PCG64(7 + pad))
    dy = rng.uniform(-1, 1, dy_s)
    w = rng.uniform(-1, 1, w_s)
    dx, _ = oracle.dgrad(g, layout, dy, w)
    if layout == oracle.LAYOUT_NCHW:
        dyc = dy[:, :, pad:pad + H, pad:pad + W]                   # [N][K][H][W]
        ref = np.einsum("nkhw,kc->nchw", dyc, w[:, :, 0, 0])
    else:
        dyc = dy[:, pad:pad + H, pad:pad + W, :]                   # [N][H][W][K]
        ref = dyc.reshape(-1, K) @ w.reshape(K, C)
        ref = ref.reshape(N, H, W, C)
    np.testing.assert_allclose(dx, ref, rtol=0, atol=1e-13)


@pytest.mark.parametrize("geo", [
    dict(Hi=9, Wi=8, Y=3, X=2, pad=(1, 0), stride=(2, 3), dil=(1, 2)),
    dict(Hi=7, Wi=7, Y=5, X=5, pad=(2, 2), stride=(3, 3), dil=(1, 1)),
    dict(Hi=10, Wi=6, Y=3, X=3, pad=(1, 1), stride=(2, 2), dil=(2, 2)),
])
def test_impulse_response_fixes_flip(geo):
    """A one-hot dy at (n, k, ho, wo) must give w[k, :, y, x] at
    (ho*sh - ph + y*dh, wo*sw - pw + x*dw), clipped to dx: this fixes which
    way the filter is flipped (the Fusilli IR on the page has no flip)."""
    N, C, K = 1, 3, 2
    g = oracle.geom(N, C, K, geo["Hi"], geo["Wi"], geo["Y"], geo["X"], geo["pad"], geo["stride"], geo["dil"], 1)
    rng = np.random.Generator(np.random.PCG64(3))
    _, w_s, _ = oracle.shapes(g, oracle.LAYOUT_NCHW)
    w = rng.uniform(1, 2, w_s)  # strictly positive, all distinct
    for (k, ho, wo) in [(0, 0, 0), (1, g.Ho - 1, g.Wo - 1), (1, g.Ho // 2, 0)]:
        dy = np.zeros((N, K, g.Ho, g.Wo))
        dy[0, k, ho, wo] = 1.0
        dx, _ = oracle.dgrad(g, oracle.LAYOUT_NCHW, dy, w)
        exp = np.zeros_like(dx)
        for y in range(geo["Y"]):
            for x in range(geo["X"]):
                hi = ho * geo["stride"][0] - geo["pad"][0] + y * geo["dil"][0]
                wi = wo * geo["stride"][1] - geo["pad"][1] + x * geo["dil"][1]
                if 0 <= hi < geo["Hi"] and 0 <= wi < geo["Wi"]:
                    exp[0, :, hi, wi] = w[k, :, y, x]
        np.testing.assert_array_equal(dx, exp)


@pytest.mark.parametrize("c", TINY[:80], ids=lambda c: c.name)
def test_uncovered_pixels_exact_zero(c):
    g, dy, w = _inputs(c)
    dx, ab = oracle.dgrad(g, oracle.LAYOUT_NCHW, dy, w)
    hit = np.zeros((c.Hi, c.Wi), dtype=bool)
    for ho in range(g.Ho):
        for wo in range(g.Wo):
            for y in range(c.Y):
                for x in range(c.X):
                    hi = ho * c.stride[0] - c.pad[0] + y * c.dil[0]
                    wi = wo * c.stride[1] - c.pad[1] + x * c.dil[1]
                    if 0 <= hi < c.Hi and 0 <= wi < c.Wi:
                        hit[hi, wi] = True
    assert np.all(dx[:, :, ~hit] == 0.0)
    assert np.all(ab[:, :, ~hit] == 0.0)
    # where a tap lands the magnitude sum is positive (inputs are never 0 here)
    assert np.all(ab[:, :, hit] > 0.0)


@pytest.mark.parametrize("c", TINY, ids=lambda c: c.name)
def test_against_torch_fp64_conv_transpose(c):
    """torch.nn.grad.conv2d_input (conv_transpose2d underneath), fp64, CPU."""
    g, dy, w = _inputs(c)
    dx, _ = oracle.dgrad(g, oracle.LAYOUT_NCHW, dy, w)
    ref = torch.nn.grad.conv2d_input((c.N, c.C, c.Hi, c.Wi), torch.from_numpy(oracle.widen(w)),
                                     torch.from_numpy(oracle.widen(dy)), stride=c.stride, padding=c.pad,
                                     dilation=c.dil, groups=c.groups).numpy()
    scale = max(1.0, np.abs(ref).max())
    assert np.abs(dx - ref).max() <= 1e-12 * scale


@pytest.mark.parametrize("c", TINY_NHWC, ids=lambda c: c.name)
def test_nhwc_layout_matches_transposed_nchw(c):
    """The NHWC/KYXC oracle equals torch's fp64 result transposed."""
    g, dy, w = _inputs(c)
    dx, _ = oracle.dgrad(g, oracle.LAYOUT_NHWC, dy, w)
    dy_nchw = torch.from_numpy(oracle.widen(dy)).permute(0, 3, 1, 2)
    w_kcyx = torch.from_numpy(oracle.widen(w)).permute(0, 3, 1, 2)
    ref = torch.nn.grad.conv2d_input((c.N, c.C, c.Hi, c.Wi), w_kcyx.contiguous(), dy_nchw.contiguous(),
                                     stride=c.stride, padding=c.pad, dilation=c.dil,
                                     groups=c.groups).permute(0, 2, 3, 1).numpy()
    scale = max(1.0, np.abs(ref).max())
    assert np.abs(dx - ref).max() <= 1e-12 * scale


@pytest.mark.parametrize("c", TINY[:30] + TINY_NHWC[:10], ids=lambda c: c.name + c.layout)
def test_point_evaluation_matches_scatter(c):
    g, dy, w = _inputs(c)
    lay = _layout(c)
    dx, ab = oracle.dgrad(g, lay, dy, w)
    pts = [(n, ch, h, x) for n in range(c.N) for ch in range(c.C) for h in range(c.Hi) for x in range(c.Wi)]
    vals, abss = oracle.dgrad_points(g, lay, dy, w, pts)
    for (n, ch, h, x), v, a in zip(pts, vals, abss):
        idx = (n, ch, h, x) if lay == oracle.LAYOUT_NCHW else (n, h, x, ch)
        assert abs(dx[idx] - v) <= 1e-13 * max(1.0, abs(v))
        assert abs(ab[idx] - a) <= 1e-13 * max(1.0, a)


def test_batch_range_sampling_is_a_slice():
    c = wl.case("fp32_2x16x15x15")
    g, dy, w = _inputs(c)
    full, fab = oracle.dgrad(g, oracle.LAYOUT_NCHW, dy, w)
    part, pab = oracle.dgrad(g, oracle.LAYOUT_NCHW, dy, w, n_range=(1, 2))
    np.testing.assert_array_equal(part[1], full[1])
    np.testing.assert_array_equal(pab[1], fab[1])
    assert np.all(part[0] == 0)
    part2, _ = oracle.dgrad(g, oracle.LAYOUT_NCHW, dy, w, n_range=(0, 2), c_range=(3, 11))
    np.testing.assert_array_equal(part2[:, 3:11], full[:, 3:11])
    assert np.all(part2[:, :3] == 0) and np.all(part2[:, 11:] == 0)
    c2 = wl.random_tiny_cases(1, seed=5, accept=_valid)[0]
    c2 = wl.Case(**{**c2.__dict__, "C": 3 * 4, "groups": 3, "name": "grp"})
    g2, dy2, w2 = _inputs(c2)
    f2, _ = oracle.dgrad(g2, oracle.LAYOUT_NCHW, dy2, w2)
    p2, _ = oracle.dgrad(g2, oracle.LAYOUT_NCHW, dy2, w2, c_range=(1, 3))
    for gi in range(3):
        np.testing.assert_array_equal(p2[:, gi * 4 + 1:gi * 4 + 3], f2[:, gi * 4 + 1:gi * 4 + 3])


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.00390625, 1.005859375, 1.0078125, -2.5, 3.0e-3, 65504.0], dtype=np.float32)
    bits = wl.f32_to_bf16_bits(vals)
    back = wl.bf16_bits_to_f32(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa -> 1.0
    assert back[1] == 1.0
    # 1 + 3*2^-9 is above the tie -> 1 + 2^-7
    assert back[2] == np.float32(1.0078125)
    ref = torch.from_numpy(vals).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(back, ref)


def test_invalid_geometry_rejected():
    with pytest.raises(ValueError):
        oracle.geom(1, 4, 4, 2, 2, 5, 5)          # filter larger than padded input
    with pytest.raises(ValueError):
        oracle.geom(1, 3, 4, 8, 8, 3, 3, groups=2)  # C not divisible by groups
