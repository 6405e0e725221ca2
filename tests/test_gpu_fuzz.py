"""Randomised GPU parity (seeded): moderate random geometries on every kernel
path, each compared element by element with the fp64 oracle, plus the two
extra shapes of the tested driver command lines in "Backward data" (14x14 ...
20x20 with 1x1 filters and pad 1: H = 18 and H = 20 are not among the five
benchmark configs).  Tolerances as in test_gpu_parity.py."""
import numpy as np
import pytest
import torch

import oracle
from conv2d_backward_implicit_bwd_gb300 import workloads as wl

from test_gpu_parity import B, check_full, gpu_dgrad, inputs  # noqa: F401  (fixture + helpers)

pytestmark = pytest.mark.gpu

P1_EXTRA = [
    wl.Case(name=f"p1_{h}x{h}_1x1_p1", N=32, C=32, K=32, Hi=h, Wi=h, Y=1, X=1, pad=(1, 1), dtype=wl.F32,
            layout=wl.NCHW, dist="uniform", seed=2100 + h) for h in (18, 20)
]


@pytest.mark.parametrize("c", P1_EXTRA, ids=lambda c: c.name)
def test_p1_extra_shapes(B, c):
    g, dy, w = inputs(c)
    got, plan = gpu_dgrad(B, c, dy, w)
    check_full(c, got, g, dy, w)


def _ok(c):
    return (c.Hi + 2 * c.pad[0] - c.dil[0] * (c.Y - 1) - 1 >= 0 and
            c.Wi + 2 * c.pad[1] - c.dil[1] * (c.X - 1) - 1 >= 0)


def fuzz_cases(kind, count, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    while len(out) < count:
        sh, sw = int(rng.integers(1, 5)), int(rng.integers(1, 5))
        dh, dw = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        ph, pw = int(rng.integers(0, 4)), int(rng.integers(0, 4))
        Y, X = int(rng.integers(1, 6)), int(rng.integers(1, 6))
        Hi, Wi = int(rng.integers(3, 21)), int(rng.integers(3, 21))
        N = int(rng.integers(1, 4))
        if kind == "tc":          # bf16 NHWC, C/G >= 64 (1-SM and 2-SM tensor-core kernels)
            G = int(rng.choice([1, 1, 1, 2]))
            Cg = int(rng.choice([64, 128, 192, 256, 320]))
            Kg = 8 * int(rng.integers(1, 25))
            dtype, layout = wl.BF16, wl.NHWC
        elif kind == "band":      # bf16 NHWC, C/G = K/G in {8, 16, 32}, C % 64 == 0, strides <= 2
            sh, sw = int(rng.integers(1, 3)), int(rng.integers(1, 3))
            dh, dw = int(rng.integers(1, 3)), int(rng.integers(1, 3))
            Y, X = int(rng.integers(1, 5)), int(rng.integers(1, 5))
            Cg = int(rng.choice([8, 16, 32]))
            Kg = Cg
            G = (64 // Cg) * int(rng.integers(1, 4))
            Wi = int(rng.integers(3, 80))
            dtype, layout = wl.BF16, wl.NHWC
        elif kind == "grouped":   # bf16 NHWC, C/G = K/G in {8, 16}
            Cg = int(rng.choice([8, 16]))
            Kg = Cg
            G = 8 * int(rng.integers(1, 5))
            Y, X = int(rng.integers(1, 5)), int(rng.integers(1, 5))
            dtype, layout = wl.BF16, wl.NHWC
        elif kind == "simt_tap":  # fp32 CUDA-core kernel, K/G a multiple of 16 (slices within one tap)
            G = int(rng.integers(1, 4))
            Cg, Kg = int(rng.integers(1, 80)), 16 * int(rng.integers(1, 4))
            dtype, layout = wl.F32, (wl.NCHW if rng.integers(2) else wl.NHWC)
        else:                     # fp32 CUDA-core kernel, either layout
            G = int(rng.integers(1, 4))
            Cg, Kg = int(rng.integers(1, 40)), int(rng.integers(1, 40))
            dtype, layout = wl.F32, (wl.NCHW if rng.integers(2) else wl.NHWC)
        c = wl.Case(name=f"{kind}{len(out)}", N=N, C=G * Cg, K=G * Kg, Hi=Hi, Wi=Wi, Y=Y, X=X, pad=(ph, pw),
                    stride=(sh, sw), dil=(dh, dw), groups=G, dtype=dtype, layout=layout,
                    dist="uniform" if dtype == wl.F32 else "normal", sigma=0.5, seed=seed * 1000 + len(out))
        if _ok(c) and (kind != "band" or _band_stage_bytes(c) <= 40 * 1024):
            out.append(c)
    return out


def _band_stage_bytes(c):
    """Shared memory of one staged band of the banded narrow-group kernel: 4
    output rows plus the row offsets' span, 32 pixels x 128 bytes per row."""
    def offsets(s, p, d, F):
        return [(r + p - f * d) // s for r in range(s) for f in range(F) if (r + p - f * d) % s == 0]
    oy = offsets(c.stride[0], c.pad[0], c.dil[0], c.Y)
    return (4 + max(oy) - min(oy)) * 32 * 128


FUZZ = (fuzz_cases("tc", 24, 71) + fuzz_cases("grouped", 10, 72) + fuzz_cases("band", 30, 74) +
        fuzz_cases("simt", 10, 73) + fuzz_cases("simt_tap", 12, 75))


@pytest.mark.parametrize("c", FUZZ, ids=lambda c: c.name)
def test_fuzz_against_oracle(B, c):
    g, dy, w = inputs(c)
    got, plan = gpu_dgrad(B, c, dy, w)
    if c.name.startswith("band"):
        assert plan.grouped_kernel() == "band", (plan.path(), plan.grouped_kernel())
    check_full(c, got, g, dy, w)


# The C/G >= 256 draws are small enough that the planner gives them 1-SM
# tiles: run them again on SM pairs (those with im2col A loads: K/G a multiple
# of 64 when G > 1).
FUZZ_PAIRS = [c for c in FUZZ if c.name.startswith("tc") and c.C // c.groups >= 256 and
              (c.groups == 1 or (c.K // c.groups) % 64 == 0)]


@pytest.mark.parametrize("c", FUZZ_PAIRS, ids=lambda c: c.name + "_pairs")
def test_fuzz_on_sm_pairs(B, monkeypatch, c):
    monkeypatch.setenv("CONVBWD_DEBUG_2SM", "1")
    g, dy, w = inputs(c)
    got, plan = gpu_dgrad(B, c, dy, w)
    assert plan.tile()[2] == 2, plan.tile()
    check_full(c, got, g, dy, w)
