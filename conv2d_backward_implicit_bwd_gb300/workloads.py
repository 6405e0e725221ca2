"""Seeded synthetic workloads: case definitions and input generators.

This module holds no convolution arithmetic.  It only names the problem
shapes and draws the input tensors, so that the CUDA path, the CPU oracle,
the tests and the benchmark all consume byte-identical inputs.

Recipe (one ``numpy.random.Generator(PCG64(seed))`` per case, seed =
1000*config + subcase, dy drawn first, then w):
  * fp32 cases: ``uniform(-1, 1)`` rounded to float32;
  * bf16 cases: ``standard_normal() * sigma`` as float32, then rounded to
    bf16 with round-to-nearest-even, stored as uint16 bit patterns.

Shapes follow the pages: the "padding issue" sweep in "Backward data" (the
rocMLIR pull request's list of tested driver command lines), the dgrad shape
of "Non-unit stride input backward different input and dispatches between BOO
and Fusilli", and a ResNeXt-50-style grouped layer (named as a workload in
"[igemm_dynamic] v4r1 bwd dynamic kernel"; shapes only, no weights).
"""
from __future__ import annotations

from dataclasses import dataclass, field, asdict

import numpy as np

F32 = "f32"
BF16 = "bf16"
NCHW = "nchw"  # dy [N][K][Ho][Wo], w [K][C/G][Y][X], dx [N][C][Hi][Wi]
NHWC = "nhwc"  # dy [N][Ho][Wo][K], w [K][Y][X][C/G], dx [N][Hi][Wi][C]


@dataclass(frozen=True)
class Case:
    name: str
    N: int
    C: int
    K: int
    Hi: int
    Wi: int
    Y: int
    X: int
    pad: tuple = (0, 0)
    stride: tuple = (1, 1)
    dil: tuple = (1, 1)
    groups: int = 1
    dtype: str = F32
    layout: str = NCHW
    dist: str = "uniform"       # "uniform" -> U[-1,1]; "normal" -> N(0,1)*sigma
    sigma: float = 1.0
    seed: int = 0
    tags: tuple = field(default=())

    def desc(self) -> dict:
        d = asdict(self)
        for k in ("dist", "sigma", "seed", "tags", "name"):
            d.pop(k)
        return d


def _sweep():
    base = dict(N=32, C=32, K=32, groups=1, dtype=F32, layout=NCHW, dist="uniform")
    rows = [(14, 1, 1, 1), (14, 3, 1, 1), (15, 1, 1, 1), (16, 1, 1, 1), (14, 3, 1, 2)]
    out = []
    for i, (h, f, p, s) in enumerate(rows):
        out.append(Case(name=f"fp32_32x32x{h}x{h}_{f}x{f}_p{p}_s{s}", Hi=h, Wi=h, Y=f, X=f,
                        pad=(p, p), stride=(s, s), seed=2000 + i, tags=("fp32_small",), **base))
    return out


CASES = [
    Case(name="fp32_2x16x15x15_3x3_p1_s2", N=2, C=16, K=16, Hi=15, Wi=15, Y=3, X=3, pad=(1, 1),
         stride=(2, 2), dtype=F32, layout=NCHW, dist="uniform", seed=1000, tags=("fp32_small",)),
    *_sweep(),
    Case(name="bf16_16x1x512x2048_1x2_s1x2", N=16, C=2048, K=2048, Hi=1, Wi=512, Y=1, X=2,
         pad=(0, 0), stride=(1, 2), dtype=BF16, layout=NHWC, dist="normal", sigma=0.02, seed=3000,
         tags=("large",)),
    Case(name="bf16_resnext_64x56x56x256_g32_3x3_s2", N=64, C=256, K=256, Hi=56, Wi=56, Y=3, X=3,
         pad=(1, 1), stride=(2, 2), groups=32, dtype=BF16, layout=NHWC, dist="normal", sigma=0.05,
         seed=4000, tags=("grouped",)),
    Case(name="bf16_32x28x28x512_3x3_s2_p1_d2", N=32, C=512, K=512, Hi=28, Wi=28, Y=3, X=3,
         pad=(1, 1), stride=(2, 2), dil=(2, 2), dtype=BF16, layout=NHWC, dist="normal", sigma=0.05,
         seed=5000, tags=("large",)),
    Case(name="bf16_32x14x14_1024_2048_1x1_s2", N=32, C=1024, K=2048, Hi=14, Wi=14, Y=1, X=1,
         pad=(0, 0), stride=(2, 2), dtype=BF16, layout=NHWC, dist="normal", sigma=0.05, seed=5001,
         tags=("ridge",)),
    Case(name="bf16_32x57x57x128_5x5_s3_p2", N=32, C=128, K=128, Hi=57, Wi=57, Y=5, X=5,
         pad=(2, 2), stride=(3, 3), dtype=BF16, layout=NHWC, dist="normal", sigma=0.05, seed=5002,
         tags=("ridge",)),
    # fp32 problems large enough for the fp32 tensor-core path: the dilated
    # stress shape in fp32 (NHWC, and NCHW as the fp32 sweep is laid out), and
    # the 3x3 stride-1 sweep shape with 256 channels
    Case(name="fp32_nhwc_32x28x28x512_3x3_s2_p1_d2", N=32, C=512, K=512, Hi=28, Wi=28, Y=3, X=3,
         pad=(1, 1), stride=(2, 2), dil=(2, 2), dtype=F32, layout=NHWC, dist="uniform", seed=6000,
         tags=("fp32_large",)),
    Case(name="fp32_nchw_32x28x28x512_3x3_s2_p1_d2", N=32, C=512, K=512, Hi=28, Wi=28, Y=3, X=3,
         pad=(1, 1), stride=(2, 2), dil=(2, 2), dtype=F32, layout=NCHW, dist="uniform", seed=6001,
         tags=("fp32_large",)),
    Case(name="fp32_nchw_32x256x14x14_3x3_p1_s1", N=32, C=256, K=256, Hi=14, Wi=14, Y=3, X=3,
         pad=(1, 1), dtype=F32, layout=NCHW, dist="uniform", seed=6002, tags=("fp32_large",)),
]

BY_NAME = {c.name: c for c in CASES}


def case(name: str) -> Case:
    """A workload by its name or by a prefix of it that only one name has."""
    if name in BY_NAME:
        return BY_NAME[name]
    hits = [c for c in CASES if c.name.startswith(name)]
    if len(hits) == 1:
        return hits[0]
    raise KeyError(name)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round-to-nearest-even.

    NaN inputs are not expected (the generators never produce them)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def draw(c: Case, dy_shape, w_shape, seed: int | None = None):
    """Draw (dy, w) for case ``c`` with the given tensor shapes.

    Returns float32 arrays for fp32 cases and uint16 bf16 bit patterns for
    bf16 cases.  The shapes are supplied by the caller (they depend on the
    forward output size, which this module does not compute)."""
    rng = np.random.Generator(np.random.PCG64(c.seed if seed is None else seed))
    ndy = int(np.prod(dy_shape))
    nw = int(np.prod(w_shape))
    if c.dist == "uniform":
        dy = rng.uniform(-1.0, 1.0, ndy).astype(np.float32)
        w = rng.uniform(-1.0, 1.0, nw).astype(np.float32)
    else:
        dy = (rng.standard_normal(ndy, dtype=np.float32) * np.float32(c.sigma)).astype(np.float32)
        w = (rng.standard_normal(nw, dtype=np.float32) * np.float32(c.sigma)).astype(np.float32)
    if c.dtype == BF16:
        return f32_to_bf16_bits(dy).reshape(dy_shape), f32_to_bf16_bits(w).reshape(w_shape)
    return dy.reshape(dy_shape), w.reshape(w_shape)


def random_tiny_cases(count: int, seed: int, dtype=F32, layout=NCHW, max_groups=3, accept=None):
    """Random small geometries: stride 1-4, dilation 1-3, pad 0-3, filter 1-5,
    groups 1..max_groups, spatial sizes 1-11 (including ones below the filter
    extent).  ``accept(case) -> bool`` lets the caller drop geometries it
    cannot use (for instance ones whose forward output would be empty)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    tries = 0
    while len(out) < count and tries < 100 * count:
        tries += 1
        G = int(rng.integers(1, max_groups + 1))
        Cg = int(rng.integers(1, 4))
        Kg = int(rng.integers(1, 4))
        Y, X = int(rng.integers(1, 6)), int(rng.integers(1, 6))
        sh, sw = int(rng.integers(1, 5)), int(rng.integers(1, 5))
        dh, dw = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        ph, pw = int(rng.integers(0, 4)), int(rng.integers(0, 4))
        Hi, Wi = int(rng.integers(1, 12)), int(rng.integers(1, 12))
        c = Case(name=f"tiny{len(out)}", N=int(rng.integers(1, 3)), C=G * Cg, K=G * Kg, Hi=Hi, Wi=Wi,
                 Y=Y, X=X, pad=(ph, pw), stride=(sh, sw), dil=(dh, dw), groups=G, dtype=dtype,
                 layout=layout, dist="uniform" if dtype == F32 else "normal", sigma=0.5,
                 seed=seed * 7919 + len(out))
        if accept is not None and not accept(c):
            continue
        out.append(c)
    return out
