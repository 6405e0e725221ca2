"""CPU oracle for 2-D convolution backward-data (dgrad), fp64.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  The product library
never imports, links or calls it, and it imports nothing from the product.

The arithmetic lives in ``dgrad_oracle.c`` (plain C, double precision, an
OpenMP split over disjoint dx slices).  This module compiles it with gcc on
first use and marshals numpy arrays.  Inputs arrive as float32 arrays or as
bf16 bit patterns (uint16); both are widened exactly to float64 before any
arithmetic, so the oracle consumes the very values the GPU consumes.

Semantics (page "Non-unit stride input backward different input and
dispatches between BOO and Fusilli", torch-IR input,
``torch.aten.convolution_backward`` with output_mask [true, false, false]):
dx is the gradient of a forward cross-correlation with respect to its input,
see ``dgrad_oracle.c`` for the formula and the two layouts.

Pins (tests/test_oracle_pins.py, no GPU): the zero-insertion formulation, the
adjoint identity with an independent forward correlation, the closed-form
GEMM of 1x1 stride-1 filters, one-hot impulse responses (they fix the filter
flip), exact zeros on uncovered pixels, torch's own fp64 CPU
``conv_transpose2d``/``conv2d_input`` on random tiny shapes, the point
evaluation against the scatter loop, and hand-derived golden fixtures.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dgrad_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_dgrad.so")
_lock = threading.Lock()
_lib = None

LAYOUT_NCHW = 0  # dy [N][K][Ho][Wo], w [K][Cg][Y][X], dx [N][C][Hi][Wi]
LAYOUT_NHWC = 1  # dy [N][Ho][Wo][K], w [K][Y][X][Cg], dx [N][Hi][Wi][C]


class Geom(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "N", "C", "K", "Hi", "Wi", "Y", "X", "pad_h", "pad_w", "stride_h", "stride_w",
        "dil_h", "dil_w", "groups", "Ho", "Wo")]


def build(force: bool = False) -> str:
    """Compile the oracle shared object (gcc, -O2, OpenMP) if it is missing or stale."""
    global _lib
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c99",
                                   "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB_PATH)
            _lib = None
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.POINTER
        d = P(ctypes.c_double)
        g = P(Geom)
        i64 = ctypes.c_int64
        lib.oracle_out_dims.argtypes = [g]
        lib.oracle_out_dims.restype = ctypes.c_int
        lib.oracle_dgrad_scatter.argtypes = [g, ctypes.c_int, d, d, d, d, i64, i64, i64, i64]
        lib.oracle_dgrad_scatter.restype = None
        lib.oracle_dgrad_point.argtypes = [g, ctypes.c_int, d, d, i64, i64, i64, i64, d, d]
        lib.oracle_dgrad_point.restype = None
        lib.oracle_dgrad_zero_insert.argtypes = [g, ctypes.c_int, d, d, d]
        lib.oracle_dgrad_zero_insert.restype = ctypes.c_int
        lib.oracle_conv_fwd.argtypes = [g, ctypes.c_int, d, d, d]
        lib.oracle_conv_fwd.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def geom(N, C, K, Hi, Wi, Y, X, pad=(0, 0), stride=(1, 1), dil=(1, 1), groups=1) -> Geom:
    """Build and validate a geometry; fills the forward output size Ho, Wo."""
    g = Geom(N, C, K, Hi, Wi, Y, X, pad[0], pad[1], stride[0], stride[1], dil[0], dil[1], groups, 0, 0)
    if _load().oracle_out_dims(ctypes.byref(g)) != 0:
        raise ValueError("invalid convolution geometry")
    return g


def out_dims(g: Geom):
    return int(g.Ho), int(g.Wo)


def shapes(g: Geom, layout: int):
    """(dy, w, dx) shapes for a geometry in a layout."""
    Cg = g.C // g.groups
    if layout == LAYOUT_NCHW:
        return (g.N, g.K, g.Ho, g.Wo), (g.K, Cg, g.Y, g.X), (g.N, g.C, g.Hi, g.Wi)
    return (g.N, g.Ho, g.Wo, g.K), (g.K, g.Y, g.X, Cg), (g.N, g.Hi, g.Wi, g.C)


def widen(a: np.ndarray) -> np.ndarray:
    """float32 / float64 / bf16-bits(uint16) -> contiguous float64 (exact)."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def dgrad(g: Geom, layout: int, dy, w, n_range=None, c_range=None, with_absdot=True):
    """Scatter-loop dgrad.  Returns (dx, absdot) as float64 arrays in dx's shape.

    ``n_range=(a, b)`` restricts the work to images a..b-1 and
    ``c_range=(u, v)`` to channels u..v-1 within every group; entries outside
    the selection are left at zero.  Used for bounded samples of large
    problems.
    """
    dy_s, w_s, dx_s = shapes(g, layout)
    dy64 = widen(dy).reshape(dy_s)
    w64 = widen(w).reshape(w_s)
    dx = np.zeros(dx_s, dtype=np.float64)
    ab = np.zeros(dx_s, dtype=np.float64) if with_absdot else None
    a, b = (0, g.N) if n_range is None else n_range
    u, v = (0, g.C // g.groups) if c_range is None else c_range
    if not (0 <= a <= b <= g.N and 0 <= u <= v <= g.C // g.groups):
        raise ValueError("sample range outside the problem")
    _load().oracle_dgrad_scatter(ctypes.byref(g), layout, _ptr(dy64), _ptr(w64), _ptr(dx),
                                 _ptr(ab) if ab is not None else None, a, b, u, v)
    return dx, ab


def dgrad_points(g: Geom, layout: int, dy, w, points):
    """Gather-form dgrad at listed elements ``points`` = [(n, c, hi, wi), ...]."""
    dy_s, w_s, _ = shapes(g, layout)
    dy64 = widen(dy).reshape(dy_s)
    w64 = widen(w).reshape(w_s)
    lib = _load()
    vals = np.zeros(len(points))
    abss = np.zeros(len(points))
    v = ctypes.c_double()
    s = ctypes.c_double()
    for i, (n, c, hi, wi) in enumerate(points):
        lib.oracle_dgrad_point(ctypes.byref(g), layout, _ptr(dy64), _ptr(w64),
                               int(n), int(c), int(hi), int(wi), ctypes.byref(v), ctypes.byref(s))
        vals[i] = v.value
        abss[i] = s.value
    return vals, abss


def dgrad_zero_insert(g: Geom, layout: int, dy, w):
    """Zero-insertion formulation (tiny shapes only)."""
    dy_s, w_s, dx_s = shapes(g, layout)
    dy64 = widen(dy).reshape(dy_s)
    w64 = widen(w).reshape(w_s)
    dx = np.zeros(dx_s, dtype=np.float64)
    if _load().oracle_dgrad_zero_insert(ctypes.byref(g), layout, _ptr(dy64), _ptr(w64), _ptr(dx)) != 0:
        raise MemoryError("oracle_dgrad_zero_insert: allocation failed")
    return dx


def conv_fwd(g: Geom, layout: int, x, w):
    """Forward cross-correlation with the same geometry (x has dx's shape)."""
    dy_s, w_s, dx_s = shapes(g, layout)
    x64 = widen(x).reshape(dx_s)
    w64 = widen(w).reshape(w_s)
    out = np.zeros(dy_s, dtype=np.float64)
    _load().oracle_conv_fwd(ctypes.byref(g), layout, _ptr(x64), _ptr(w64), _ptr(out))
    return out


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def tolerance(ref: np.ndarray, absdot: np.ndarray, dtype: str) -> np.ndarray:
    """Per-element error bound.

    fp32 output:  |err| <= 1e-5 * sum|dy*w|
    bf16 output:  |err| <= 2^-8 * |ref| + 1e-4 * sum|dy*w|
    """
    if dtype == "f32":
        return 1e-5 * absdot
    if dtype == "bf16":
        return 2.0 ** -8 * np.abs(ref) + 1e-4 * absdot
    raise ValueError(dtype)
