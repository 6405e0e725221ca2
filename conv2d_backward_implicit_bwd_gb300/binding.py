"""Thin ctypes binding of the C ABI in include/conv_bwd_data.h.

Argument marshalling only: every step of the computation runs in the CUDA
library ``lib/libconv_bwd_data.so``.  Tensors are PyTorch tensors (device
memory and streams); only their data pointers cross the boundary.  If the
library is missing, importing this module raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "libconv_bwd_data.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_MISALIGNED, ERR_CUDA, ERR_DEVICE_TIMEOUT, ERR_DEVICE_FAULT = range(7)
F32, BF16 = 0, 1
NCHW_GKCYX, NHWC_KYXC = 0, 1
PATH_TCGEN05, PATH_SIMT, PATH_GROUPED, PATH_TF32 = 0, 1, 2, 3
PATH_NAMES = {PATH_TCGEN05: "tcgen05", PATH_SIMT: "simt", PATH_GROUPED: "grouped", PATH_TF32: "tf32"}

EXPORTED = [
    "conv_bwd_data_create", "conv_bwd_data_destroy", "conv_bwd_data_out_dims", "conv_bwd_data_num_subgemms",
    "conv_bwd_data_subgemm_info", "conv_bwd_data_coverage", "conv_bwd_data_path", "conv_bwd_data_tile", "conv_bwd_data_work",
    "conv_bwd_data_run", "conv_bwd_data_run_host", "conv_bwd_data_get_status", "conv_bwd_data_set_timing",
    "conv_bwd_data_last_timing", "conv_bwd_data_selftest_wait_timeout", "conv_bwd_status_string",
    "conv_bwd_data_version", "conv_bwd_data_run_noalloc", "conv_bwd_data_run_forward", "conv_bwd_data_a_operand",
    "conv_bwd_data_k_splits", "conv_bwd_data_grouped_kernel",
]


class ConvBwdError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)}")
        self.status = status


class Desc(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("C", ctypes.c_int64), ("K", ctypes.c_int64), ("Hi", ctypes.c_int64),
                ("Wi", ctypes.c_int64), ("Y", ctypes.c_int64), ("X", ctypes.c_int64),
                ("pad_h", ctypes.c_int32), ("pad_w", ctypes.c_int32), ("stride_h", ctypes.c_int32),
                ("stride_w", ctypes.c_int32), ("dil_h", ctypes.c_int32), ("dil_w", ctypes.c_int32),
                ("groups", ctypes.c_int32), ("layout", ctypes.c_int32), ("dtype", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"CUDA library not built: {LIB_PATH} (run conv2d_backward_implicit_bwd_gb300.build)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    P = ctypes.POINTER
    sig = {
        "conv_bwd_data_create": [P(Desc), P(vp)],
        "conv_bwd_data_destroy": [vp],
        "conv_bwd_data_out_dims": [vp, P(i64), P(i64)],
        "conv_bwd_data_num_subgemms": [vp, P(i32)],
        "conv_bwd_data_subgemm_info": [vp, i32, P(i32), P(i32), P(i64), P(i64), P(i64), P(i32), P(i32)],
        "conv_bwd_data_coverage": [vp, vp, vp],
        "conv_bwd_data_path": [vp, P(i32), P(i32)],
        "conv_bwd_data_tile": [vp, P(i32), P(i32), P(i32)],
        "conv_bwd_data_work": [vp, P(ctypes.c_double), P(ctypes.c_double)],
        "conv_bwd_data_a_operand": [vp, P(i32)],
        "conv_bwd_data_k_splits": [vp, P(i32)],
        "conv_bwd_data_grouped_kernel": [vp, P(i32)],
        "conv_bwd_data_run": [vp, vp, vp, vp, vp],
        "conv_bwd_data_run_forward": [vp, vp, vp, vp, vp],
        "conv_bwd_data_run_host": [vp, vp, vp, vp, vp, vp, vp, vp],
        "conv_bwd_data_get_status": [vp, vp, P(i32)],
        "conv_bwd_data_set_timing": [vp, i32],
        "conv_bwd_data_last_timing": [vp, P(ctypes.c_float), P(ctypes.c_float)],
        "conv_bwd_data_selftest_wait_timeout": [vp, i64, P(i32)],
        "conv_bwd_data_run_noalloc": [P(Desc), vp, vp, vp, vp, P(i32)],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.conv_bwd_status_string.argtypes = [ctypes.c_int]
    lib.conv_bwd_status_string.restype = ctypes.c_char_p
    lib.conv_bwd_data_version.argtypes = []
    lib.conv_bwd_data_version.restype = ctypes.c_int32
    return lib


_lib = _load()


def lib():
    return _lib


def status_string(s: int) -> str:
    return _lib.conv_bwd_status_string(int(s)).decode()


def _check(status: int, what: str):
    if status != OK:
        raise ConvBwdError(status, what)


def _stream_handle(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


class Plan:
    """A planned convolution backward-data problem (wraps conv_bwd_plan)."""

    def __init__(self, N, C, K, Hi, Wi, Y, X, pad=(0, 0), stride=(1, 1), dil=(1, 1), groups=1,
                 layout="nchw", dtype="f32"):
        lay = {"nchw": NCHW_GKCYX, "nhwc": NHWC_KYXC}[layout] if isinstance(layout, str) else int(layout)
        dt = {"f32": F32, "bf16": BF16}[dtype] if isinstance(dtype, str) else int(dtype)
        self.desc = Desc(N, C, K, Hi, Wi, Y, X, pad[0], pad[1], stride[0], stride[1], dil[0], dil[1], groups, lay, dt)
        h = ctypes.c_void_p()
        _check(_lib.conv_bwd_data_create(ctypes.byref(self.desc), ctypes.byref(h)), "conv_bwd_data_create")
        self._h = h
        ho, wo = ctypes.c_int64(), ctypes.c_int64()
        _check(_lib.conv_bwd_data_out_dims(h, ctypes.byref(ho), ctypes.byref(wo)), "conv_bwd_data_out_dims")
        self.Ho, self.Wo = ho.value, wo.value
        self.layout, self.dtype = lay, dt

    @classmethod
    def from_case(cls, c):
        return cls(c.N, c.C, c.K, c.Hi, c.Wi, c.Y, c.X, c.pad, c.stride, c.dil, c.groups, c.layout, c.dtype)

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib.conv_bwd_data_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- queries ----------------------------------------------------------
    def shapes(self):
        d = self.desc
        Cg = d.C // d.groups
        if self.layout == NCHW_GKCYX:
            return (d.N, d.K, self.Ho, self.Wo), (d.K, Cg, d.Y, d.X), (d.N, d.C, d.Hi, d.Wi)
        return (d.N, self.Ho, self.Wo, d.K), (d.K, d.Y, d.X, Cg), (d.N, d.Hi, d.Wi, d.C)

    def num_subgemms(self) -> int:
        n = ctypes.c_int32()
        _check(_lib.conv_bwd_data_num_subgemms(self._h, ctypes.byref(n)), "num_subgemms")
        return n.value

    def subgemm(self, i: int) -> dict:
        ty, tx, ta, tb = (ctypes.c_int32() for _ in range(4))
        M, N, K = (ctypes.c_int64() for _ in range(3))
        _check(_lib.conv_bwd_data_subgemm_info(self._h, i, ctypes.byref(ty), ctypes.byref(tx), ctypes.byref(M),
                                               ctypes.byref(N), ctypes.byref(K), ctypes.byref(ta), ctypes.byref(tb)),
               "subgemm_info")
        return dict(ty=ty.value, tx=tx.value, M=M.value, N=N.value, K=K.value, taps_y=ta.value, taps_x=tb.value)

    def coverage(self):
        import numpy as np
        rows = np.zeros(self.desc.Hi, dtype=np.uint8)
        cols = np.zeros(self.desc.Wi, dtype=np.uint8)
        _check(_lib.conv_bwd_data_coverage(self._h, rows.ctypes.data, cols.ctypes.data), "coverage")
        return rows.astype(bool), cols.astype(bool)

    def path(self):
        p, n = ctypes.c_int32(), ctypes.c_int32()
        _check(_lib.conv_bwd_data_path(self._h, ctypes.byref(p), ctypes.byref(n)), "path")
        return PATH_NAMES.get(p.value, str(p.value)), n.value

    def tile(self):
        """(rows, columns, SMs) of one output tile of the GEMM kernel."""
        m, n, k = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check(_lib.conv_bwd_data_tile(self._h, ctypes.byref(m), ctypes.byref(n), ctypes.byref(k)), "tile")
        return m.value, n.value, k.value

    def a_operand(self) -> str:
        """How the GEMM kernel loads dy: "im2col", "plain" (2-D tiles of dy as a
        matrix; the specialised kernel), "gather" or "band" (tiled loads of a
        band of dy rows read by every tap)."""
        m = ctypes.c_int32()
        _check(_lib.conv_bwd_data_a_operand(self._h, ctypes.byref(m)), "a_operand")
        return {0: "im2col", 1: "plain", 2: "gather", 3: "band"}[m.value]

    def grouped_kernel(self) -> str:
        """Narrow-group kernel of the plan: "band", "mma", "tc" or "" (another path)."""
        m = ctypes.c_int32()
        _check(_lib.conv_bwd_data_grouped_kernel(self._h, ctypes.byref(m)), "grouped_kernel")
        return {0: "", 1: "mma", 2: "tc", 3: "band"}[m.value]

    def k_splits(self) -> int:
        """SM pairs that share each tile of the split-K schedule (1: whole tiles)."""
        m = ctypes.c_int32()
        _check(_lib.conv_bwd_data_k_splits(self._h, ctypes.byref(m)), "k_splits")
        return m.value

    def work(self):
        f, b = ctypes.c_double(), ctypes.c_double()
        _check(_lib.conv_bwd_data_work(self._h, ctypes.byref(f), ctypes.byref(b)), "work")
        return f.value, b.value

    # ---- execution --------------------------------------------------------
    def run(self, dy, w, dx, stream=None):
        """dx <- dgrad(dy, w) on ``stream`` (torch CUDA tensors, plan layout/dtype)."""
        _check(_lib.conv_bwd_data_run(self._h, ctypes.c_void_p(dy.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                      ctypes.c_void_p(dx.data_ptr()), _stream_handle(stream)), "conv_bwd_data_run")

    def run_ptr(self, dy_ptr: int, w_ptr: int, dx_ptr: int, stream_handle: int = 0) -> int:
        """Raw-pointer form; returns the status code instead of raising."""
        return _lib.conv_bwd_data_run(self._h, ctypes.c_void_p(dy_ptr), ctypes.c_void_p(w_ptr),
                                      ctypes.c_void_p(dx_ptr), ctypes.c_void_p(stream_handle))

    def run_forward(self, x, w, y, stream=None):
        """y <- conv(x, w), the forward convolution of the plan's geometry (x has
        dx's shape, y has dy's shape; bf16 NHWC plans)."""
        _check(_lib.conv_bwd_data_run_forward(self._h, ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                              ctypes.c_void_p(y.data_ptr()), _stream_handle(stream)),
               "conv_bwd_data_run_forward")

    def run_forward_ptr(self, x_ptr: int, w_ptr: int, y_ptr: int, stream_handle: int = 0) -> int:
        """Raw-pointer form of run_forward; returns the status code."""
        return _lib.conv_bwd_data_run_forward(self._h, ctypes.c_void_p(x_ptr), ctypes.c_void_p(w_ptr),
                                              ctypes.c_void_p(y_ptr), ctypes.c_void_p(stream_handle))

    def run_host(self, dy_h, w_h, dx_h, dy_d, w_d, dx_d, stream=None):
        """Host buffers in, host buffer out (copies ordered on the stream)."""
        _check(_lib.conv_bwd_data_run_host(self._h, ctypes.c_void_p(dy_h.data_ptr()), ctypes.c_void_p(w_h.data_ptr()),
                                           ctypes.c_void_p(dx_h.data_ptr()), ctypes.c_void_p(dy_d.data_ptr()),
                                           ctypes.c_void_p(w_d.data_ptr()), ctypes.c_void_p(dx_d.data_ptr()),
                                           _stream_handle(stream)), "conv_bwd_data_run_host")

    def status(self, stream=None):
        det = ctypes.c_int32()
        s = _lib.conv_bwd_data_get_status(self._h, _stream_handle(stream), ctypes.byref(det))
        return s, det.value

    def set_timing(self, on: bool):
        _check(_lib.conv_bwd_data_set_timing(self._h, 1 if on else 0), "set_timing")

    def last_timing(self):
        f, g = ctypes.c_float(), ctypes.c_float()
        _check(_lib.conv_bwd_data_last_timing(self._h, ctypes.byref(f), ctypes.byref(g)), "last_timing")
        return f.value, g.value


def run_noalloc(desc: Desc, dy, w, dx, stream=None, sync: bool = False):
    """conv_bwd_data_run_noalloc: tensor-core dgrad without any device
    allocation (status word in the library's static device scratch).
    Returns (status, device_status)."""
    det = ctypes.c_int32(0)
    st = _lib.conv_bwd_data_run_noalloc(ctypes.byref(desc), ctypes.c_void_p(dy.data_ptr()),
                                        ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(dx.data_ptr()),
                                        _stream_handle(stream), ctypes.byref(det) if sync else None)
    return st, det.value


def selftest_wait_timeout(budget_cycles: int, stream=None) -> int:
    obs = ctypes.c_int32(-1)
    _check(_lib.conv_bwd_data_selftest_wait_timeout(_stream_handle(stream), int(budget_cycles), ctypes.byref(obs)),
           "selftest_wait_timeout")
    return obs.value


def dgrad(dy, w, Hi, Wi, pad=(0, 0), stride=(1, 1), dil=(1, 1), groups=1, layout="nchw", out=None, stream=None):
    """Convenience: dx = dgrad(dy, w) for torch CUDA tensors (fp32 or bf16)."""
    import torch
    dtype = {torch.float32: "f32", torch.bfloat16: "bf16"}[dy.dtype]
    if layout == "nchw":
        N, K = dy.shape[0], dy.shape[1]
        Kw, Cg, Y, X = w.shape
    else:
        N, K = dy.shape[0], dy.shape[3]
        Kw, Y, X, Cg = w.shape
    plan = Plan(N, Cg * groups, K, Hi, Wi, Y, X, pad, stride, dil, groups, layout, dtype)
    dy_s, w_s, dx_s = plan.shapes()
    if tuple(dy.shape) != dy_s or tuple(w.shape) != w_s:
        raise ValueError(f"shape mismatch: dy {tuple(dy.shape)} vs {dy_s}, w {tuple(w.shape)} vs {w_s}")
    if out is None:
        out = torch.empty(dx_s, dtype=dy.dtype, device=dy.device)
    plan.run(dy.contiguous(), w.contiguous(), out, stream)
    return out
