"""The no-allocation entry point (conv_bwd_data_run_noalloc) against the
oracle and against the regular entry point (conv_bwd_data_run).

Callers such as plugin hosts with their own device-memory pool, or loops that
must not call cudaMalloc, use the no-allocation call: its kernel keeps its
status word in a static device array instead of a buffer from
conv_bwd_data_create.  Two calls in a row must each match the oracle's dx
within the bf16 bound, and the regular entry point's dx within that bound too
(the array keeps the previous call's contents, so the second call checks that
the status word is cleared again).  The cases cover the 1-SM tensor-core
kernel and the SM-pair kernel (C/G >= 256, held on pairs by the override).  This file is
collected last on purpose and must pass alone in a fresh process too.
"""
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


CASES = [
    wl.Case(name="noalloc_3x3s2", N=3, C=192, K=136, Hi=13, Wi=11, Y=3, X=3, pad=(1, 1), stride=(2, 2),
            dtype=wl.BF16, layout=wl.NHWC, dist="normal", sigma=0.5, seed=901),
    wl.Case(name="noalloc_fill", N=2, C=128, K=64, Hi=15, Wi=14, Y=3, X=3, pad=(1, 1), stride=(4, 4),
            dtype=wl.BF16, layout=wl.NHWC, dist="normal", sigma=0.5, seed=902),
    # C/G >= 256: 256-row tiles on SM pairs (CONVBWD_DEBUG_2SM=1 in the test)
    wl.Case(name="noalloc_pair", N=2, C=256, K=256, Hi=9, Wi=10, Y=3, X=3, pad=(1, 1), stride=(2, 2),
            dtype=wl.BF16, layout=wl.NHWC, dist="normal", sigma=0.5, seed=903),
]


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("c", CASES, ids=lambda c: c.name)
def test_noalloc_matches_oracle_and_regular_entry_point_twice(B, monkeypatch, c):
    if c.name == "noalloc_pair":
        # a layer this small fits one round of 1-SM tiles, which the planner
        # prefers; the override keeps it on SM pairs
        monkeypatch.setenv("CONVBWD_DEBUG_2SM", "1")
    g = oracle.geom(c.N, c.C, c.K, c.Hi, c.Wi, c.Y, c.X, c.pad, c.stride, c.dil, c.groups)
    dy_s, w_s, dx_s = oracle.shapes(g, oracle.LAYOUT_NHWC)
    dy, w = wl.draw(c, dy_s, w_s)
    dyd, wd = _dev(dy), _dev(w)
    ref_o, absdot = oracle.dgrad(g, oracle.LAYOUT_NHWC, dy, w)
    bound = oracle.tolerance(ref_o, absdot, "bf16")
    plan = B.Plan.from_case(c)
    assert plan.path()[0] == "tcgen05"
    want_sms = 2 if c.name == "noalloc_pair" else 1
    assert plan.tile()[2] == want_sms, plan.tile()
    reg = torch.full(dx_s, float("nan"), dtype=torch.bfloat16, device="cuda")
    plan.run(dyd, wd, reg)
    assert plan.status() == (B.OK, 0)
    reg = reg.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(reg - ref_o) <= bound)
    for call in range(2):
        out = torch.full(dx_s, float("nan"), dtype=torch.bfloat16, device="cuda")
        st, det = B.run_noalloc(plan.desc, dyd, wd, out, sync=True)
        assert st == B.OK and det == 0, (call, B.status_string(st), det)
        got = out.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), call
        assert np.all(np.abs(got - ref_o) <= bound), call
        assert np.all(np.abs(got - reg) <= bound), call


def test_noalloc_rejects_other_paths(B):
    d = B.Plan(1, 16, 16, 8, 8, 3, 3, (1, 1)).desc  # fp32 NCHW: CUDA-core path, no variant
    x = torch.zeros(16 * 64, device="cuda")
    st, _ = B.run_noalloc(d, x, x[:16 * 9 * 16], torch.zeros(16 * 64, device="cuda"), sync=True)
    assert st == B.ERR_UNSUPPORTED
