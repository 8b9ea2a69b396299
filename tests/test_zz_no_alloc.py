"""The allocation-free forward projection, tp_project_3d_2d_noalloc.

Some callers cannot allocate device memory where they call the library (for
example during a CUDA-graph capture, or under an allocator of their own), so
they cannot hand tp_project_3d_2d the scratch workspace it needs.  The
no-allocation entry point keeps that scratch in a fixed array inside the
library.  These checks call it through the C ABI and compare it with the
regular entry point on the same inputs, on consecutive calls of different
sizes (the shared array keeps the previous call's contents), and check that
a problem too large for the array is refused.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

FWD_TOL = 1e-5


@pytest.fixture(scope="module")
def tp():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import backprojection_tp_project_gather_b300 as m
    return m


def dev(x):
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda()


def rel(a, b):
    a = torch.view_as_real(a).double().cpu().numpy()
    b = torch.view_as_real(b).double().cpu().numpy()
    return np.linalg.norm(a - b) / np.linalg.norm(b)


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(tp):
    cases = []
    w1 = synth.workload(1)
    t1 = synth.uniform_shifts(w1["P"], 3.0, synth.streams(11, 1)[0])[None]
    cases.append((w1["vol"], w1["rot"], t1, dict(interp="cubic", radius=w1["radius"])))
    w3 = synth.workload(3, poses=96)
    cases.append((w3["vol"], w3["rot"], None, dict(interp="cubic", radius=w3["radius"])))
    cases.append(cases[0])                         # back to the first size
    for vol, R, t, kw in cases:
        v, r, s = dev(vol), dev(R), dev(t)
        ref = tp.tp_project_3d_2d(v, r, s, **kw)
        out = torch.full_like(ref, float("nan"))
        tp.tp_project_3d_2d_noalloc(v, r, s, out=out, **kw)
        torch.cuda.synchronize()
        assert torch.isfinite(torch.view_as_real(out)).all()
        assert rel(out, ref) <= FWD_TOL


def test_noalloc_refuses_problems_beyond_its_array(tp):
    # 200000 poses against a 256^3 volume need far more than the fixed array.
    # The array pointers are NULL: the size check refuses the call first, and
    # were it ever to let the call through, the NULL check behind it would
    # refuse it too (a different status), so nothing is launched either way.
    o = tp.TPOptions(1, 1.0, -1.0, 0)
    st = tp._fn("tp_project_3d_2d_noalloc")(None, 1, 256, None, 1, 200000, None, 1, 256, o, None,
                                             None)
    assert st == 2   # TP_ERR_SHAPE
    msg = tp.tp_last_error()
    assert "tp_project_3d_2d_noalloc" in msg and "bytes of scratch" in msg, msg
    assert tp.tp_workspace_bytes(1, 1, 200000, 256, "cubic") > 16 << 20
