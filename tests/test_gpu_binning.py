"""GPU: the binning kept in a caller's workspace between 3D calls.

A call keeps the brick masks and work units already in its workspace only
when the poses and sizes are bit-identical to the ones they were made for;
every case here reuses one workspace across calls whose poses or sizes
differ, or stay the same, and checks the results against the float64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

FWD_TOL = 1e-5
ATOMIC_TOL = 1e-4


@pytest.fixture(scope="module")
def tp():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import backprojection_tp_project_gather_b300 as m
    return m


def rel(a, b):
    a = np.asarray(a, np.complex128)
    b = np.asarray(b, np.complex128)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def dev(x):
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def crandn(rng, shape):
    return (rng.standard_normal(shape) + 1j * rng.standard_normal(shape)).astype(np.complex64)


M = N = 24
P = 5


def _problem(seed):
    rng = np.random.default_rng(seed)
    vol = crandn(rng, (1, M, M, M // 2 + 1))
    R = synth.random_rotations(P, rng).reshape(1, P, 3, 3)
    t = rng.uniform(-3, 3, (1, P, 2)).astype(np.float32)
    g = crandn(rng, (1, P, N, N // 2 + 1))
    return vol, R, t, g


@pytest.fixture()
def ws(tp):
    # Large enough for every call below; filled with garbage first.
    n = 4 * tp.tp_workspace_bytes(1, 1, P, M, "cubic")
    return torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda")


CUBIC = dict(interp="cubic")


def _fwd(tp, vol, R, t, ws, **kw):
    kw = {**CUBIC, **kw}
    return host(tp.tp_project_3d_2d(dev(vol), dev(R), dev(t), workspace=ws, **kw))


@pytest.mark.parametrize("interp", ["linear", "cubic"])
def test_forward_then_backward_on_the_same_poses(tp, ws, interp):
    vol, R, t, g = _problem(1)
    kw = dict(interp=interp)
    out = _fwd(tp, vol, R, t, ws, **kw)
    assert rel(out, oracle.project(3, vol, R, shift=t, **kw)) <= FWD_TOL
    gv, gr, gt = tp.tp_project_3d_2d_backward(dev(g), dev(vol), dev(R), dev(t), workspace=ws, **kw)
    rv, rr, rt = oracle.project_backward(3, g, vol, R, shift=t, **kw)
    assert rel(host(gv), rv) <= ATOMIC_TOL
    assert rel(host(gr), rr) <= ATOMIC_TOL
    assert rel(host(gt), rt) <= ATOMIC_TOL


def test_other_poses_in_the_same_workspace(tp, ws):
    vol, R, t, _ = _problem(2)
    _, R2, t2, _ = _problem(3)
    _fwd(tp, vol, R, t, ws)
    out = _fwd(tp, vol, R2, t2, ws)
    assert rel(out, oracle.project(3, vol, R2, shift=t2, **CUBIC)) <= FWD_TOL


def test_rotations_changed_in_place(tp, ws):
    vol, R, t, _ = _problem(4)
    dR, dt, dv = dev(R), dev(t), dev(vol)
    tp.tp_project_3d_2d(dv, dR, dt, workspace=ws, **CUBIC)
    dR[0, 2] = dR[0, 2] @ torch.tensor([[0.0, -1.0, 0.0], [1.0, 0.0, 0.0], [0.0, 0.0, 1.0]],
                                       device="cuda")
    out = host(tp.tp_project_3d_2d(dv, dR, dt, workspace=ws, **CUBIC))
    assert rel(out, oracle.project(3, vol, host(dR), shift=t, **CUBIC)) <= FWD_TOL


def test_radius_and_box_changes(tp, ws):
    vol, R, t, _ = _problem(5)
    _fwd(tp, vol, R, t, ws)
    out = _fwd(tp, vol, R, t, ws, radius=6.5)
    assert rel(out, oracle.project(3, vol, R, shift=t, radius=6.5, **CUBIC)) <= FWD_TOL
    out = _fwd(tp, vol, R, t, ws, N=16, oversampling=1.5)
    ref = oracle.project(3, vol, R, shift=t, N=16, oversampling=1.5, **CUBIC)
    assert rel(out, ref) <= FWD_TOL


def test_alternating_pose_sets_many_calls(tp, ws):
    vol, R, t, g = _problem(6)
    _, R2, t2, _ = _problem(7)
    dv = dev(vol)
    for i in range(6):
        Ri, ti = (R, t) if i % 2 == 0 else (R2, t2)
        out = host(tp.tp_project_3d_2d(dv, dev(Ri), dev(ti), workspace=ws, **CUBIC))
        gv, _, _ = tp.tp_project_3d_2d_backward(dev(g), dv, dev(Ri), dev(ti), workspace=ws,
                                                want_rot=False, want_shift=False, **CUBIC)
    assert rel(out, oracle.project(3, vol, R2, shift=t2, **CUBIC)) <= FWD_TOL
    rv, _, _ = oracle.project_backward(3, g, vol, R2, shift=t2, need_rot=False, need_shift=False,
                                       **CUBIC)
    assert rel(host(gv), rv) <= ATOMIC_TOL


def _bp(tp, proj, R, t, om, ws, **kw):
    kw = {**CUBIC, **kw}
    d, w = tp.tp_backproject_2d_3d(dev(proj), dev(R), dev(t), dev(om), Nv=M, workspace=ws, **kw)
    return host(d), host(w)


def test_scatter_sample_lists_kept_and_rebuilt(tp, ws):
    # The cubic scatters sort the output pixels into lists kept in the
    # workspace with the binning: reused for the same poses, rebuilt after a
    # call on other poses, after poses changed in place and for another image
    # box; a kept list must never serve other poses.
    rng = np.random.default_rng(8)
    _, R, t, proj = _problem(8)
    _, R2, t2, _ = _problem(9)
    om = rng.uniform(0.5, 1.5, proj.shape).astype(np.float32)
    ref = oracle.backproject(3, proj, R, shift=t, M=M, weights=om, **CUBIC)
    for _ in range(2):   # built, then kept
        d, w = _bp(tp, proj, R, t, om, ws)
        assert rel(d, ref[0]) <= ATOMIC_TOL and rel(w, ref[1]) <= ATOMIC_TOL
    vol = crandn(rng, (1, M, M, M // 2 + 1))
    _fwd(tp, vol, R2, t2, ws)   # other poses: the binning and the lists change
    d, w = _bp(tp, proj, R, t, om, ws)
    assert rel(d, ref[0]) <= ATOMIC_TOL and rel(w, ref[1]) <= ATOMIC_TOL
    # One rotation changed in place between two calls.
    dR, dt, dp, dom = dev(R), dev(t), dev(proj), dev(om)
    tp.tp_backproject_2d_3d(dp, dR, dt, dom, Nv=M, workspace=ws, **CUBIC)
    dR[0, 1] = dR[0, 1] @ torch.tensor([[0.0, 0.0, 1.0], [0.0, 1.0, 0.0], [-1.0, 0.0, 0.0]],
                                       device="cuda")
    d, w = tp.tp_backproject_2d_3d(dp, dR, dt, dom, Nv=M, workspace=ws, **CUBIC)
    ref2 = oracle.backproject(3, proj, host(dR), shift=t, M=M, weights=om, **CUBIC)
    assert rel(host(d), ref2[0]) <= ATOMIC_TOL and rel(host(w), ref2[1]) <= ATOMIC_TOL
    # Volume gradient of a smaller image box on the same workspace, then the
    # original box again.
    g16 = crandn(rng, (1, P, 16, 9))
    gv, _, _ = tp.tp_project_3d_2d_backward(dev(g16), dev(vol), dev(R), dev(t), workspace=ws,
                                            want_rot=False, want_shift=False, **CUBIC)
    rv, _, _ = oracle.project_backward(3, g16, vol, R, shift=t, need_rot=False,
                                       need_shift=False, **CUBIC)
    assert rel(host(gv), rv) <= ATOMIC_TOL
    d, w = _bp(tp, proj, R, t, om, ws)
    assert rel(d, ref[0]) <= ATOMIC_TOL and rel(w, ref[1]) <= ATOMIC_TOL


def test_scatter_sample_lists_in_a_workspace_of_random_bytes(tp):
    # Random contents, including the list flags: the key cannot match, so the
    # binning and the lists are rebuilt.
    _, R, t, proj = _problem(10)
    om = np.ones(proj.shape, np.float32)
    ref = oracle.backproject(3, proj, R, shift=t, M=M, weights=om, **CUBIC)
    for seed in range(3):
        gen = torch.Generator(device="cuda").manual_seed(seed)
        n = tp.tp_workspace_bytes(1, 1, P, M, "cubic")
        ws = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda", generator=gen)
        d, w = _bp(tp, proj, R, t, om, ws)
        assert rel(d, ref[0]) <= ATOMIC_TOL and rel(w, ref[1]) <= ATOMIC_TOL
