"""GPU parity of the save-for-backward split of the 3D projection gradients.

tp_project_3d_2d_save writes the forward output and D_a = phase * dS/dp_a
per pixel; tp_project_3d_2d_backward_saved turns (grad_out, out, D) into the
rotation and shift gradients.  Both are held to the float64 oracle at the
same tolerances as the recomputing backward pass, and D itself is pinned
through the oracle's rotation gradient of single-pixel upstream gradients.
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


# (interp, M, N, s, shifted, radius, Bv, Bp, P): ragged boxes, oversampling,
# radii (including 0: only the DC pixel) and broadcast batches.
CASES = []
for interp in ("linear", "cubic"):
    CASES += [
        (interp, 16, 16, 1.0, True, -1.0, 1, 1, 3),
        (interp, 18, 14, 1.3, True, 5.5, 2, 1, 2),
        (interp, 32, 16, 2.0, False, 100.0, 2, 2, 3),
        (interp, 12, 16, 0.75, True, -1.0, 1, 2, 2),
        (interp, 20, 10, 2.0, True, 0.0, 2, 2, 2),
    ]


def _inputs(M, N, shifted, Bv, Bp, P, seed):
    rng = np.random.default_rng(seed)
    vol = crandn(rng, (Bv, M, M, M // 2 + 1))
    R = synth.random_rotations(Bp * P, rng).reshape(Bp, P, 3, 3)
    B = max(Bv, Bp)
    t = rng.uniform(-6, 6, (B, P, 2)).astype(np.float32) if shifted else None
    g = crandn(rng, (B, P, N, N // 2 + 1))
    return vol, R, t, g


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_saved_forward_and_pose_gradients(tp, case):
    interp, M, N, s, shifted, radius, Bv, Bp, P = case
    vol, R, t, g = _inputs(M, N, shifted, Bv, Bp, P, seed=3000 + CASES.index(case))
    kw = dict(interp=interp, oversampling=s, radius=radius)
    dv, dR, dt = dev(vol), dev(R), dev(t)
    out, dout = tp.tp_project_3d_2d_save(dv, dR, dt, N=N, **kw)
    ref = oracle.project(3, vol, R, shift=t, N=N, **kw)
    assert rel(host(out), ref) <= FWD_TOL
    plain = host(tp.tp_project_3d_2d(dv, dR, dt, N=N, **kw))
    assert rel(host(out), plain) <= 1e-6
    gr, gt = tp.tp_project_3d_2d_backward_saved(dev(g), out, dout, dR, dt, **kw)
    _, rr, rt = oracle.project_backward(3, g, vol, R, shift=t, need_src=False, **kw)
    assert rel(host(gr), rr) <= ATOMIC_TOL
    if shifted:
        assert rel(host(gt), rt) <= ATOMIC_TOL
    else:
        assert gt is None


def test_saved_derivatives_pinned_by_single_pixel_gradients(tp):
    """With g = c * delta at pixel (kx, ky), the oracle's dL/dR[0][a] equals
    s * kx * Re(conj(c) D_a): c = 1 and c = i read off Re D_a and Im D_a."""
    rng = np.random.default_rng(77)
    M = N = 16
    s = 1.0
    vol = crandn(rng, (1, M, M, M // 2 + 1))
    R = synth.random_rotations(1, rng).reshape(1, 1, 3, 3)
    t = rng.uniform(-3, 3, (1, 1, 2)).astype(np.float32)
    kw = dict(interp="cubic", oversampling=s, radius=-1.0)
    _, dout = tp.tp_project_3d_2d_save(dev(vol), dev(R), dev(t), **kw)
    D = host(dout)
    for (iy, kx) in [(3, 2), (13, 5), (1, 7), (9, 1)]:
        got = D[0, 0, iy, kx]
        want = np.zeros(3, np.complex128)
        for c in (1.0, 1j):
            g = np.zeros((1, 1, N, N // 2 + 1), np.complex64)
            g[0, 0, iy, kx] = c
            _, rr, _ = oracle.project_backward(3, g, vol, R, shift=t, need_src=False,
                                               need_shift=False, **kw)
            part = rr[0, 0, 0, :] / (s * kx)       # Re(conj(c) D_a)
            want += part if c == 1.0 else 1j * part
        assert rel(got, want) <= 1e-5, (iy, kx)


def test_saved_derivatives_vanish_outside_radius(tp):
    rng = np.random.default_rng(5)
    M = N = 24
    vol = crandn(rng, (1, M, M, M // 2 + 1))
    R = synth.random_rotations(4, rng).reshape(1, 4, 3, 3)
    out, dout = tp.tp_project_3d_2d_save(dev(vol), dev(R), None, radius=7.0, interp="cubic")
    ky = np.fft.fftfreq(N, 1.0 / N)[:, None]
    kx = np.arange(N // 2 + 1)[None, :]
    outside = kx * kx + ky * ky > 49
    assert np.all(host(out)[:, :, outside] == 0)
    assert np.all(host(dout)[:, :, outside] == 0)
    assert np.any(host(dout)[:, :, ~outside] != 0)


def test_saved_empty_pose_list(tp):
    vol = torch.zeros((1, 8, 8, 5), dtype=torch.complex64, device="cuda")
    rot = torch.zeros((1, 0, 3, 3), device="cuda")
    out, dout = tp.tp_project_3d_2d_save(vol, rot)
    assert out.shape == (1, 0, 8, 5) and dout.shape == (1, 0, 8, 5, 3)
    gr, gt = tp.tp_project_3d_2d_backward_saved(out, out, dout, rot)
    assert gr.shape == rot.shape and gt is None


def test_cfg5_box256_saved_step_sampled(tp):
    """The benchmark's launch: the box-256 cubic forward with saved
    derivatives for all 512 poses, then the saved-path gradients; sampled
    poses against the oracle."""
    w = synth.workload(5)
    kw = dict(interp=w["interp"], oversampling=1.0, radius=w["radius"])
    vol, R, t, g = w["vol"], w["rot"], w["shift"], w["grad"]
    dv, dR, dt = dev(vol), dev(R), dev(t)
    out, dout = tp.tp_project_3d_2d_save(dv, dR, dt, **kw)
    pick = np.arange(5, 512, 64)
    ref = oracle.project(3, vol, R[:, pick], shift=t[:, pick], **kw)
    assert rel(host(out)[:, pick], ref) <= FWD_TOL
    gr, gt = tp.tp_project_3d_2d_backward_saved(dev(g), out, dout, dR, dt, **kw)
    _, rr, rt = oracle.project_backward(3, g[:, pick], vol, R[:, pick], shift=t[:, pick],
                                        need_src=False, **kw)
    assert rel(host(gr)[:, pick], rr) <= ATOMIC_TOL
    assert rel(host(gt)[:, pick], rt) <= ATOMIC_TOL
