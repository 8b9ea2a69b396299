"""GPU parity of the symmetrised zero-frequency axis (TP_FLAG_HERMITIAN_X0
and tp_hermitian_x0) against the float64 oracle's hermitian_x0 composed
with its backprojection and backward operators."""
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


@pytest.mark.parametrize("dim,M,B", [(3, 2, 1), (3, 16, 2), (3, 34, 1), (2, 2, 3), (2, 30, 2)])
def test_standalone_matches_oracle(tp, dim, M, B):
    rng = np.random.default_rng(300 + M)
    shape = (B,) + (M,) * (dim - 1) + (M // 2 + 1,)
    V = crandn(rng, shape)
    W = rng.standard_normal(shape).astype(np.float32)
    rv, rw = oracle.hermitian_x0(V, dim, W)
    dv, dw = dev(V), dev(W)
    tp.tp_hermitian_x0(dv, dw, dim=dim)
    assert rel(host(dv), rv) <= 1e-6
    assert np.abs(host(dw) - rw).max() <= 1e-6 * np.abs(rw).max()
    assert np.array_equal(host(dv)[..., 1:], V[..., 1:])     # other planes untouched
    # weight only, and spec only
    dw2 = dev(W)
    tp.tp_hermitian_x0(None, dw2, dim=dim)
    assert np.array_equal(host(dw2), host(dw))
    dv2 = dev(V)
    tp.tp_hermitian_x0(dv2, None, dim=dim)
    assert np.array_equal(host(dv2), host(dv))


@pytest.mark.parametrize("interp", ["linear", "cubic"])
@pytest.mark.parametrize("Bv", [1, 2])
def test_backprojection_flag(tp, interp, Bv):
    rng = np.random.default_rng(310 + Bv)
    B, P, N, M = 2, 5, 18, 20
    proj = crandn(rng, (B, P, N, N // 2 + 1))
    om = rng.uniform(0.5, 1.5, proj.shape).astype(np.float32)
    R = synth.random_rotations(B * P, rng).reshape(B, P, 3, 3)
    t = rng.uniform(-3, 3, (B, P, 2)).astype(np.float32)
    kw = dict(interp=interp, oversampling=1.1, radius=8.5)
    d, w = tp.tp_backproject_2d_3d(dev(proj), dev(R), dev(t), dev(om), Nv=M, Bv=Bv,
                                   hermitian_x0=True, **kw)
    rd, rw = oracle.backproject(3, proj, R, shift=t, M=M, weights=om, Bdst=Bv, **kw)
    rd, rw = oracle.hermitian_x0(rd, 3, rw)
    assert rel(host(d), rd) <= ATOMIC_TOL
    assert rel(host(w), rw) <= ATOMIC_TOL


def test_volume_gradient_flag_3d(tp):
    rng = np.random.default_rng(320)
    M = N = 16
    vol = crandn(rng, (1, M, M, M // 2 + 1))
    R = synth.random_rotations(4, rng).reshape(1, 4, 3, 3)
    t = rng.uniform(-3, 3, (1, 4, 2)).astype(np.float32)
    g = crandn(rng, (1, 4, N, N // 2 + 1))
    kw = dict(interp="cubic", oversampling=1.0, radius=-1.0)
    gv, gr, gs = tp.tp_project_3d_2d_backward(dev(g), dev(vol), dev(R), dev(t),
                                              hermitian_x0=True, **kw)
    rv, rr, rs = oracle.project_backward(3, g, vol, R, shift=t, **kw)
    assert rel(host(gv), oracle.hermitian_x0(rv, 3)[0]) <= ATOMIC_TOL
    assert rel(host(gr), rr) <= ATOMIC_TOL          # pose gradients are not affected
    assert rel(host(gs), rs) <= ATOMIC_TOL


def test_image_gradient_flag_2d(tp):
    rng = np.random.default_rng(330)
    M = N = 20
    img = crandn(rng, (2, M, M // 2 + 1))
    R = synth.planar_rotations(rng.uniform(0, 2 * np.pi, 6)).reshape(2, 3, 2, 2)
    g = crandn(rng, (2, 3, N, N // 2 + 1))
    kw = dict(interp="linear", oversampling=1.0, radius=-1.0)
    gi, gr, _ = tp.tp_project_2d_2d_backward(dev(g), dev(img), dev(R), hermitian_x0=True, **kw)
    ri, rr, _ = oracle.project_backward(2, g, img, R, **kw)
    assert rel(host(gi), oracle.hermitian_x0(ri, 2)[0]) <= ATOMIC_TOL
    assert rel(host(gr), rr) <= ATOMIC_TOL


def test_real_object_adjoint_identity_at_box128(tp):
    """Re<F V, y> = Re<V, H(B y)> for the spectrum V of a real volume, at the
    box-128 size of the forward workload (1024 poses), on the GPU alone."""
    rng = np.random.default_rng(340)
    M = N = 128
    P = 1024
    x = torch.from_numpy(rng.standard_normal((M, M, M)).astype(np.float32)).cuda()
    V = torch.fft.rfftn(x).unsqueeze(0).contiguous()
    R = dev(synth.random_rotations(P, rng)[None])
    y = dev(crandn(rng, (1, P, N, N // 2 + 1)))
    kw = dict(interp="cubic", oversampling=1.0, radius=60.0)
    lhs = torch.vdot(y.flatten(), tp.tp_project_3d_2d(V, R, **kw).flatten()).real.item()
    d, _ = tp.tp_backproject_2d_3d(y, R, Nv=M, want_weights=False, hermitian_x0=True, **kw)
    rhs = torch.vdot(d.flatten(), V.flatten()).real.item()
    assert abs(lhs - rhs) <= 1e-4 * abs(lhs)


def test_autograd_flag(tp):
    import backprojection_tp_project_gather_b300.autograd as ag
    rng = np.random.default_rng(350)
    M = N = 16
    vol = crandn(rng, (1, M, M, M // 2 + 1))
    R = synth.random_rotations(3, rng).reshape(1, 3, 3, 3)
    g = crandn(rng, (1, 3, N, N // 2 + 1))
    v = dev(vol).requires_grad_(True)
    y = ag.project_3d_2d(v, dev(R), interp="cubic", hermitian_x0=True)
    (y * dev(np.conj(g))).real.sum().backward()          # upstream gradient g
    rv, _, _ = oracle.project_backward(3, g, vol, R, interp="cubic", need_rot=False)
    assert rel(v.grad.cpu().numpy(), oracle.hermitian_x0(rv, 3)[0]) <= ATOMIC_TOL
