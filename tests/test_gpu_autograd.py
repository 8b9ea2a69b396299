"""GPU: the torch.autograd wrappers give the oracle's gradients for an L2 loss."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

FWD_TOL = 1e-5
ATOMIC_TOL = 1e-4


@pytest.fixture(scope="module")
def ag():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import backprojection_tp_project_gather_b300.autograd as m
    return m


def rel(a, b):
    a = np.asarray(a, np.complex128)
    b = np.asarray(b, np.complex128)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def crandn(rng, shape):
    return (rng.standard_normal(shape) + 1j * rng.standard_normal(shape)).astype(np.complex64)


def leaf(x, grad=True):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda().requires_grad_(grad)


@pytest.mark.parametrize("interp", ["linear", "cubic"])
def test_l2_loss_3d(ag, interp):
    rng = np.random.default_rng(61)
    M, N, P = 20, 16, 3
    vol = crandn(rng, (1, M, M, M // 2 + 1))
    R = synth.random_rotations(2 * P, rng).reshape(2, P, 3, 3)
    t = rng.uniform(-3, 3, (2, P, 2)).astype(np.float32)
    target = crandn(rng, (2, P, N, N // 2 + 1))
    kw = dict(interp=interp, oversampling=1.2, radius=7.5)
    v, r, s = leaf(vol), leaf(R), leaf(t)
    y = ag.project_3d_2d(v, r, s, N=N, **kw)
    loss = (y - torch.from_numpy(target).cuda()).abs().pow(2).sum()
    loss.backward()
    ref = oracle.project(3, vol, R, shift=t, N=N, **kw)
    assert rel(y.detach().cpu().numpy(), ref) <= FWD_TOL
    gv, gr, gt = oracle.project_backward(3, 2 * (ref - target), vol, R, shift=t, **kw)
    assert rel(v.grad.cpu().numpy(), gv) <= ATOMIC_TOL
    assert rel(r.grad.cpu().numpy(), gr) <= ATOMIC_TOL
    assert rel(s.grad.cpu().numpy(), gt) <= ATOMIC_TOL


def test_volume_only_3d(ag):
    rng = np.random.default_rng(62)
    M = N = 16
    vol = crandn(rng, (1, M, M, M // 2 + 1))
    R = synth.random_rotations(4, rng).reshape(1, 4, 3, 3)
    g = crandn(rng, (1, 4, N, N // 2 + 1))
    v = leaf(vol)
    y = ag.project_3d_2d(v, leaf(R, grad=False), interp="cubic")
    (y * torch.from_numpy(np.conj(g)).cuda()).real.sum().backward()     # upstream gradient g
    gv, _, _ = oracle.project_backward(3, g, vol, R, interp="cubic", need_rot=False)
    assert rel(v.grad.cpu().numpy(), gv) <= ATOMIC_TOL


def test_l2_loss_2d(ag):
    rng = np.random.default_rng(63)
    M = N = 24
    img = crandn(rng, (3, M, M // 2 + 1))
    R = synth.planar_rotations(rng.uniform(0, 2 * np.pi, 3)).reshape(3, 1, 2, 2)
    t = rng.uniform(-4, 4, (3, 1, 2)).astype(np.float32)
    target = crandn(rng, (3, 1, N, N // 2 + 1))
    i_, r, s = leaf(img), leaf(R), leaf(t)
    y = ag.project_2d_2d(i_, r, s, interp="cubic")
    (y - torch.from_numpy(target).cuda()).abs().pow(2).sum().backward()
    ref = oracle.project(2, img, R, shift=t, interp="cubic")
    gi, gr, gt = oracle.project_backward(2, 2 * (ref - target), img, R, shift=t, interp="cubic")
    assert rel(i_.grad.cpu().numpy(), gi) <= ATOMIC_TOL
    assert rel(r.grad.cpu().numpy(), gr) <= ATOMIC_TOL
    assert rel(s.grad.cpu().numpy(), gt) <= ATOMIC_TOL
