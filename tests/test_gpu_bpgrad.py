"""GPU parity of tp_backproject_2d_3d_backward (gradients of the 3D
backprojection) against the float64 oracle's backproject_backward, which
the CPU tests pin with finite differences of the backprojection itself."""
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


# (interp, M, N, s, radius, shifted, B, Bv, Bp, P, image weights, weight-spectrum gradient)
CASES = []
for interp in ("linear", "cubic"):
    CASES += [
        (interp, 16, 16, 1.0, -1.0, True, 1, 1, 1, 3, False, False),
        (interp, 20, 14, 1.3, 5.5, True, 2, 1, 1, 2, True, True),
        (interp, 24, 12, 2.0, -1.0, False, 2, 2, 2, 3, False, True),
        (interp, 18, 18, 0.8, 100.0, True, 2, 2, 1, 2, True, False),
    ]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_backprojection_gradients(tp, case):
    interp, M, N, s, radius, shifted, B, Bv, Bp, P, with_w, with_gw = case
    rng = np.random.default_rng(5000 + CASES.index(case))
    proj = crandn(rng, (B, P, N, N // 2 + 1))
    om = rng.uniform(0.5, 1.5, proj.shape).astype(np.float32) if with_w else None
    R = synth.random_rotations(Bp * P, rng).reshape(Bp, P, 3, 3)
    t = rng.uniform(-4, 4, (B, P, 2)).astype(np.float32) if shifted else None
    G = crandn(rng, (Bv, M, M, M // 2 + 1))
    GW = rng.standard_normal((Bv, M, M, M // 2 + 1)).astype(np.float32) if with_gw else None
    kw = dict(interp=interp, oversampling=s, radius=radius)
    gp, gw, gr, gt = tp.tp_backproject_2d_3d_backward(dev(G), dev(proj), dev(R), dev(t),
                                                      weights=dev(om), grad_weight_vol=dev(GW), **kw)
    rp, rw, rr, rt = oracle.backproject_backward(3, G, proj, R, shift=t, grad_weight=GW,
                                                 weights=om, **kw)
    assert rel(host(gp), rp) <= FWD_TOL
    assert rel(host(gr), rr) <= ATOMIC_TOL
    if shifted:
        assert rel(host(gt), rt) <= ATOMIC_TOL
    else:
        assert gt is None
    if with_gw:
        assert rel(host(gw), rw) <= FWD_TOL
    else:
        assert gw is None


def test_weight_terms_only(tp):
    """No data-spectrum gradient: only the weight terms of grad_rot."""
    rng = np.random.default_rng(41)
    M = N = 16
    proj = crandn(rng, (1, 3, N, N // 2 + 1))
    R = synth.random_rotations(3, rng).reshape(1, 3, 3, 3)
    GW = rng.standard_normal((1, M, M, M // 2 + 1)).astype(np.float32)
    zero = np.zeros((1, M, M, M // 2 + 1), np.complex64)
    _, gw, gr, _ = tp.tp_backproject_2d_3d_backward(dev(zero), dev(proj), dev(R),
                                                    grad_weight_vol=dev(GW), want_proj=False,
                                                    interp="cubic")
    _, rw, rr, _ = oracle.backproject_backward(3, zero, proj, R, grad_weight=GW, interp="cubic")
    assert rel(host(gw), rw) <= FWD_TOL
    assert rel(host(gr), rr) <= ATOMIC_TOL


def test_cfg4_box256_2048_images_sampled(tp):
    """The cfg-4 launch (2048 images into 256^3, cubic, radius 128) with
    random upstream spectra, compared on sampled images and poses."""
    w = synth.workload(4)
    proj, R = w["proj"], w["rot"]
    rng = np.random.default_rng(44)
    M = w["box"]
    G = crandn(rng, (1, M, M, M // 2 + 1))
    GW = rng.standard_normal((1, M, M, M // 2 + 1)).astype(np.float32)
    kw = dict(interp="cubic", oversampling=1.0, radius=w["radius"])
    gp, gw, gr, _ = tp.tp_backproject_2d_3d_backward(dev(G), dev(proj), dev(R),
                                                     grad_weight_vol=dev(GW), **kw)
    pick = np.arange(7, proj.shape[1], 256)
    rp, rw, rr, _ = oracle.backproject_backward(3, G, proj[:, pick], R[:, pick], grad_weight=GW,
                                                **kw)
    assert rel(host(gp)[:, pick], rp) <= FWD_TOL
    assert rel(host(gw)[:, pick], rw) <= FWD_TOL
    assert rel(host(gr)[:, pick], rr) <= ATOMIC_TOL
