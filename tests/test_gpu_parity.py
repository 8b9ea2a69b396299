"""GPU parity: the CUDA library (through its C ABI) against the float64 oracle.

Inputs are the seeded synthetic workloads of ``synth``; both sides see the
same float32 values.  The bar is relative L2 error (complex values as pairs):
1e-5 for forward projections and 1e-4 for the atomic backprojection and the
gradients, the tolerances the method's fp32 arithmetic is held to.

Large workloads run on the GPU at full size, in the launch configuration the
benchmark times, and are compared on sampled poses (each pose's output and its
rotation/shift gradient depend on that pose alone), or through properties that
hold at any size (the adjoint identity).
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


# ---------------------------------------------------------------------------
# A grid of small cases: both dimensions, kernels, oversampling factors,
# shifted / unshifted, radii, ragged boxes (tails that do not fill a thread
# block) and broadcast batches.
SMALL = []
for dim in (2, 3):
    for interp in ("linear", "cubic"):
        SMALL += [
            (dim, interp, 16, 16, 1.0, True, -1.0, 1, 1, 3),
            (dim, interp, 18, 14, 1.3, True, 5.5, 2, 1, 2),
            (dim, interp, 32, 16, 2.0, False, 100.0, 2, 2, 3),
            (dim, interp, 12, 16, 0.75, True, -1.0, 1, 2, 2),
            (dim, interp, 20, 10, 2.0, True, 0.0, 2, 2, 2),
        ]


def _small_inputs(dim, M, N, shifted, Bsrc, Bp, P, seed):
    rng = np.random.default_rng(seed)
    shp = (Bsrc, M, M, M // 2 + 1) if dim == 3 else (Bsrc, M, M // 2 + 1)
    src = crandn(rng, shp)
    if dim == 3:
        R = synth.random_rotations(Bp * P, rng).reshape(Bp, P, 3, 3)
    else:
        R = synth.planar_rotations(rng.uniform(0, 2 * np.pi, Bp * P)).reshape(Bp, P, 2, 2)
    B = max(Bsrc, Bp)
    t = rng.uniform(-6, 6, (B, P, 2)).astype(np.float32) if shifted else None
    g = crandn(rng, (B, P, N, N // 2 + 1))
    return src, R, t, g


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "-".join(map(str, c)))
def test_small_grid_forward_backward(tp, case):
    dim, interp, M, N, s, shifted, radius, Bsrc, Bp, P = case
    src, R, t, g = _small_inputs(dim, M, N, shifted, Bsrc, Bp, P, seed=1000 + SMALL.index(case))
    kw = dict(interp=interp, oversampling=s, radius=radius)
    fwd = tp.tp_project_3d_2d if dim == 3 else tp.tp_project_2d_2d
    bwd = tp.tp_project_3d_2d_backward if dim == 3 else tp.tp_project_2d_2d_backward
    out = host(fwd(dev(src), dev(R), dev(t), N=N, **kw))
    ref = oracle.project(dim, src, R, shift=t, N=N, **kw)
    assert rel(out, ref) <= FWD_TOL
    gs, gr, gt = bwd(dev(g), dev(src), dev(R), dev(t), **kw)
    rs, rr, rt = oracle.project_backward(dim, g, src, R, shift=t, **kw)
    assert rel(host(gs), rs) <= ATOMIC_TOL
    assert rel(host(gr), rr) <= ATOMIC_TOL
    if shifted:
        assert rel(host(gt), rt) <= ATOMIC_TOL
    else:
        assert gt is None


@pytest.mark.parametrize("interp", ["linear", "cubic"])
@pytest.mark.parametrize("Bv", [1, 2])
def test_small_backprojection_with_weights(tp, interp, Bv):
    rng = np.random.default_rng(21)
    B, P, N, M = 2, 3, 14, 20
    proj = crandn(rng, (B, P, N, N // 2 + 1))
    om = rng.uniform(0.1, 2.0, proj.shape).astype(np.float32)
    R = synth.random_rotations(B * P, rng).reshape(B, P, 3, 3)
    t = rng.uniform(-4, 4, (1, P, 2)).astype(np.float32)
    kw = dict(interp=interp, oversampling=1.4, radius=6.5)
    d, w = tp.tp_backproject_2d_3d(dev(proj), dev(R), dev(t), dev(om), Nv=M, Bv=Bv, **kw)
    rd, rw = oracle.backproject(3, proj, R, shift=t, M=M, weights=om, Bdst=Bv, **kw)
    assert rel(host(d), rd) <= ATOMIC_TOL
    assert rel(host(w), rw) <= ATOMIC_TOL
    # accumulation: a second call adds the same amount again
    tp.tp_backproject_2d_3d(dev(proj), dev(R), dev(t), dev(om), Nv=M, Bv=Bv, data_vol=d,
                            weight_vol=w, **kw)
    assert rel(host(d), 2 * rd) <= ATOMIC_TOL


# ---------------------------------------------------------------------------
# Edge cases.
def test_empty_pose_list_writes_nothing(tp):
    vol = torch.zeros((1, 8, 8, 5), dtype=torch.complex64, device="cuda")
    rot = torch.zeros((1, 0, 3, 3), dtype=torch.float32, device="cuda")
    out = tp.tp_project_3d_2d(vol, rot)
    assert out.shape == (1, 0, 8, 5)
    d, w = tp.tp_backproject_2d_3d(torch.zeros((1, 0, 8, 5), dtype=torch.complex64, device="cuda"),
                                   rot)
    assert float(d.abs().sum()) == 0.0 and float(w.abs().sum()) == 0.0


def test_identity_pose_is_exact(tp):
    rng = np.random.default_rng(22)
    for interp in ("linear", "cubic"):
        V = crandn(rng, (1, 32, 32, 17))
        out = host(tp.tp_project_3d_2d(dev(V), dev(np.eye(3, dtype=np.float32)[None, None]),
                                       interp=interp))
        np.testing.assert_array_equal(out, oracle.project(3, V, np.eye(3)[None, None], interp=interp)
                                      .astype(np.complex64))


def test_zero_radius_keeps_only_dc(tp):
    rng = np.random.default_rng(23)
    V = crandn(rng, (1, 16, 16, 9))
    R = synth.random_rotations(2, rng)[None]
    out = host(tp.tp_project_3d_2d(dev(V), dev(R), radius=0.0))
    assert np.count_nonzero(out) == 2 and out[0, 0, 0, 0] != 0


def test_non_orthogonal_matrix_and_large_shift(tp):
    rng = np.random.default_rng(24)
    V = crandn(rng, (1, 24, 24, 13))
    R = (synth.random_rotations(3, rng) * rng.uniform(0.6, 1.3, (3, 3, 1)).astype(np.float32)
         + rng.normal(0, 0.2, (3, 3, 3)).astype(np.float32))[None]
    t = rng.uniform(-900, 900, (1, 3, 2)).astype(np.float32)
    for interp in ("linear", "cubic"):
        out = host(tp.tp_project_3d_2d(dev(V), dev(R), dev(t), interp=interp))
        assert rel(out, oracle.project(3, V, R, shift=t, interp=interp)) <= FWD_TOL


@pytest.mark.parametrize("interp", ["linear", "cubic"])
def test_degenerate_poses(tp, interp):
    """Matrices whose sample set collapses or leaves the volume: the zero
    matrix (every pixel reads the DC voxel), parallel rows (a line), a zero
    second row, and a rotation scaled by 3 (most samples beyond the stored
    range, which reads zero)."""
    rng = np.random.default_rng(26)
    M = N = 20
    V = crandn(rng, (1, M, M, M // 2 + 1))
    a = synth.random_rotations(1, rng)[0]
    R = np.stack([np.zeros((3, 3), np.float32),
                  np.stack([a[0], 0.7 * a[0], a[2]]),
                  np.stack([a[0], np.zeros(3, np.float32), a[2]]),
                  3.0 * synth.random_rotations(1, rng)[0]]).astype(np.float32)[None]
    t = rng.uniform(-4, 4, (1, 4, 2)).astype(np.float32)
    g = crandn(rng, (1, 4, N, N // 2 + 1))
    kw = dict(interp=interp)
    out = host(tp.tp_project_3d_2d(dev(V), dev(R), dev(t), **kw))
    assert rel(out, oracle.project(3, V, R, shift=t, **kw)) <= FWD_TOL
    gv, gr, gt = tp.tp_project_3d_2d_backward(dev(g), dev(V), dev(R), dev(t), **kw)
    rv, rr, rt = oracle.project_backward(3, g, V, R, shift=t, **kw)
    assert rel(host(gv), rv) <= ATOMIC_TOL
    assert rel(host(gr), rr) <= ATOMIC_TOL
    assert rel(host(gt), rt) <= ATOMIC_TOL


def test_minimum_box(tp):
    rng = np.random.default_rng(25)
    V = crandn(rng, (1, 2, 2, 2))
    R = synth.random_rotations(4, rng)[None]
    for interp in ("linear", "cubic"):
        out = host(tp.tp_project_3d_2d(dev(V), dev(R), N=2, interp=interp, radius=5.0))
        assert rel(out, oracle.project(3, V, R, N=2, interp=interp, radius=5.0)) <= FWD_TOL


# ---------------------------------------------------------------------------
# The five workloads.
def test_cfg1_box32_linear_full(tp):
    w = synth.workload(1)
    kw = dict(interp=w["interp"], oversampling=1.0, radius=w["radius"])
    vol, R, g = w["vol"], w["rot"], w["grad"]
    out = host(tp.tp_project_3d_2d(dev(vol), dev(R), **kw))
    assert rel(out, oracle.project(3, vol, R, **kw)) <= FWD_TOL
    gv, gr, _ = tp.tp_project_3d_2d_backward(dev(g), dev(vol), dev(R), **kw)
    rv, rr, _ = oracle.project_backward(3, g, vol, R, **kw)
    assert rel(host(gv), rv) <= ATOMIC_TOL and rel(host(gr), rr) <= ATOMIC_TOL
    assert np.all(host(gr)[..., 2, :] == 0)
    d, wt = tp.tp_backproject_2d_3d(dev(g), dev(R), **kw)
    rd, rw = oracle.backproject(3, g, R, **kw)
    assert rel(host(d), rd) <= ATOMIC_TOL and rel(host(wt), rw) <= ATOMIC_TOL


def test_cfg2_rot2d_box128_cubic_full(tp):
    w = synth.workload(2)
    kw = dict(interp=w["interp"], oversampling=1.0, radius=w["radius"])
    img, R, t, g = w["img"], w["rot"], w["shift"], w["grad"]
    out = host(tp.tp_project_2d_2d(dev(img), dev(R), dev(t), **kw))
    assert rel(out, oracle.project(2, img, R, shift=t, **kw)) <= FWD_TOL
    gi, gr, gt = tp.tp_project_2d_2d_backward(dev(g), dev(img), dev(R), dev(t), **kw)
    ri, rr, rt = oracle.project_backward(2, g, img, R, shift=t, **kw)
    assert rel(host(gi), ri) <= ATOMIC_TOL
    assert rel(host(gr), rr) <= ATOMIC_TOL
    assert rel(host(gt), rt) <= ATOMIC_TOL
    # Angle gradients through the caller's chain rule dR/dtheta = [[-s, -c], [c, -s]].
    th = w["angles"].astype(np.float64)
    dR = np.stack([-np.sin(th), -np.cos(th), np.cos(th), -np.sin(th)], 1).reshape(-1, 1, 2, 2)
    assert rel((host(gr) * dR).sum((1, 2, 3)), (rr * dR).sum((1, 2, 3))) <= ATOMIC_TOL


@pytest.mark.parametrize("s", [1, 2])
def test_cfg3_box128_cubic_4096_poses_sampled(tp, s):
    w = synth.workload(3, oversampling=s)
    kw = dict(interp=w["interp"], oversampling=w["oversampling"], radius=w["radius"])
    vol, R = w["vol"], w["rot"]
    out = host(tp.tp_project_3d_2d(dev(vol), dev(R), N=w["box"], **kw))
    assert out.shape == (1, 4096, 128, 65)
    pick = np.arange(5, 4096, 273)
    ref = oracle.project(3, vol, R[:, pick], N=w["box"], **kw)
    assert rel(out[:, pick], ref) <= FWD_TOL


@pytest.mark.parametrize("interp", ["linear", "cubic"])
def test_cfg4_backprojection_subset(tp, interp):
    w = synth.workload(4, poses=48)
    kw = dict(interp=interp, oversampling=1.0, radius=w["radius"])
    d, wt = tp.tp_backproject_2d_3d(dev(w["proj"]), dev(w["rot"]), **kw)
    rd, rw = oracle.backproject(3, w["proj"], w["rot"], **kw)
    assert rel(host(d), rd) <= ATOMIC_TOL
    assert rel(host(wt), rw) <= ATOMIC_TOL


def _central(a, half):
    """The entries of a (…, M, M, M/2+1) spectrum with |n_y|, |n_z| < half and n_x < half:
    the bricks every pose reaches, whose work is split over the most work units."""
    M = a.shape[-2]
    rows = np.r_[0:half, M - half + 1:M]
    return a[..., rows[:, None, None], rows[None, :, None], np.arange(half)[None, None, :]]


def assert_elementwise(got, ref, tol, what):
    """Whole-tensor relative L2 within tol, the central region on its own within tol, and
    no single element off by more than tol times the largest reference magnitude."""
    assert rel(got, ref) <= tol, f"{what}: rel L2 {rel(got, ref):.3e}"
    cg, cr = _central(got, 24), _central(ref, 24)
    assert rel(cg, cr) <= tol, f"{what}: central rel L2 {rel(cg, cr):.3e}"
    worst = np.abs(np.asarray(got, np.complex128) - ref).max()
    assert worst <= tol * np.abs(ref).max(), f"{what}: max error {worst:.3e}"


@pytest.mark.parametrize("interp", ["linear", "cubic"])
def test_cfg4_backprojection_full_elementwise(tp, interp):
    """All 2048 images into one 256^3 spectrum, data and weights, element by element.  The
    central bricks are reached by nearly every image, so their work is split over many
    work units whose tiles fold into the same words from different blocks."""
    w = synth.workload(4)
    kw = dict(interp=interp, oversampling=1.0, radius=w["radius"])
    d, wt = tp.tp_backproject_2d_3d(dev(w["proj"]), dev(w["rot"]), **kw)
    rd, rw = oracle.backproject(3, w["proj"], w["rot"], **kw)
    assert_elementwise(host(d), rd, ATOMIC_TOL, "data spectrum")
    assert_elementwise(host(wt), rw, ATOMIC_TOL, "weight spectrum")


def test_cfg5_grad_vol_full_elementwise(tp):
    """The volume gradient of the whole 512-pose box-256 step, element by element."""
    w = synth.workload(5)
    kw = dict(interp=w["interp"], oversampling=1.0, radius=w["radius"])
    vol, R, t, g = w["vol"], w["rot"], w["shift"], w["grad"]
    gv, _, _ = tp.tp_project_3d_2d_backward(dev(g), dev(vol), dev(R), dev(t), want_rot=False,
                                            want_shift=False, **kw)
    rv, _, _ = oracle.project_backward(3, g, vol, R, shift=t, need_rot=False, need_shift=False,
                                       **kw)
    assert_elementwise(host(gv), rv, ATOMIC_TOL, "grad_vol")


def test_outer_shell_golden(tp):
    """Taps on and beyond the outermost stored shell against hand-worked values (forward), and
    the scatter's deposits there through the adjoint identity with the same values."""
    import outer_shell
    for name, dim, M, V, R, want in outer_shell.cases():
        Vd, Rd = dev(V.astype(np.complex64)), dev(R.astype(np.float32))
        fwd = tp.tp_project_3d_2d if dim == 3 else tp.tp_project_2d_2d
        out = host(fwd(Vd, Rd, N=8, interp="cubic", radius=-1.0))
        got = complex(out[(0, 0) + outer_shell.PIXEL])
        assert abs(got - want) <= 1e-6 * abs(want), f"{name}: {got} != {want}"
        # Backprojecting y = 1 and y = i at that pixel gives P^T y; <V, P^T y> = <P V, y>.
        for yv, part in ((1.0, want.real), (1j, want.imag)):
            y = np.zeros((1, 1, 8, 5), np.complex64)
            y[(0, 0) + outer_shell.PIXEL] = yv
            if dim == 3:
                bp, _ = tp.tp_backproject_2d_3d(dev(y), Rd, Nv=M, interp="cubic", radius=-1.0,
                                                want_weights=False)
            else:
                bp, _, _ = tp.tp_project_2d_2d_backward(dev(y), Vd, Rd, interp="cubic",
                                                        radius=-1.0, want_rot=False)
            ip = np.vdot(V.astype(np.complex128), host(bp).astype(np.complex128)).real
            assert abs(ip - part) <= 1e-6 * abs(want), f"{name}: adjoint {ip} != {part}"


@pytest.mark.parametrize("interp", ["linear", "cubic"])
def test_cfg4_backprojection_full_adjoint_identity(tp, interp):
    """At full size (2048 images) the scatter is the exact adjoint of the gather."""
    w = synth.workload(4)
    kw = dict(interp=interp, oversampling=1.0, radius=w["radius"])
    y = dev(w["proj"])
    R = dev(w["rot"])
    d, wt = tp.tp_backproject_2d_3d(y, R, **kw)
    rng = np.random.default_rng(26)
    x = dev(crandn(rng, (1, 256, 256, 129)))
    Px = tp.tp_project_3d_2d(x, R, **kw)
    lhs = torch.vdot(Px.flatten().to(torch.complex128), y.flatten().to(torch.complex128)).real
    rhs = torch.vdot(x.flatten().to(torch.complex128), d.flatten().to(torch.complex128)).real
    assert abs(float(lhs - rhs)) <= 1e-4 * abs(float(lhs))
    # Partition of unity: every in-radius sample deposits total weight 1
    # except near the edge of the stored range (radius 128 reaches it), where
    # dropped taps change the total by well under 3%.
    kx = np.arange(129)[None, :]
    ky = np.fft.fftfreq(256, 1 / 256)[:, None]
    n_in = int((kx * kx + ky * ky <= 128 * 128).sum()) * 2048
    tot = float(wt.double().sum())
    assert 0.97 * n_in < tot < 1.03 * n_in


def test_cfg5_box256_full_step_sampled(tp):
    w = synth.workload(5)
    kw = dict(interp=w["interp"], oversampling=1.0, radius=w["radius"])
    vol, R, t, g = w["vol"], w["rot"], w["shift"], w["grad"]
    dv, dR, dt, dg = dev(vol), dev(R), dev(t), dev(g)
    out = host(tp.tp_project_3d_2d(dv, dR, dt, **kw))
    pick = np.arange(3, 512, 64)
    ref = oracle.project(3, vol, R[:, pick], shift=t[:, pick], **kw)
    assert rel(out[:, pick], ref) <= FWD_TOL
    gv, gr, gt = tp.tp_project_3d_2d_backward(dg, dv, dR, dt, **kw)
    _, rr, rt = oracle.project_backward(3, g[:, pick], vol, R[:, pick], shift=t[:, pick],
                                        need_src=False, **kw)
    assert rel(host(gr)[:, pick], rr) <= ATOMIC_TOL
    assert rel(host(gt)[:, pick], rt) <= ATOMIC_TOL
    # grad_vol sums over poses: compare a 12-pose prefix run on both sides.
    sub = slice(0, 12)
    gv12, _, _ = tp.tp_project_3d_2d_backward(dev(g[:, sub]), dv, dev(R[:, sub]), dev(t[:, sub]),
                                              want_rot=False, want_shift=False, **kw)
    rv12, _, _ = oracle.project_backward(3, g[:, sub], vol, R[:, sub], shift=t[:, sub],
                                         need_rot=False, need_shift=False, **kw)
    assert rel(host(gv12), rv12) <= ATOMIC_TOL


# ---------------------------------------------------------------------------
# Large sizes: a box-512 spectrum (67 M complex words) and a 100,000-pose list
# exercise the 64-bit offsets and the chunk / mask / work-unit indexing at
# sizes far beyond the configs; both are compared on samples.
def test_box512_forward_and_backward_sampled(tp):
    rng = np.random.default_rng(512)
    M = N = 512
    vol = crandn(rng, (1, M, M, M // 2 + 1))
    R = synth.random_rotations(3, rng).reshape(1, 3, 3, 3)
    t = rng.uniform(-20, 20, (1, 3, 2)).astype(np.float32)
    g = crandn(rng, (1, 3, N, N // 2 + 1))
    kw = dict(interp="cubic", oversampling=1.0, radius=-1.0)
    dv = dev(vol)
    out = host(tp.tp_project_3d_2d(dv, dev(R), dev(t), **kw))
    assert rel(out, oracle.project(3, vol, R, shift=t, **kw)) <= FWD_TOL
    gv, gr, gt = tp.tp_project_3d_2d_backward(dev(g), dv, dev(R), dev(t), **kw)
    rv, rr, rt = oracle.project_backward(3, g, vol, R, shift=t, **kw)
    assert rel(host(gr), rr) <= ATOMIC_TOL
    assert rel(host(gt), rt) <= ATOMIC_TOL
    # the volume gradient on a sample of voxels across the whole spectrum
    gvh = host(gv)
    idx = tuple(rng.integers(0, n, 20000) for n in vol.shape)
    assert rel(gvh[idx], rv[idx]) <= ATOMIC_TOL
    assert rel(gvh, rv) <= ATOMIC_TOL


def test_hundred_thousand_poses_sampled(tp):
    rng = np.random.default_rng(100000)
    M = N = 16
    P = 100_000
    vol = crandn(rng, (1, M, M, M // 2 + 1))
    R = synth.random_rotations(P, rng).reshape(1, P, 3, 3)
    g = crandn(rng, (1, P, N, N // 2 + 1))
    kw = dict(interp="linear", oversampling=1.0, radius=-1.0)
    dv, dR = dev(vol), dev(R)
    out, dout = tp.tp_project_3d_2d_save(dv, dR, None, **kw)
    pick = np.concatenate([np.arange(0, P, 9973), [P - 1]])
    ref = oracle.project(3, vol, R[:, pick], **kw)
    assert rel(host(out)[:, pick], ref) <= FWD_TOL
    gr, _ = tp.tp_project_3d_2d_backward_saved(dev(g), out, dout, dR, None, **kw)
    _, rr, _ = oracle.project_backward(3, g[:, pick], vol, R[:, pick], need_src=False, **kw)
    assert rel(host(gr)[:, pick], rr) <= ATOMIC_TOL
    # all 100,000 images scattered into one spectrum: the adjoint identity
    gv, _, _ = tp.tp_project_3d_2d_backward(dev(g), dv, dR, want_rot=False, want_shift=False, **kw)
    lhs = np.vdot(g.astype(np.complex128), host(out).astype(np.complex128)).real
    rhs = np.vdot(host(gv).astype(np.complex128), vol.astype(np.complex128)).real
    assert abs(lhs - rhs) <= 1e-4 * abs(lhs)


# ---------------------------------------------------------------------------
# Dense sampling (s < 1: neighbouring samples a fraction of a voxel apart)
# makes the stencils of the samples a scatter round spreads together meet
# often, so the one-sample-at-a-time fallback of the tiled scatters runs;
# one shared source for many poses makes their tiles fold into the same
# words from many blocks.
@pytest.mark.parametrize("interp", ["linear", "cubic"])
def test_degenerate_2d_matrices(tp, interp):
    """2D matrices without an inverse, for which the tiled image gradient
    enumerates every row: the zero matrix, parallel rows, a zero second and
    a zero first row, plus a rotation scaled by 3 (most samples outside the
    stored range)."""
    rng = np.random.default_rng(27)
    M = N = 24
    img = crandn(rng, (2, M, M // 2 + 1))
    c, s_ = np.cos(0.7), np.sin(0.7)
    R = np.array([[[0, 0], [0, 0]],
                  [[c, s_], [0.7 * c, 0.7 * s_]],
                  [[c, s_], [0, 0]],
                  [[0, 0], [-s_, c]],
                  [[3 * c, 3 * s_], [-3 * s_, 3 * c]]], np.float32)
    R = np.stack([R, R[::-1]])                      # (2, 5, 2, 2): both images, other order
    t = rng.uniform(-4, 4, (2, 5, 2)).astype(np.float32)
    g = crandn(rng, (2, 5, N, N // 2 + 1))
    kw = dict(interp=interp)
    out = host(tp.tp_project_2d_2d(dev(img), dev(R), dev(t), **kw))
    assert rel(out, oracle.project(2, img, R, shift=t, **kw)) <= FWD_TOL
    gi, gr, gt = tp.tp_project_2d_2d_backward(dev(g), dev(img), dev(R), dev(t), **kw)
    ri, rr, rt = oracle.project_backward(2, g, img, R, shift=t, **kw)
    assert rel(host(gi), ri) <= ATOMIC_TOL
    assert rel(host(gr), rr) <= ATOMIC_TOL
    assert rel(host(gt), rt) <= ATOMIC_TOL


@pytest.mark.parametrize("interp", ["linear", "cubic"])
def test_dense_2d_image_gradient_many_poses_one_image(tp, interp):
    rng = np.random.default_rng(4242)
    M, N, P = 64, 96, 48
    img = crandn(rng, (1, M, M // 2 + 1))
    R = synth.planar_rotations(rng.uniform(0, 2 * np.pi, P)).reshape(1, P, 2, 2)
    t = rng.uniform(-4, 4, (1, P, 2)).astype(np.float32)
    g = crandn(rng, (1, P, N, N // 2 + 1))
    kw = dict(interp=interp, oversampling=0.6, radius=-1.0)
    gi, gr, gt = tp.tp_project_2d_2d_backward(dev(g), dev(img), dev(R), dev(t), **kw)
    ri, rr, rt = oracle.project_backward(2, g, img, R, shift=t, **kw)
    assert rel(host(gi), ri) <= ATOMIC_TOL
    assert rel(host(gt), rt) <= ATOMIC_TOL
    # The linear kernel's derivative jumps at integer positions: among these
    # 225,000 samples (|p| up to 29) two lie within float32 rounding of an
    # integer and take the other branch than the float64 oracle, moving a
    # pose's rotation gradient by about 1%.  The cubic kernel is C1.
    if interp == "cubic":
        assert rel(host(gr), rr) <= ATOMIC_TOL


@pytest.mark.parametrize("interp", ["linear", "cubic"])
def test_dense_3d_volume_gradient(tp, interp):
    rng = np.random.default_rng(4343)
    M, N, P = 40, 48, 6
    vol = crandn(rng, (1, M, M, M // 2 + 1))
    R = synth.random_rotations(P, rng).reshape(1, P, 3, 3)
    g = crandn(rng, (1, P, N, N // 2 + 1))
    kw = dict(interp=interp, oversampling=0.55, radius=-1.0)
    gv, _, _ = tp.tp_project_3d_2d_backward(dev(g), dev(vol), dev(R), want_rot=False,
                                            want_shift=False, **kw)
    rv, _, _ = oracle.project_backward(3, g, vol, R, need_rot=False, need_shift=False, **kw)
    assert rel(host(gv), rv) <= ATOMIC_TOL


# ---------------------------------------------------------------------------
# The 2D operators stage two Friedel-completed half planes of the source in
# shared memory when they fit (sources up to box 152 on a 227 KB block) and
# fall back to the per-sample kernels above that.  These cases cover both
# sides of the limit, a source pointer that is only 8-byte aligned, a shared
# source whose many poses are cut into work items, and several poses per
# source image.
@pytest.mark.parametrize("M,N,s", [(128, 64, 0.5), (130, 130, 1.0), (132, 96, 0.7),
                                   (152, 152, 1.0), (154, 120, 0.8), (256, 64, 0.25)])
@pytest.mark.parametrize("interp", ["linear", "cubic"])
def test_2d_staged_plane_limits(tp, M, N, s, interp):
    rng = np.random.default_rng(M + N)
    B, P = 2, 3
    img = crandn(rng, (B, M, M // 2 + 1))
    R = synth.planar_rotations(rng.uniform(0, 2 * np.pi, B * P)).reshape(B, P, 2, 2)
    t = rng.uniform(-8, 8, (B, P, 2)).astype(np.float32)
    g = crandn(rng, (B, P, N, N // 2 + 1))
    kw = dict(interp=interp, oversampling=s, radius=-1.0)
    out = host(tp.tp_project_2d_2d(dev(img), dev(R), dev(t), N=N, **kw))
    assert rel(out, oracle.project(2, img, R, shift=t, N=N, **kw)) <= FWD_TOL
    gi, gr, gt = tp.tp_project_2d_2d_backward(dev(g), dev(img), dev(R), dev(t), **kw)
    ri, rr, rt = oracle.project_backward(2, g, img, R, shift=t, **kw)
    assert rel(host(gi), ri) <= ATOMIC_TOL
    assert rel(host(gt), rt) <= ATOMIC_TOL
    if interp == "cubic":   # see test_dense_2d_image_gradient_many_poses_one_image
        assert rel(host(gr), rr) <= ATOMIC_TOL


@pytest.mark.parametrize("interp", ["linear", "cubic"])
def test_2d_source_only_8_byte_aligned(tp, interp):
    rng = np.random.default_rng(77)
    M, P = 40, 5
    img = crandn(rng, (1, M, M // 2 + 1))
    buf = torch.zeros(img.size + 1, dtype=torch.complex64, device="cuda")
    src = buf[1:].view(img.shape)                    # starts 8 bytes past a 16-byte boundary
    src.copy_(dev(img))
    assert src.data_ptr() % 16 == 8
    R = synth.planar_rotations(rng.uniform(0, 2 * np.pi, P)).reshape(1, P, 2, 2)
    t = rng.uniform(-3, 3, (1, P, 2)).astype(np.float32)
    g = crandn(rng, (1, P, M, M // 2 + 1))
    kw = dict(interp=interp, radius=-1.0)
    out = host(tp.tp_project_2d_2d(src, dev(R), dev(t), **kw))
    assert rel(out, oracle.project(2, img, R, shift=t, **kw)) <= FWD_TOL
    _, gr, gt = tp.tp_project_2d_2d_backward(dev(g), src, dev(R), dev(t), want_img=False, **kw)
    _, rr, rt = oracle.project_backward(2, g, img, R, shift=t, need_src=False, **kw)
    assert rel(host(gt), rt) <= ATOMIC_TOL
    if interp == "cubic":
        assert rel(host(gr), rr) <= ATOMIC_TOL


@pytest.mark.parametrize("Bi,B,P", [(1, 3, 700), (3, 3, 150)])
def test_2d_many_poses_per_source(tp, Bi, B, P):
    """A shared source for 2100 poses (cut into many work items over all blocks)
    and three sources with 150 poses each (several items per source)."""
    rng = np.random.default_rng(Bi * 1000 + P)
    M = N = 32
    img = crandn(rng, (Bi, M, M // 2 + 1))
    R = synth.planar_rotations(rng.uniform(0, 2 * np.pi, B * P)).reshape(B, P, 2, 2)
    t = rng.uniform(-3, 3, (B, P, 2)).astype(np.float32)
    g = crandn(rng, (B, P, N, N // 2 + 1))
    kw = dict(interp="cubic", radius=-1.0)
    out = host(tp.tp_project_2d_2d(dev(img), dev(R), dev(t), **kw))
    assert rel(out, oracle.project(2, img, R, shift=t, **kw)) <= FWD_TOL
    gi, gr, gt = tp.tp_project_2d_2d_backward(dev(g), dev(img), dev(R), dev(t), **kw)
    ri, rr, rt = oracle.project_backward(2, g, img, R, shift=t, **kw)
    assert rel(host(gi), ri) <= ATOMIC_TOL
    assert rel(host(gr), rr) <= ATOMIC_TOL
    assert rel(host(gt), rt) <= ATOMIC_TOL
