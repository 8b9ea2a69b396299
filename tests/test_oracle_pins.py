"""Pins of the float64 oracle against facts fixed outside the oracle itself.

Each test checks the oracle against mathematics or physics that does not
depend on its code: exact real-space permutations and numpy FFTs, the exact
discrete-time Fourier transform, closed-form Gaussian line integrals, the
polynomial reproduction of the interpolation kernels, textbook Catmull-Rom
weights, the adjoint identity and finite differences.  A plausible slip in
the oracle (a transposed rotation, a wrong tap offset, a dropped conjugate, a
flipped phase sign) fails at least one of them.
"""
import itertools
import os

import numpy as np
import pytest

import oracle
import synth


def crandn(rng, shape):
    return rng.standard_normal(shape) + 1j * rng.standard_normal(shape)


def fftfreq_int(M):
    return np.fft.fftfreq(M, 1.0 / M).astype(int)


def pixel_freqs(N):
    """(N, N/2+1) arrays of kx, ky for an output image."""
    ky = fftfreq_int(N)[:, None] * np.ones((1, N // 2 + 1), int)
    kx = np.arange(N // 2 + 1)[None, :] * np.ones((N, 1), int)
    return kx, ky


def in_radius(N, r):
    kx, ky = pixel_freqs(N)
    return kx * kx + ky * ky <= r * r


def signed_permutation_rotations():
    """The 24 proper rotations that map the integer grid onto itself."""
    out = []
    for perm in itertools.permutations(range(3)):
        for signs in itertools.product((1, -1), repeat=3):
            R = np.zeros((3, 3))
            for i in range(3):
                R[i, perm[i]] = signs[i]
            if np.linalg.det(R) > 0:
                out.append(R)
    assert len(out) == 24
    return out


def rotate_density_exact(d, R):
    """d'(x) = d(R^T x) on the periodic grid centred at index M/2 (R a signed permutation)."""
    M = d.shape[0]
    c = np.arange(M) - M // 2
    Z, Y, X = np.meshgrid(c, c, c, indexing="ij")
    coords = np.stack([X.ravel(), Y.ravel(), Z.ravel()])       # (x, y, z) per voxel
    src = np.rint(R.T @ coords).astype(int)                     # R^T x
    sx, sy, sz = ((src + M // 2) % M)
    return d[sz, sy, sx].reshape(d.shape)


# --------------------------------------------------------------------------
# P1: identity pose reads the z = 0 plane exactly (both kernels interpolate).
@pytest.mark.parametrize("interp", ["linear", "cubic"])
def test_identity_pose_reads_central_plane(interp):
    rng = np.random.default_rng(1)
    M = 16
    V = crandn(rng, (1, M, M, M // 2 + 1))
    out = oracle.project(3, V, np.eye(3)[None, None], N=M, interp=interp)
    mask = in_radius(M, M / 2)
    np.testing.assert_array_equal(out[0, 0], np.where(mask, V[0, 0], 0))


# P2: the 24 grid rotations against an exact real-space rotation + projection.
def test_grid_rotations_match_real_space_projection():
    rng = np.random.default_rng(2)
    M = 16
    d = rng.standard_normal((M, M, M))
    V = np.fft.rfftn(np.fft.ifftshift(d))[None]
    r = M / 2 - 1                          # keeps the Nyquist shell out
    mask = in_radius(M, r)
    for R in signed_permutation_rotations():
        img = rotate_density_exact(d, R).sum(axis=0)              # line integral along z
        ref = np.fft.rfft2(np.fft.ifftshift(img))
        for interp in ("linear", "cubic"):
            out = oracle.project(3, V, R[None, None], N=M, interp=interp, radius=r)[0, 0]
            np.testing.assert_allclose(out[mask], ref[mask], rtol=0, atol=1e-9 * np.abs(ref).max())
            assert np.all(out[~mask] == 0)


def test_quarter_turn_is_not_its_transpose():
    """A quarter turn about z distinguishes R from R^T; the real-space truth decides."""
    rng = np.random.default_rng(3)
    M = 16
    d = rng.standard_normal((M, M, M))
    V = np.fft.rfftn(np.fft.ifftshift(d))[None]
    Rz = np.array([[0.0, -1.0, 0.0], [1.0, 0.0, 0.0], [0.0, 0.0, 1.0]])
    ref = np.fft.rfft2(np.fft.ifftshift(rotate_density_exact(d, Rz).sum(axis=0)))
    mask = in_radius(M, M / 2 - 1)
    good = oracle.project(3, V, Rz[None, None], interp="cubic", radius=M / 2 - 1)[0, 0]
    bad = oracle.project(3, V, Rz.T[None, None], interp="cubic", radius=M / 2 - 1)[0, 0]
    assert np.abs(good[mask] - ref[mask]).max() < 1e-9 * np.abs(ref).max()
    assert np.abs(bad[mask] - ref[mask]).max() > 1e-2 * np.abs(ref).max()


def test_2d_quarter_turns_match_rot90():
    """2D rotation convention: the forward by a quarter turn R equals the rfft2 of the image
    turned by np.rot90 about the grid origin, and its transpose (the inverse turn) does not."""
    rng = np.random.default_rng(31)
    M = 16
    e = np.fft.ifftshift(rng.standard_normal((M, M)))      # object centre at index 0
    V = np.fft.rfft2(e)[None]
    # np.rot90 turns the array about the centre of its corner pixels; rolling one row puts
    # the turn's fixed point back on index 0: new[y][x] = old[x][-y], i.e. d'(x, y) =
    # d(-y, x) = d(R^T (x, y)) with R = [[0, 1], [-1, 0]].
    Q = np.array([[0.0, 1.0], [-1.0, 0.0]])
    mask = in_radius(M, M / 2 - 1)                          # keeps the Nyquist shell out
    turned = e
    R = np.eye(2)
    for quarter in range(1, 4):
        turned = np.roll(np.rot90(turned), 1, axis=0)
        R = R @ Q
        ref = np.fft.rfft2(turned)
        for interp in ("linear", "cubic"):
            out = oracle.project(2, V, R[None, None], interp=interp, radius=M / 2 - 1)[0, 0]
            np.testing.assert_allclose(out[mask], ref[mask], rtol=0, atol=1e-10 * np.abs(ref).max())
        if quarter != 2:                                    # a half turn is its own transpose
            bad = oracle.project(2, V, R.T[None, None], interp="cubic", radius=M / 2 - 1)[0, 0]
            assert np.abs(bad[mask] - ref[mask]).max() > 1e-2 * np.abs(ref).max()


def test_outer_shell_golden_values():
    """Taps on and beyond the outermost stored shell, against hand-worked values: -M/2 is
    stored, +M/2 and x > M/2 read zero, Friedel taps reflect before the range test."""
    import outer_shell
    for name, dim, M, V, R, want in outer_shell.cases():
        out = oracle.project(dim, V, R, N=8, interp="cubic", radius=-1.0)
        got = out[(0, 0) + outer_shell.PIXEL]
        assert abs(got - want) <= 1e-15, f"{name}: {got} != {want}"


# P3: kernels reproduce polynomials; Catmull-Rom midpoint weights are textbook.
def _poly(c, x, y, z, cubic):
    v = c[0] + c[1] * x + c[2] * y + c[3] * z + c[5] * y * z + c[6] * x * y * z
    if cubic:
        v = v + c[4] * x * x + c[7] * y * y * z + c[8] * x * x * y * y * z * z
    return v


@pytest.mark.parametrize("interp", ["linear", "cubic"])
def test_polynomial_reproduction(interp):
    """Trilinear reproduces multilinear terms; Keys a=-1/2 reproduces per-axis quadratics."""
    cubic = interp == "cubic"
    rng = np.random.default_rng(4)
    M = 32
    c = crandn(rng, 9) * np.array([1, 0.3, 0.3, 0.3, 0.02, 0.02, 0.003, 0.002, 1e-6])
    X = M // 2 + 1
    f = fftfreq_int(M)
    Z, Y, Xg = np.meshgrid(f, f, np.arange(X), indexing="ij")
    V = _poly(c, Xg, Y, Z, cubic)[None]
    R = synth.random_rotations(6, np.random.default_rng(5)).astype(np.float64)
    s = 1.0
    N = 32
    out = oracle.project(3, V, R[None], N=N, interp=interp, oversampling=s)
    kx, ky = pixel_freqs(N)
    lo, hi = (1, 2) if cubic else (0, 1)
    checked = 0
    for pi in range(R.shape[0]):
        p = s * (R[pi][0][:, None, None] * kx + R[pi][1][:, None, None] * ky)
        fl = np.floor(p)
        direct = (fl[0] - lo >= 0) & (fl[0] + hi <= M // 2)
        friedel = (fl[0] + hi < 0) & (-(fl[0] - lo) <= M // 2)
        inside = np.ones_like(direct)
        for a in (1, 2):
            inside &= (fl[a] - lo >= -M // 2) & (fl[a] + hi <= M // 2 - 1)
            inside &= (-(fl[a] + hi) >= -M // 2) & (-(fl[a] - lo) <= M // 2 - 1)
        m1 = direct & inside & in_radius(N, N / 2)
        m2 = friedel & inside & in_radius(N, N / 2)
        want_d = _poly(c, p[0], p[1], p[2], cubic)
        want_f = np.conj(_poly(c, -p[0], -p[1], -p[2], cubic))
        np.testing.assert_allclose(out[0, pi][m1], want_d[m1], rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(out[0, pi][m2], want_f[m2], rtol=1e-11, atol=1e-11)
        checked += m1.sum() + m2.sum()
    assert checked > 500


def test_catmull_rom_golden_weights(golden_dir):
    """Sampling at x0 + t with s = t-fraction reproduces Keys' tabulated weights."""
    rows = np.loadtxt(os.path.join(golden_dir, "catmull_rom_midpoint.txt"))
    rng = np.random.default_rng(6)
    M = 32
    V = crandn(rng, (1, M, M, M // 2 + 1))
    for t, *w in rows:
        # Identity rotation scaled by s = 1 + t/8 moves pixel kx = 8 to p_x = 8 + t.
        s = 1.0 + t / 8.0
        out = oracle.project(3, V, np.eye(3)[None, None], N=M, interp="cubic", oversampling=s,
                             radius=8.0)
        want = sum(wj * V[0, 0, 0, 7 + j] for j, wj in enumerate(w))
        np.testing.assert_allclose(out[0, 0, 0, 8], want, rtol=1e-13)


# P4: Fourier-slice theorem against brute force.
def _dtft(d, pts, M):
    """Exact DTFT of a centred density d at (n, 3) frequency points p (units of 1/M)."""
    c = np.arange(M) - M // 2
    Z, Y, X = np.meshgrid(c, c, c, indexing="ij")
    coords = np.stack([X.ravel(), Y.ravel(), Z.ravel()], 1).astype(float)
    return np.exp(-2j * np.pi * (pts @ coords.T) / M) @ d.ravel()


def test_fourier_slice_vs_exact_dtft():
    """Interpolated central slices approach the exact DTFT; cubic beats linear, s=2 beats s=1."""
    M = 16
    rng = synth.streams(77, 2)
    cen, sig, amp = synth.blob_params(M, 6, rng[0], 3)
    d = synth.blob_density(M, cen, sig, amp, 3)
    R = synth.random_rotations(3, rng[1]).astype(np.float64)
    N = M
    r = N / 2 - 1
    mask = in_radius(N, r)
    kx, ky = pixel_freqs(N)
    k = np.stack([kx[mask], ky[mask], np.zeros(mask.sum())], 1).astype(float)
    errs = {}
    for s, box in ((1, M), (2, 2 * M)):
        dp = np.zeros((box,) * 3)
        o = box // 2 - M // 2
        dp[o:o + M, o:o + M, o:o + M] = d                      # real-space zero padding
        V = np.fft.rfftn(np.fft.ifftshift(dp))[None]
        for interp in ("linear", "cubic"):
            out = oracle.project(3, V, R[None], N=N, interp=interp, oversampling=s, radius=r)
            e2 = n2 = 0.0
            for pi in range(R.shape[0]):
                exact = _dtft(d, k @ R[pi], M)                  # p = R^T k (row vector k @ R)
                e2 += np.sum(np.abs(out[0, pi][mask] - exact) ** 2)
                n2 += np.sum(np.abs(exact) ** 2)
            errs[(s, interp)] = np.sqrt(e2 / n2)
    assert errs[(1, "cubic")] < errs[(1, "linear")]
    assert errs[(2, "cubic")] < errs[(2, "linear")]
    assert errs[(2, "linear")] < errs[(1, "linear")]
    # Calibrated bounds (box 16, six blobs): the error is interpolation only.
    assert errs[(1, "cubic")] < 0.08 and errs[(2, "cubic")] < 0.015
    assert errs[(1, "linear")] < 0.2
    # Cubic at 1x is comparable to linear at 2x oversampling (the pages' accuracy claim).
    assert errs[(1, "cubic")] < 2.0 * errs[(2, "linear")]


def test_fourier_slice_vs_analytic_gaussian_projection():
    """A rotated, shifted 3D Gaussian projects to a 2D Gaussian of amplitude a*sqrt(2 pi)*sigma.

    The reference is the closed-form line integral sampled on the image grid;
    a flipped shift sign or a transposed rotation is off by O(1).
    """
    M = 32
    rng = np.random.default_rng(8)
    c3 = rng.uniform(-4, 4, 3)
    sigma, a = 2.0, 0.8
    R = synth.random_rotations(2, rng).astype(np.float64)
    t = rng.uniform(-3, 3, (2, 2))
    g = np.arange(M) - M // 2
    Y2, X2 = np.meshgrid(g, g, indexing="ij")
    mask = in_radius(M, M / 2 - 1)
    bound = {(1, "cubic"): 0.03, (2, "cubic"): 0.004, (1, "linear"): 0.12, (2, "linear"): 0.04}
    for s in (1, 2):
        box = s * M
        gg = np.arange(box) - box // 2
        Z, Y, X = np.meshgrid(gg, gg, gg, indexing="ij")
        d = a * np.exp(-((X - c3[0]) ** 2 + (Y - c3[1]) ** 2 + (Z - c3[2]) ** 2) / (2 * sigma ** 2))
        V = np.fft.rfftn(np.fft.ifftshift(d))[None]
        for interp in ("linear", "cubic"):
            out = oracle.project(3, V, R[None], shift=t[None], N=M, interp=interp,
                                 oversampling=s, radius=M / 2 - 1)
            for pi in range(2):
                cr = R[pi] @ c3                                 # rotated centre
                for sign, ok in ((1, True), (-1, False)):       # shifted by +t (not -t)
                    cx, cy = cr[0] + sign * t[pi, 0], cr[1] + sign * t[pi, 1]
                    img = a * np.sqrt(2 * np.pi) * sigma * np.exp(
                        -((X2 - cx) ** 2 + (Y2 - cy) ** 2) / (2 * sigma ** 2))
                    ref = np.fft.rfft2(np.fft.ifftshift(img))
                    err = np.linalg.norm(out[0, pi][mask] - ref[mask]) / np.linalg.norm(ref[mask])
                    if ok:
                        assert err < bound[(s, interp)], (s, interp, err)
                    else:
                        assert err > 0.5


# P5: adjoint identity Re<P x, y> = Re<x, P^T y> on non-Hermitian data.
@pytest.mark.parametrize("dim", [2, 3])
@pytest.mark.parametrize("interp", ["linear", "cubic"])
@pytest.mark.parametrize("s,M,N,radius,shifted", [
    (1.0, 16, 16, -1.0, False), (2.0, 32, 16, 6.5, True), (0.75, 12, 16, -1.0, True),
    (1.3, 18, 14, 5.0, True),
])
def test_adjoint_identity(dim, interp, s, M, N, radius, shifted):
    rng = np.random.default_rng(9)
    B, P = 2, 3
    shp = (1, M, M, M // 2 + 1) if dim == 3 else (1, M, M // 2 + 1)
    x = crandn(rng, shp)
    R = (synth.random_rotations(B * P, rng).reshape(B, P, 3, 3) if dim == 3 else
         synth.planar_rotations(rng.uniform(0, 2 * np.pi, B * P)).reshape(B, P, 2, 2)).astype(np.float64)
    t = rng.uniform(-4, 4, (B, P, 2)) if shifted else None
    y = crandn(rng, (B, P, N, N // 2 + 1))
    Px = oracle.project(dim, x, R, shift=t, N=N, interp=interp, oversampling=s, radius=radius)
    PTy, _ = oracle.backproject(dim, y, R, shift=t, M=M, interp=interp, oversampling=s,
                                radius=radius, Bdst=1, want_weights=False)
    lhs = np.vdot(Px, y).real
    rhs = np.vdot(x, PTy).real
    assert abs(lhs - rhs) <= 1e-12 * max(abs(lhs), 1.0) * 10


# P6: finite differences of L = Re<g, P(V; R, t)> for rotation and shift gradients.
@pytest.mark.parametrize("dim", [2, 3])
@pytest.mark.parametrize("interp", ["linear", "cubic"])
@pytest.mark.parametrize("s,M", [(1.0, 16), (1.5, 24)])
def test_finite_difference_gradients(dim, interp, s, M):
    rng = np.random.default_rng(10)
    N = 16
    shp = (1, M, M, M // 2 + 1) if dim == 3 else (1, M, M // 2 + 1)
    V = crandn(rng, shp)
    P = 2
    R = (synth.random_rotations(P, rng)[None] if dim == 3 else
         synth.planar_rotations(rng.uniform(0, 2 * np.pi, P))[None]).astype(np.float64)
    t = rng.uniform(-3, 3, (1, P, 2))
    g = crandn(rng, (1, P, N, N // 2 + 1))

    def loss(V_, R_, t_):
        return np.vdot(g, oracle.project(dim, V_, R_, shift=t_, N=N, interp=interp,
                                         oversampling=s, radius=7.0)).real

    gV, gR, gt = oracle.project_backward(dim, g, V, R, shift=t, interp=interp, oversampling=s,
                                         radius=7.0)
    h = 1e-6 if interp == "cubic" else 1e-7
    for idx in itertools.product(range(P), range(dim), range(dim)):
        Rp, Rm = R.copy(), R.copy()
        Rp[(0,) + idx] += h
        Rm[(0,) + idx] -= h
        fd = (loss(V, Rp, t) - loss(V, Rm, t)) / (2 * h)
        assert abs(fd - gR[(0,) + idx]) <= 1e-6 * (abs(fd) + np.abs(gR).max()), (idx, fd, gR[(0,) + idx])
    for idx in itertools.product(range(P), range(2)):
        tp, tm = t.copy(), t.copy()
        tp[(0,) + idx] += h
        tm[(0,) + idx] -= h
        fd = (loss(V, R, tp) - loss(V, R, tm)) / (2 * h)
        assert abs(fd - gt[(0,) + idx]) <= 1e-6 * (abs(fd) + np.abs(gt).max())
    # volume entries (the map is linear in V, so the difference is exact up to rounding)
    for _ in range(6):
        e = tuple(rng.integers(0, n) for n in V.shape)
        for comp, dv in ((0, 1.0), (1, 1j)):
            Vp, Vm = V.copy(), V.copy()
            Vp[e] += dv
            Vm[e] -= dv
            fd = (loss(Vp, R, t) - loss(Vm, R, t)) / 2
            want = gV[e].real if comp == 0 else gV[e].imag
            assert abs(fd - want) <= 1e-10 * (1 + abs(fd))
    if dim == 3:
        assert np.all(gR[..., 2, :] == 0)      # P12: k_z = 0 gives no gradient in row 3


# P7: integer shifts roll the real-space image.
def test_integer_shift_rolls_image():
    rng = np.random.default_rng(11)
    N = 16
    img = rng.standard_normal((N, N))
    F = np.fft.rfft2(img)[None]
    for sx, sy in ((1, 0), (0, 2), (-3, 5), (7, -4)):
        out = oracle.project(2, F, np.eye(2)[None, None], shift=np.array([[[sx, sy]]], float),
                             interp="cubic", radius=float(N))
        back = np.fft.irfft2(out[0, 0], s=(N, N))
        np.testing.assert_allclose(back, np.roll(img, (sy, sx), axis=(0, 1)), atol=1e-12)


# P8: real data project to spectra whose kx = 0 column is Hermitian.
def test_hermitian_input_gives_hermitian_column():
    rng = np.random.default_rng(12)
    M = N = 24
    d = rng.standard_normal((M, M, M))
    V = np.fft.rfftn(d)[None]
    R = synth.random_rotations(4, rng).astype(np.float64)[None]
    t = rng.uniform(-5, 5, (1, 4, 2))
    for interp in ("linear", "cubic"):
        out = oracle.project(3, V, R, shift=t, N=N, interp=interp, radius=N / 2 - 3)
        col = out[0, :, :, 0]
        mirrored = np.conj(col[:, (-np.arange(N)) % N])
        np.testing.assert_allclose(col, mirrored, atol=1e-12 * np.abs(col).max())


# P9: the radius cutoff.
def test_radius_cutoff_forward_and_adjoint():
    rng = np.random.default_rng(13)
    M = N = 16
    r = 5.0
    V = crandn(rng, (1, M, M, M // 2 + 1))
    R = synth.random_rotations(3, rng).astype(np.float64)[None]
    out = oracle.project(3, V, R, N=N, interp="cubic", radius=r)
    mask = in_radius(N, r)
    assert np.all(out[0][:, ~mask] == 0) and np.all(np.abs(out[0][:, mask]) > 0)
    y = crandn(rng, (1, 3, N, N // 2 + 1)) * (~mask)
    om = rng.uniform(0.5, 2.0, y.shape) * (~mask)
    data, wt = oracle.backproject(3, y, R, M=M, interp="cubic", radius=r, weights=om)
    assert np.all(data == 0) and np.all(wt == 0)
    _, wt1 = oracle.backproject(3, y, R, M=M, interp="cubic", radius=r)
    assert abs(wt1.sum() - 3 * mask.sum()) < 1e-9


# P10: one identity-pose backprojection writes the image into the z = 0 plane.
@pytest.mark.parametrize("interp", ["linear", "cubic"])
def test_identity_backprojection(interp):
    rng = np.random.default_rng(14)
    M = N = 16
    img = crandn(rng, (1, 1, N, N // 2 + 1))
    data, wt = oracle.backproject(3, img, np.eye(3)[None, None], M=M, interp=interp)
    mask = in_radius(N, N / 2)
    np.testing.assert_array_equal(data[0, 0], np.where(mask, img[0, 0], 0))
    np.testing.assert_array_equal(wt[0, 0], mask.astype(float))
    assert np.all(data[0, 1:] == 0) and np.all(wt[0, 1:] == 0)


def test_weight_volume_partition_of_unity():
    """With omega = 1 every in-radius sample deposits total weight 1 (taps in range)."""
    rng = np.random.default_rng(15)
    M = N = 32
    r = N / 2 - 3
    R = synth.random_rotations(5, rng).astype(np.float64)[None]
    y = crandn(rng, (1, 5, N, N // 2 + 1))
    om = rng.uniform(0.5, 2.0, y.shape)
    for interp in ("linear", "cubic"):
        _, wt = oracle.backproject(3, y, R, M=M, interp=interp, radius=r)
        assert abs(wt.sum() - 5 * in_radius(N, r).sum()) < 1e-9
        _, wt = oracle.backproject(3, y, R, M=M, interp=interp, radius=r, weights=om)
        assert abs(wt.sum() - (om[0][:, in_radius(N, r)]).sum()) < 1e-9


# P11: rotating by theta and back is close to the identity; cubic beats linear.
def test_rotate_back_and_forth_2d():
    rng = synth.streams(16, 2)
    N = 64
    img = synth.blob_images(1, N, 8, rng[0]).astype(np.complex128)
    r = N / 2 - 4
    mask = in_radius(N, r)
    errs = {}
    for interp in ("linear", "cubic"):
        e = []
        for th in (0.3, 1.1, 2.5):
            a = oracle.project(2, img, synth.planar_rotations(np.array([th]))[None].astype(float),
                               interp=interp, radius=r)[0]
            b = oracle.project(2, a, synth.planar_rotations(np.array([-th]))[None].astype(float),
                               interp=interp, radius=r)[0, 0]
            e.append(np.linalg.norm(b[mask] - img[0][mask]) / np.linalg.norm(img[0][mask]))
        errs[interp] = max(e)
    assert errs["cubic"] < errs["linear"] and errs["cubic"] < 0.05


def test_batch_broadcast_matches_separate_calls():
    rng = np.random.default_rng(17)
    M = N = 16
    V = crandn(rng, (2, M, M, M // 2 + 1))
    R = synth.random_rotations(3, rng).astype(np.float64)[None]
    t = rng.uniform(-2, 2, (2, 3, 2))
    out = oracle.project(3, V, R, shift=t, interp="cubic")
    for b in range(2):
        np.testing.assert_array_equal(out[b], oracle.project(3, V[b:b + 1], R, shift=t[b:b + 1],
                                                             interp="cubic")[0])
    g = crandn(rng, out.shape)
    gV, gR, gt = oracle.project_backward(3, g, V, R, shift=t, interp="cubic")
    acc = np.zeros_like(gR)
    for b in range(2):
        _, gRb, _ = oracle.project_backward(3, g[b:b + 1], V[b:b + 1], R, shift=t[b:b + 1],
                                            interp="cubic")
        acc += gRb
    np.testing.assert_allclose(gR, acc, rtol=1e-12, atol=1e-12)


# P16: gradients of the backprojection (data and weight spectra) against
# finite differences of backproject() itself, for
#   L = Re<G, data(y, w; R, t)> + <GW, weight(y, w; R, t)>.
@pytest.mark.parametrize("interp", ["linear", "cubic"])
@pytest.mark.parametrize("with_weights", [False, True])
def test_backprojection_gradients_finite_differences(interp, with_weights):
    rng = np.random.default_rng(16)
    M, N, P = 18, 16, 2
    s, r = 1.2, 7.0
    y = crandn(rng, (2, P, N, N // 2 + 1))
    om = rng.uniform(0.5, 1.5, y.shape) if with_weights else None
    R = synth.random_rotations(P, rng).astype(np.float64)[None]          # broadcast over B = 2
    t = rng.uniform(-3, 3, (2, P, 2))
    G = crandn(rng, (1, M, M, M // 2 + 1))
    GW = rng.standard_normal((1, M, M, M // 2 + 1))
    kw = dict(interp=interp, oversampling=s, radius=r)

    def loss(y_, om_, R_, t_):
        data, wt = oracle.backproject(3, y_, R_, shift=t_, M=M, weights=om_, **kw)
        return np.vdot(G, data).real + np.sum(GW * wt)

    gy, gw, gR, gt = oracle.backproject_backward(3, G, y, R, shift=t, grad_weight=GW, weights=om,
                                                 **kw)
    h = 1e-6 if interp == "cubic" else 1e-7
    for idx in itertools.product(range(P), range(3), range(3)):
        Rp, Rm = R.copy(), R.copy()
        Rp[(0,) + idx] += h
        Rm[(0,) + idx] -= h
        fd = (loss(y, om, Rp, t) - loss(y, om, Rm, t)) / (2 * h)
        assert abs(fd - gR[(0,) + idx]) <= 1e-6 * (abs(fd) + np.abs(gR).max()), (idx, fd)
    for idx in itertools.product(range(2), range(P), range(2)):
        tp, tm = t.copy(), t.copy()
        tp[idx] += h
        tm[idx] -= h
        fd = (loss(y, om, R, tp) - loss(y, om, R, tm)) / (2 * h)
        assert abs(fd - gt[idx]) <= 1e-6 * (abs(fd) + np.abs(gt).max()), (idx, fd)
    # The map is linear in the images and in the weights: unit differences are exact.
    for _ in range(6):
        e = tuple(rng.integers(0, n) for n in y.shape)
        for dv in (1.0, 1j):
            yp, ym = y.copy(), y.copy()
            yp[e] += dv
            ym[e] -= dv
            fd = (loss(yp, om, R, t) - loss(ym, om, R, t)) / 2
            want = gy[e].real if dv == 1.0 else gy[e].imag
            assert abs(fd - want) <= 1e-10 * (1 + abs(fd))
        if with_weights:
            op, omm = om.copy(), om.copy()
            op[e] += 1.0
            omm[e] -= 1.0
            fd = (loss(y, op, R, t) - loss(y, omm, R, t)) / 2
            assert abs(fd - gw[e]) <= 1e-10 * (1 + abs(fd))
    if not with_weights:
        # The weight spectrum with unit image weights still depends on the poses.
        gy1, gw1, gR1, _ = oracle.backproject_backward(3, G, y, R, shift=t, grad_weight=GW, **kw)
        assert gw1.shape == y.shape


# --------------------------------------------------------------------------
# P17: the symmetrised zero-frequency axis (the optional backward-pass
# treatment of [ar §2] / [de §2 "Friedel-Symmetrie"]): fixed on spectra of
# real data, closed forms for a lone coefficient, an orthogonal projector.
import hermitian_pins  # noqa: E402


@pytest.mark.parametrize("check", hermitian_pins.ALL, ids=lambda f: f.__name__)
def test_hermitian_x0(check):
    check(oracle.hermitian_x0)


def test_hermitian_x0_keeps_the_adjoint_identity_for_real_objects():
    """With the axis symmetrised after the backprojection B, Re<F V, y> =
    Re<V, H(B y)> still holds for every spectrum V of a real object (H
    fixes V and is self-adjoint), but not for a general V."""
    rng = np.random.default_rng(172)
    M = N = 12
    R = synth.random_rotations(3, rng).astype(np.float64)[None]
    t = rng.uniform(-2, 2, (1, 3, 2))
    y = hermitian_pins.crandn(rng, (1, 3, N, N // 2 + 1))
    kw = dict(interp="cubic", radius=-1.0)
    Hb, _ = oracle.hermitian_x0(oracle.backproject(3, y, R, shift=t, M=M, **kw)[0], 3)
    V = np.fft.rfftn(rng.standard_normal((M, M, M)))[None]
    lhs = np.vdot(y, oracle.project(3, V, R, shift=t, N=N, **kw)).real
    assert abs(lhs - np.vdot(Hb, V).real) <= 1e-10 * abs(lhs)
    G = hermitian_pins.crandn(rng, V.shape)
    lhs = np.vdot(y, oracle.project(3, G, R, shift=t, N=N, **kw)).real
    assert abs(lhs - np.vdot(Hb, G).real) > 1e-6 * abs(lhs)
