"""Checks that pin the symmetrised zero-frequency axis (oracle.hermitian_x0).

Each check takes the implementation h(spec, dim, weight=None) -> (spec',
weight') as an argument, so that the pin suite (test_oracle_pins.py) runs
them on the oracle and the mutation suite (test_oracle_mutations.py) runs
them on copies of it with a planted mistake.  None of them restates the
formula: they test it against numpy's FFT of real data, closed forms for a
lone coefficient, and the algebra of an orthogonal projector.
"""
import numpy as np


def crandn(rng, shape):
    return rng.standard_normal(shape) + 1j * rng.standard_normal(shape)


def check_real_object_is_fixed(h):
    """The half-spectrum of real data is already Hermitian on kx = 0: unchanged."""
    rng = np.random.default_rng(170)
    for dim, M in ((3, 8), (3, 10), (2, 12), (2, 6)):
        x = rng.standard_normal((2,) + (M,) * dim)
        V = np.fft.rfftn(x, axes=tuple(range(1, dim + 1)))
        got, _ = h(V, dim)
        np.testing.assert_allclose(got, V, rtol=0, atol=1e-12 * np.abs(V).max())


def check_lone_coefficient(h):
    """A lone coefficient c at (0, k) becomes c/2 at k and conj(c)/2 at -k
    (rows taken modulo the box); at a self-conjugate k it becomes Re c.
    The weight spectrum splits w into w/2 at k and -k likewise."""
    M = 6
    c = 2.0 + 4.0j
    # 3D: (z, y) = (1, 4) pairs with (5, 2)
    V = np.zeros((1, M, M, M // 2 + 1), complex)
    V[0, 1, 4, 0] = c
    W = np.zeros(V.shape)
    W[0, 1, 4, 0] = 3.0
    got, gw = h(V, 3, W)
    want = np.zeros_like(V)
    want[0, 1, 4, 0] = c / 2
    want[0, 5, 2, 0] = np.conj(c) / 2
    np.testing.assert_allclose(got, want, atol=1e-15)
    wantw = np.zeros(W.shape)
    wantw[0, 1, 4, 0] = wantw[0, 5, 2, 0] = 1.5
    np.testing.assert_allclose(gw, wantw, atol=1e-15)
    # self-conjugate points of the plane: (z, y) with both rows in {0, M/2}
    for z, y in ((0, 0), (0, M // 2), (M // 2, 0), (M // 2, M // 2)):
        V = np.zeros((1, M, M, M // 2 + 1), complex)
        V[0, z, y, 0] = c
        got, _ = h(V, 3)
        want = np.zeros_like(V)
        want[0, z, y, 0] = c.real
        np.testing.assert_allclose(got, want, atol=1e-15)
    # 2D: row 1 pairs with row 5; row 3 (= -3 mod 6) is self-conjugate
    V = np.zeros((1, M, M // 2 + 1), complex)
    V[0, 1, 0] = c
    V[0, 3, 0] = c
    got, _ = h(V, 2)
    want = np.zeros_like(V)
    want[0, 1, 0] = c / 2
    want[0, 5, 0] = np.conj(c) / 2
    want[0, 3, 0] = c.real
    np.testing.assert_allclose(got, want, atol=1e-15)


def check_projector(h):
    """Only the kx = 0 plane changes, applying h twice equals applying it
    once, and h is self-adjoint for the real inner products Re<a, b> and
    <u, v>: an orthogonal projector."""
    rng = np.random.default_rng(171)
    for dim, M in ((3, 8), (2, 10)):
        shape = (2,) + (M,) * (dim - 1) + (M // 2 + 1,)
        a, b = crandn(rng, shape), crandn(rng, shape)
        u, v = rng.standard_normal(shape), rng.standard_normal(shape)
        pa, pu = h(a, dim, u)
        pb, pv = h(b, dim, v)
        np.testing.assert_array_equal(pa[..., 1:], a[..., 1:])
        np.testing.assert_array_equal(pu[..., 1:], u[..., 1:])
        assert np.abs(pa[..., 0] - a[..., 0]).max() > 1e-3       # it does act on the plane
        ppa, ppu = h(pa, dim, pu)
        np.testing.assert_allclose(ppa, pa, atol=1e-14)
        np.testing.assert_allclose(ppu, pu, atol=1e-14)
        lhs = np.vdot(pa, b).real
        rhs = np.vdot(a, pb).real
        assert abs(lhs - rhs) <= 1e-12 * np.abs(a).sum()
        assert abs(np.vdot(pu, v) - np.vdot(u, pv)) <= 1e-12 * np.abs(u).sum()


ALL = (check_real_object_is_fixed, check_lone_coefficient, check_projector)
