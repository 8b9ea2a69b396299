"""Seeded synthetic inputs shared by the oracle checks, the GPU tests and the bench.

This module draws inputs only: Gaussian-blob densities and their centred
real FFTs, uniform rotations, shifts and noise.  It holds none of the
projection arithmetic, so the oracle and the CUDA path stay independent.

Recipe (one ``numpy.random.default_rng`` per component, spawned from
``SeedSequence(seed)``):
  - blob densities: centres uniform in a ball of radius box/4 about the box
    centre (index box/2), sigma ~ U(1, 3) px, amplitude ~ U(0.5, 1); the
    density is sampled at integer pixel positions;
  - spectra: ``rfftn(ifftshift(density))`` in float64, cast to complex64, so
    rotations act about the box centre;
  - rotations: unit quaternions from a normalised 4D standard normal (uniform
    on SO(3)), converted to matrices; in-plane angles ~ U(0, 2 pi);
  - shifts ~ U(-lim, lim)^2 in pixels;
  - noise spectra: iid complex normal with E|z|^2 = 1 scaled by 1/(1+|k|).
"""
from __future__ import annotations

import numpy as np

# Workloads: the five configurations measured and tested by this project.
CONFIGS = {
    1: dict(name="proj3d-box32-linear-8poses", box=32, blobs=20, poses=8, interp="linear",
            oversampling=1.0, radius=16.0),
    2: dict(name="rot2d-box128-cubic-1024img", box=128, blobs=10, images=1024, interp="cubic",
            shift_lim=5.0, radius=64.0),
    3: dict(name="proj3d-box128-cubic-4096poses", box=128, blobs=200, poses=4096, interp="cubic",
            radius=64.0),
    4: dict(name="backproj-box256-2048img", box=256, images=2048, radius=128.0),
    5: dict(name="fwdbwd-box256-cubic-512poses", box=256, blobs=1000, poses=512, interp="cubic",
            shift_lim=10.0, radius=128.0),
}


def streams(seed: int, n: int):
    """n independent generators spawned from one seed."""
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]


def blob_params(box: int, n_blobs: int, rng, dim: int = 3):
    """Centres (n, dim) in pixel coordinates (x, y[, z]), sigmas (n,), amplitudes (n,)."""
    d = rng.standard_normal((n_blobs, dim))
    d /= np.linalg.norm(d, axis=1, keepdims=True)
    rad = (box / 4.0) * rng.random(n_blobs) ** (1.0 / dim)
    centres = box / 2.0 + d * rad[:, None]
    sigmas = rng.uniform(1.0, 3.0, n_blobs)
    amps = rng.uniform(0.5, 1.0, n_blobs)
    return centres, sigmas, amps


def blob_density(box: int, centres, sigmas, amps, dim: int = 3):
    """Sum of Gaussians sampled on the integer grid; array indexed [z][y][x] (or [y][x]).

    Each blob is evaluated within +-6 sigma of its centre (exp(-18) ~ 1.5e-8
    of its amplitude is dropped beyond), which keeps box-256 volumes cheap.
    """
    out = np.zeros((box,) * dim, np.float64)
    for c, s, a in zip(centres, sigmas, amps):
        lo = [max(0, int(np.floor(c[j] - 6.0 * s))) for j in range(dim)]
        hi = [min(box, int(np.ceil(c[j] + 6.0 * s)) + 1) for j in range(dim)]
        g = [np.exp(-((np.arange(lo[j], hi[j]) - c[j]) ** 2) / (2.0 * s * s)) for j in range(dim)]
        if dim == 3:
            out[lo[2]:hi[2], lo[1]:hi[1], lo[0]:hi[0]] += (
                a * g[2][:, None, None] * g[1][None, :, None] * g[0][None, None, :])
        else:
            out[lo[1]:hi[1], lo[0]:hi[0]] += a * g[1][:, None] * g[0][None, :]
    return out


def centred_rfft(density):
    """Half spectrum of a density whose centre is at index box/2 on every axis."""
    axes = tuple(range(-density.ndim, 0))
    return np.fft.rfftn(np.fft.ifftshift(density, axes=axes), axes=axes)


def random_rotations(n: int, rng):
    """(n, 3, 3) float32 rotation matrices, uniform on SO(3)."""
    q = rng.standard_normal((n, 4))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    w, x, y, z = q.T
    R = np.stack([
        1 - 2 * (y * y + z * z), 2 * (x * y - z * w), 2 * (x * z + y * w),
        2 * (x * y + z * w), 1 - 2 * (x * x + z * z), 2 * (y * z - x * w),
        2 * (x * z - y * w), 2 * (y * z + x * w), 1 - 2 * (x * x + y * y),
    ], axis=1).reshape(n, 3, 3)
    return R.astype(np.float32)


def planar_rotations(angles):
    """(n, 2, 2) float32 matrices [[cos, -sin], [sin, cos]]."""
    c, s = np.cos(angles), np.sin(angles)
    return np.stack([c, -s, s, c], axis=1).reshape(-1, 2, 2).astype(np.float32)


def uniform_shifts(n: int, lim: float, rng):
    return rng.uniform(-lim, lim, (n, 2)).astype(np.float32)


def complex_normal(shape, rng):
    """iid complex normal, E|z|^2 = 1, complex64."""
    z = rng.standard_normal(shape + (2,)) * np.sqrt(0.5)
    return (z[..., 0] + 1j * z[..., 1]).astype(np.complex64)


def spectral_falloff(N: int):
    """1/(1+|k|) over an (N, N/2+1) half-spectrum (rows in fftfreq order)."""
    ky = np.fft.fftfreq(N, 1.0 / N)[:, None]
    kx = np.arange(N // 2 + 1)[None, :]
    return 1.0 / (1.0 + np.sqrt(kx * kx + ky * ky))


def noise_images(B: int, P: int, N: int, rng):
    """(B, P, N, N/2+1) complex64 Gaussian spectra scaled by 1/(1+|k|)."""
    return (complex_normal((B, P, N, N // 2 + 1), rng) * spectral_falloff(N)).astype(np.complex64)


def blob_volume(box: int, n_blobs: int, rng):
    """(1, box, box, box/2+1) complex64 spectrum of a blob density."""
    c, s, a = blob_params(box, n_blobs, rng, 3)
    return centred_rfft(blob_density(box, c, s, a, 3)).astype(np.complex64)[None]


def padded_blob_volume(box: int, n_blobs: int, rng, factor: int = 2):
    """(1, f*box, f*box, f*box/2+1) spectrum of the same blob density zero-padded
    in real space to f times the box (draws exactly what blob_volume draws)."""
    c, s, a = blob_params(box, n_blobs, rng, 3)
    d = blob_density(box, c, s, a, 3)
    big = factor * box
    o = big // 2 - box // 2
    dp = np.zeros((big,) * 3, np.float64)
    dp[o:o + box, o:o + box, o:o + box] = d
    return centred_rfft(dp).astype(np.complex64)[None]


def blob_images(n: int, box: int, n_blobs: int, rng):
    """(n, box, box/2+1) complex64 spectra of 2D blob images (one rng draw per image)."""
    out = np.empty((n, box, box // 2 + 1), np.complex64)
    for i in range(n):
        c, s, a = blob_params(box, n_blobs, rng, 2)
        out[i] = centred_rfft(blob_density(box, c, s, a, 2))
    return out


def workload(cfg: int, *, poses: int | None = None, seed: int | None = None,
             oversampling: int = 1):
    """Inputs of configuration cfg as numpy arrays (seed 1000 + cfg by default).

    ``poses`` truncates the pose / image count.  Every per-pose draw is made
    in C order with the pose axis leading, so a truncated workload is exactly
    the leading prefix of the full one.
    Keys: name, box, radius, interp, oversampling, P, rot, shift (or None),
    and vol (cfg 1, 3, 5), img (cfg 2) or proj (cfg 4); grad is a seeded
    upstream gradient for the backward checks.  For cfg 3, ``oversampling=2``
    returns the same blob density zero-padded to twice the box (the volume the
    operator then samples at p = 2 R^T k).
    """
    c = CONFIGS[cfg]
    seed = 1000 + cfg if seed is None else seed
    r_vol, r_rot, r_shift, r_img, r_grad = streams(seed, 5)
    box = c["box"]
    out = dict(cfg=cfg, name=c["name"], box=box, radius=c["radius"], oversampling=1.0)
    if cfg in (1, 3, 5):
        P = c["poses"] if poses is None else int(poses)
        vol = (padded_blob_volume(box, c["blobs"], r_vol, oversampling) if oversampling > 1
               else blob_volume(box, c["blobs"], r_vol))
        out.update(vol=vol, rot=random_rotations(P, r_rot)[None], oversampling=float(oversampling),
                   interp=c["interp"], P=P,
                   shift=(uniform_shifts(P, c["shift_lim"], r_shift)[None] if "shift_lim" in c else None),
                   grad=noise_images(1, P, box, r_grad))
    elif cfg == 2:
        n = c["images"] if poses is None else int(poses)
        ang = r_rot.uniform(0.0, 2.0 * np.pi, n)
        out.update(img=blob_images(n, box, c["blobs"], r_img), angles=ang.astype(np.float32),
                   rot=planar_rotations(ang)[:, None], P=1, interp=c["interp"],
                   shift=uniform_shifts(n, c["shift_lim"], r_shift)[:, None],
                   grad=noise_images(n, 1, box, r_grad))
    elif cfg == 4:
        n = c["images"] if poses is None else int(poses)
        out.update(proj=noise_images(1, n, box, r_img), rot=random_rotations(n, r_rot)[None],
                   shift=None, P=n)
    return out
