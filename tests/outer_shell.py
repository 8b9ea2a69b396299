"""Inputs of the outer-shell golden cases (tests/golden/outer_shell_taps.json).

Each case places a few entries in an otherwise zero box-M half-spectrum and
asks for the interpolated value at one sample position p.  The projection
operators reach a chosen p through output pixel (kx, ky) = (1, 0): its sample
position is p = s R^T k = R[0][:] for s = 1, and any matrix is accepted, so
R's first row is p and the other rows are those of the identity.  This
module only builds arrays; the expected values are the fixture's, worked out
by hand.
"""
import json
import os

import numpy as np

FIXTURE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "outer_shell_taps.json")
PIXEL = (0, 1)   # (iy, ix) of output pixel (kx, ky) = (1, 0)


def cases():
    """(name, dim, M, spectrum (1, ...) complex128, rot (1, 1, d, d), expected complex)."""
    with open(FIXTURE) as f:
        fx = json.load(f)
    M = fx["M"]
    out = []
    for c in fx["cases"]:
        dim = c["dim"]
        shape = (1, M, M // 2 + 1) if dim == 2 else (1, M, M, M // 2 + 1)
        V = np.zeros(shape, np.complex128)
        for e in c["entries"]:
            n, (re, im) = e[:dim], e[dim:]
            idx = (0,) + tuple(k % M for k in reversed(n[1:])) + (n[0],)
            V[idx] += re + 1j * im
        R = np.eye(dim)
        R[0] = c["p"]
        out.append((c["name"], dim, M, V, R[None, None], complex(*c["expect"])))
    return out
