"""float64 CPU oracle for the projection operators (test infrastructure).

This package is a checker, not part of the product: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  The arithmetic lives in ``tp_oracle.c`` (plain C, OpenMP); this
module compiles it with gcc on first use and marshals numpy arrays.

All inputs are up-cast to float64 / complex128 before the call, so the oracle
sees the same values as the CUDA path and evaluates them in double precision.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tp_oracle.c")
_LIB = os.path.join(_HERE, "libtp_oracle.so")
_lock = threading.Lock()
_lib = None

LINEAR, CUBIC = 0, 1


def build(force: bool = False) -> str:
    """Compile tp_oracle.c into libtp_oracle.so next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-Wall",
             "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # TP_ORACLE_LIB lets the oracle's own mutation test load a
            # deliberately broken build; nothing else sets it.
            lib = ctypes.CDLL(os.environ.get("TP_ORACLE_LIB") or build())
            d, i, p = ctypes.c_double, ctypes.c_int, ctypes.c_void_p
            lib.oracle_project.argtypes = [i, p, i, i, p, i, i, p, i, i, i, d, d, p]
            lib.oracle_backproject.argtypes = [i, p, p, i, i, i, p, i, p, i, i, i, i, d, d, p, p]
            lib.oracle_project_backward.argtypes = [i, p, p, i, i, p, i, i, p, i, i, i, d, d, p, p, p]
            for f in (lib.oracle_project, lib.oracle_backproject, lib.oracle_project_backward):
                f.restype = ctypes.c_int
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [i]
            lib.oracle_set_num_threads.restype = None
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """OpenMP threads for the oracle's later calls (for single-thread timing)."""
    _load().oracle_set_num_threads(int(n))


def _c(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _interp(interp):
    if interp in ("linear", LINEAR):
        return LINEAR
    if interp in ("cubic", CUBIC):
        return CUBIC
    raise ValueError(f"unknown interpolation {interp!r}")


def _batch(*bs):
    B = max(bs)
    for b in bs:
        if b not in (1, B):
            raise ValueError(f"batch sizes {bs} do not broadcast")
    return B


def _check(rc):
    if rc != 0:
        raise ValueError("oracle rejected the arguments")


def project(dim, src, rot, shift=None, N=None, interp="linear", oversampling=1.0, radius=-1.0):
    """Forward projection of a (Bsrc, M[, M], M, M/2+1) spectrum.

    dim=3: 3D->2D central slices; dim=2: 2D->2D rotation.  rot is
    (Bp, P, dim, dim), shift (Bs, P, 2) or None.  Returns (B, P, N, N/2+1)
    complex128.
    """
    src = _c(src, np.complex128)
    rot = _c(rot, np.float64)
    shift = _c(shift, np.float64)
    Bsrc, M = src.shape[0], src.shape[1]
    Bp, P = rot.shape[0], rot.shape[1]
    Bs = shift.shape[0] if shift is not None else 1
    N = M if N is None else int(N)
    B = _batch(Bsrc, Bp, Bs)
    out = np.zeros((B, P, N, N // 2 + 1), np.complex128)
    _check(_load().oracle_project(dim, _ptr(src), Bsrc, M, _ptr(rot), Bp, P, _ptr(shift), Bs,
                                  N, _interp(interp), float(oversampling), float(radius), _ptr(out)))
    return out


def backproject(dim, img, rot, shift=None, M=None, weights=None, interp="linear",
                oversampling=1.0, radius=-1.0, Bdst=1, want_weights=True):
    """Adjoint of project(): scatter (B, P, N, N/2+1) images into a spectrum.

    Returns (data, weight) with shapes (Bdst, M[, M], M, M/2+1); weight is
    None when want_weights is False.
    """
    img = _c(img, np.complex128)
    rot = _c(rot, np.float64)
    shift = _c(shift, np.float64)
    weights = _c(weights, np.float64)
    B, P, N = img.shape[0], img.shape[1], img.shape[2]
    M = N if M is None else int(M)
    Bp = rot.shape[0]
    Bs = shift.shape[0] if shift is not None else 1
    X = M // 2 + 1
    shp = (Bdst, M, M, X) if dim == 3 else (Bdst, M, X)
    data = np.zeros(shp, np.complex128)
    wt = np.zeros(shp, np.float64) if want_weights else None
    _check(_load().oracle_backproject(dim, _ptr(img), _ptr(weights), B, P, N, _ptr(rot), Bp,
                                      _ptr(shift), Bs, Bdst, M, _interp(interp),
                                      float(oversampling), float(radius), _ptr(data), _ptr(wt)))
    return data, wt


def project_backward(dim, grad_out, src, rot, shift=None, interp="linear", oversampling=1.0,
                     radius=-1.0, need_src=True, need_rot=True, need_shift=True):
    """Gradients through project() for upstream grad_out (B, P, N, N/2+1).

    Returns (grad_src, grad_rot, grad_shift); entries not requested (or
    grad_shift without a shift) are None.
    """
    grad_out = _c(grad_out, np.complex128)
    src = _c(src, np.complex128)
    rot = _c(rot, np.float64)
    shift = _c(shift, np.float64)
    B, P, N = grad_out.shape[0], grad_out.shape[1], grad_out.shape[2]
    Bsrc, M = src.shape[0], src.shape[1]
    Bp = rot.shape[0]
    Bs = shift.shape[0] if shift is not None else 1
    gsrc = np.zeros_like(src) if need_src else None
    grot = np.zeros_like(rot) if need_rot else None
    gshift = np.zeros_like(shift) if (need_shift and shift is not None) else None
    _check(_load().oracle_project_backward(dim, _ptr(grad_out), _ptr(src), Bsrc, M, _ptr(rot), Bp, P,
                                           _ptr(shift), Bs, N, _interp(interp),
                                           float(oversampling), float(radius),
                                           _ptr(gsrc), _ptr(grot), _ptr(gshift)))
    return gsrc, grot, gshift


def backproject_backward(dim, grad_data, img, rot, shift=None, grad_weight=None, weights=None,
                         interp="linear", oversampling=1.0, radius=-1.0):
    """Gradients of backproject() for upstream gradients of its two spectra.

    backproject() is the real adjoint of project() (data: taps w times
    conj(phase) times the image; weights: taps w times the image weights,
    no phase).  With grad_data (complex) and grad_weight (real, or None) the
    upstream gradients of the data and weight spectra:
      grad_img     = project(grad_data)                 (adjoint of the adjoint)
      grad_weights = Re project(grad_weight), no shift  (None without grad_weight)
      grad_rot     = project()'s rotation gradient at spectrum grad_data for
                     upstream img, plus, with grad_weight, that at spectrum
                     grad_weight without shift for upstream weights (or 1)
      grad_shift   = project()'s shift gradient at spectrum grad_data for
                     upstream img (None without shift)
    The tests pin this against finite differences of backproject() itself.
    Returns (grad_img, grad_weights, grad_rot, grad_shift).
    """
    img = _c(img, np.complex128)
    B, N = img.shape[0], img.shape[2]
    kw = dict(interp=interp, oversampling=oversampling, radius=radius)

    def upstream(a, *operands):
        # project()'s batch is that of its operands; when they are all
        # shared by the B images, the gradients (linear in the upstream)
        # take the upstream summed over the images.
        nb = max(o.shape[0] for o in operands if o is not None)
        return a.sum(axis=0, keepdims=True) if nb < a.shape[0] else a

    rot_ = _c(rot, np.float64)
    shift_ = _c(shift, np.float64)
    gd = _c(grad_data, np.complex128)
    grad_img = np.broadcast_to(project(dim, gd, rot_, shift=shift_, N=N, **kw),
                               img.shape).copy()
    _, grad_rot, grad_shift = project_backward(dim, upstream(img, gd, rot_, shift_), gd, rot_,
                                               shift=shift_, need_src=False, **kw)
    grad_weights = None
    if grad_weight is not None:
        gw = _c(grad_weight, np.complex128)
        grad_weights = np.broadcast_to(project(dim, gw, rot_, shift=None, N=N, **kw).real,
                                       img.shape).copy()
        om = np.ones(img.shape) if weights is None else _c(weights, np.float64)
        _, gr_w, _ = project_backward(dim, upstream(om, gw, rot_).astype(np.complex128), gw, rot_,
                                      shift=None, need_src=False, need_shift=False, **kw)
        grad_rot = grad_rot + gr_w
    return grad_img, grad_weights, grad_rot, grad_shift


def hermitian_x0(spec, dim, weight=None):
    """Symmetrised zero-frequency axis of accumulated half-spectra.

    The pages' backward pass accumulates the contributions that land on the
    kx = 0 axis symmetrically, so that the pair (0, k), (0, -k) -- one
    Fourier coefficient of a real object and its conjugate -- is not counted
    twice with different values ("torch-projectors", [ar §2] Friedel
    symmetry, backward pass; [de §2 "Friedel-Symmetrie"]).  The pages give no
    formula; the reading taken here is the Hermitian part of the stored
    kx = 0 plane (3D) or column (2D):

        V'(0, k) = (V(0, k) + conj(V(0, -k))) / 2,    W'(0, k) = (W(0, k) + W(0, -k)) / 2,

    with -k taken modulo the box in every stored axis (rfftn row order), so
    self-conjugate points keep their real part.  Every other coefficient is
    unchanged.  spec is (B, M, M, M/2+1) for dim 3 or (B, M, M/2+1) for dim
    2, weight (real, same shape) or None.  Returns new arrays (spec', weight').
    """
    spec = np.array(spec, dtype=np.complex128)
    out_w = None if weight is None else np.array(weight, dtype=np.float64)
    M = spec.shape[1]
    neg = (-np.arange(M)) % M          # row of -k for the row of k
    if dim == 3:
        plane = spec[:, :, :, 0].copy()                      # (B, z, y)
        mirror = plane[:, neg][:, :, neg]                    # V(0, -z, -y)
        spec[:, :, :, 0] = 0.5 * (plane + np.conj(mirror))
        if out_w is not None:
            wp = out_w[:, :, :, 0].copy()
            out_w[:, :, :, 0] = 0.5 * (wp + wp[:, neg][:, :, neg])
    elif dim == 2:
        col = spec[:, :, 0].copy()                           # (B, y)
        spec[:, :, 0] = 0.5 * (col + np.conj(col[:, neg]))
        if out_w is not None:
            wc = out_w[:, :, 0].copy()
            out_w[:, :, 0] = 0.5 * (wc + wc[:, neg])
    else:
        raise ValueError("dim must be 2 or 3")
    return spec, out_w
