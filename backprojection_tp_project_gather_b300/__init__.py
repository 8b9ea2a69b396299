"""Python binding of libtp_b300.so, the B300 Fourier-space projection library.

Argument marshalling only: every function checks tensor types, derives the
sizes the C ABI asks for, allocates outputs with PyTorch when the caller
passes none, and calls the ``tp_*`` entry point of the same name on the
current CUDA stream.  All arithmetic runs in the library's CUDA kernels; there
is no CPU path, and every call raises ImportError while the library file is
missing (the package itself imports without it, so that its build module can
run on a fresh checkout).

Layouts follow ``include/tp.h``: spectra are complex64 half-spectra in
``torch.fft.rfftn`` order, rotations float32 ``(Bp, P, d, d)``, shifts float32
``(Bs, P, 2)``.  Backward and backprojection outputs are accumulated (+=)
into the tensors passed in (fresh zeros otherwise).
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "TPError", "lib", "tp_project_3d_2d", "tp_project_3d_2d_backward", "tp_backproject_2d_3d",
    "tp_project_3d_2d_save", "tp_project_3d_2d_backward_saved", "tp_backproject_2d_3d_backward",
    "tp_project_3d_2d_l2",
    "tp_backproject_backward_scratch_bytes", "tp_project_2d_2d", "tp_project_2d_2d_backward",
    "tp_last_error", "tp_version", "tp_workspace_bytes", "tp_project_3d_2d_noalloc",
    "tp_debug_bounds_word", "tp_debug_bounds_selftest", "tp_hermitian_x0", "LINEAR", "CUBIC",
    "FLAG_HERMITIAN_X0",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
# TP_B300_LIB=debug selects the bounds-checking build (libtp_b300_debug.so).
LIB_PATH = os.path.join(_HERE, "libtp_b300_debug.so" if os.environ.get("TP_B300_LIB") == "debug"
                        else "libtp_b300.so")
LINEAR, CUBIC = 0, 1
FLAG_HERMITIAN_X0 = 1   # TP_FLAG_HERMITIAN_X0: symmetrised kx = 0 axis of accumulated spectra



class TPOptions(ctypes.Structure):
    _fields_ = [("interp", ctypes.c_int), ("oversampling", ctypes.c_float),
                ("radius", ctypes.c_float), ("flags", ctypes.c_uint)]


class TPError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"tp status {status}: {message}")
        self.status = status


_lib = None


def _library() -> ctypes.CDLL:
    """Load the library on first use.  The package itself imports without
    it, so that its build module can run on a fresh checkout; every call
    into the library fails loudly while the file is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m backprojection_tp_project_gather_b300.build` (nvcc, sm_103a)")
        _lib = ctypes.CDLL(LIB_PATH)
    return _lib


_P, _I, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_SIGS = {
    "tp_project_3d_2d": [_P, _I, _I, _P, _I, _I, _P, _I, _I, TPOptions, _P, _P, _Z, _P],
    "tp_project_2d_2d": [_P, _I, _I, _P, _I, _I, _P, _I, _I, TPOptions, _P, _P],
    "tp_project_3d_2d_noalloc": [_P, _I, _I, _P, _I, _I, _P, _I, _I, TPOptions, _P, _P],
    "tp_project_3d_2d_save": [_P, _I, _I, _P, _I, _I, _P, _I, _I, TPOptions, _P, _P, _P, _Z, _P],
    "tp_project_3d_2d_l2": [_P, _I, _I, _P, _I, _I, _P, _I, _I, TPOptions, _P, _P, _P, _P, _P, _P,
                            _Z, _P],
    "tp_project_3d_2d_backward": [_P, _P, _I, _I, _P, _I, _I, _P, _I, _I, TPOptions, _P, _P, _P,
                                  _P, _Z, _P],
    "tp_project_3d_2d_backward_saved": [_P, _P, _P, _I, _I, _I, _I, _I, TPOptions, _P, _P, _P],
    "tp_project_2d_2d_backward": [_P, _P, _I, _I, _P, _I, _I, _P, _I, _I, TPOptions, _P, _P, _P, _P],
    "tp_backproject_2d_3d": [_P, _P, _I, _I, _I, _P, _I, _P, _I, _I, _I, TPOptions, _P, _P, _P, _Z,
                             _P],
    "tp_backproject_2d_3d_backward": [_P, _P, _P, _P, _I, _I, _I, _P, _I, _P, _I, _I, _I, TPOptions,
                                      _P, _P, _P, _P, _P, _Z, _P, _Z, _P],
    "tp_backproject_backward_scratch_bytes": [_I, _I, _I, _I, _I, _I],
}
_SIGS["tp_workspace_bytes"] = [_I, _I, _I, _I, _I, TPOptions]
_SIGS["tp_debug_bounds_word"] = [_I]
_SIGS["tp_hermitian_x0"] = [_P, _P, _I, _I, _I, ctypes.c_void_p]
_SIGS["tp_debug_bounds_selftest"] = [_I, ctypes.c_void_p]
_RESTYPES = {"tp_workspace_bytes": ctypes.c_size_t, "tp_last_error": ctypes.c_char_p,
             "tp_debug_bounds_word": ctypes.c_uint,
             "tp_backproject_backward_scratch_bytes": ctypes.c_size_t,
             "tp_version": ctypes.c_char_p}
_bound = {}


def _fn(name):
    """Entry point `name` with its C signature (bound on first use, so a
    rebuild can run while an older library is on disk)."""
    f = _bound.get(name)
    if f is None:
        f = getattr(_library(), name)
        if name in _SIGS:
            f.argtypes = _SIGS[name]
        f.restype = _RESTYPES.get(name, ctypes.c_int)
        _bound[name] = f
    return f


def lib() -> ctypes.CDLL:
    """The loaded ctypes handle of libtp_b300.so."""
    return _library()


def tp_last_error() -> str:
    return _fn("tp_last_error")().decode()


def tp_version() -> str:
    return _fn("tp_version")().decode()


def tp_debug_bounds_word(reset: bool = False) -> int:
    """Failed index-check bits of the debug build (0 in the normal build); see tp.h."""
    return int(_fn("tp_debug_bounds_word")(1 if reset else 0))


def tp_debug_bounds_selftest(bit: int, stream=None) -> None:
    """Debug build: set bit `bit` of the check word through a failing check."""
    _call("tp_debug_bounds_selftest", int(bit), _stream(stream))


def tp_workspace_bytes(Bv, B, P, Nv, interp="cubic", N=None):
    """Workspace bytes the 3D entry points need for volume box Nv and image box N
    (default: Nv); see include/tp.h."""
    N = Nv if N is None else int(N)
    return int(_fn("tp_workspace_bytes")(int(Bv), int(B), int(P), int(Nv), N,
                                         _opts(interp, 1.0, -1.0)))


def _workspace(ws, Bv, B, P, Nv, N, interp, device):
    need = tp_workspace_bytes(Bv, B, P, Nv, interp, N)
    if ws is None:
        # A block fresh from the caching allocator may hold an old workspace
        # of the same shape; clearing its first 256 bytes (the key of the
        # binning kept there) makes the library recompute the binning.
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
        ws[:256].zero_()
    if ws.device.type != "cuda" or not ws.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    nbytes = ws.numel() * ws.element_size()
    return ws, nbytes


def _opts(interp, oversampling, radius, hermitian_x0=False):
    if isinstance(interp, str):
        interp = {"linear": LINEAR, "cubic": CUBIC}[interp]
    return TPOptions(int(interp), float(oversampling), float(radius),
                     FLAG_HERMITIAN_X0 if hermitian_x0 else 0)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need(t, name, dtype, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions (got shape {tuple(t.shape)})")
    return t


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _call(name, *args):
    st = _fn(name)(*args)
    if st != 0:
        raise TPError(st, tp_last_error())


def _batch(*bs):
    return max(bs)


def _poses(rot, shift, d):
    _need(rot, "rot", torch.float32, 4)
    if rot.shape[2:] != (d, d):
        raise ValueError(f"rot must be (Bp, P, {d}, {d})")
    if shift is not None:
        _need(shift, "shift", torch.float32, 3)
        if shift.shape[1] != rot.shape[1] or shift.shape[2] != 2:
            raise ValueError("shift must be (Bs, P, 2) with the rotations' P")
    return rot.shape[0], rot.shape[1], (shift.shape[0] if shift is not None else 1)


def _forward(name, dim, src, rot, shift, N, interp, oversampling, radius, out, stream,
             workspace=None):
    _need(src, "source", torch.complex64, dim + 1)
    Bsrc, M = src.shape[0], src.shape[1]
    Bp, P, Bs = _poses(rot, shift, dim)
    N = M if N is None else int(N)
    B = _batch(Bsrc, Bp, Bs)
    if out is None:
        out = torch.empty((B, P, N, N // 2 + 1), dtype=torch.complex64, device=src.device)
    _need(out, "out", torch.complex64, 4)
    if tuple(out.shape) != (B, P, N, N // 2 + 1):
        raise ValueError(f"out must be {(B, P, N, N // 2 + 1)}")
    args = [_ptr(src), Bsrc, M, _ptr(rot), Bp, P, _ptr(shift), Bs, N,
            _opts(interp, oversampling, radius), _ptr(out)]
    if dim == 3:
        ws, nbytes = _workspace(workspace, Bsrc, B, P, M, N, interp, src.device)
        args += [_ptr(ws), nbytes]
    _call(name, *args, _stream(stream))
    return out


def _backward(name, dim, grad_out, src, rot, shift, interp, oversampling, radius, grad_src,
              grad_rot, grad_shift, want_src, want_rot, want_shift, stream, workspace=None,
              hermitian_x0=False):
    _need(grad_out, "grad_out", torch.complex64, 4)
    _need(src, "source", torch.complex64, dim + 1)
    Bsrc, M = src.shape[0], src.shape[1]
    Bp, P, Bs = _poses(rot, shift, dim)
    N = grad_out.shape[2]
    if want_src and grad_src is None:
        grad_src = torch.zeros_like(src)
    if want_rot and grad_rot is None:
        grad_rot = torch.zeros_like(rot)
    if want_shift and shift is not None and grad_shift is None:
        grad_shift = torch.zeros_like(shift)
    if grad_src is not None:
        _need(grad_src, "grad_src", torch.complex64, dim + 1)
        if grad_src.shape != src.shape:
            raise ValueError("grad of the source must have the source's shape")
    if grad_rot is not None:
        _need(grad_rot, "grad_rot", torch.float32, 4)
        if grad_rot.shape != rot.shape:
            raise ValueError("grad_rot must have rot's shape")
    if grad_shift is not None:
        _need(grad_shift, "grad_shift", torch.float32, 3)
        if shift is None or grad_shift.shape != shift.shape:
            raise ValueError("grad_shift must have shift's shape")
    args = [_ptr(grad_out), _ptr(src), Bsrc, M, _ptr(rot), Bp, P, _ptr(shift), Bs, N,
            _opts(interp, oversampling, radius, hermitian_x0), _ptr(grad_src), _ptr(grad_rot),
            _ptr(grad_shift)]
    if dim == 3:
        B = grad_out.shape[0]
        ws, nbytes = _workspace(workspace, Bsrc, B, P, M, N, interp, grad_out.device)
        args += [_ptr(ws), nbytes]
    _call(name, *args, _stream(stream))
    return grad_src, grad_rot, grad_shift


def tp_project_3d_2d(vol, rot, shift=None, *, N=None, interp="cubic", oversampling=1.0,
                     radius=-1.0, out=None, workspace=None, stream=None):
    """Central slices (B, P, N, N/2+1) of vol (Bv, Nv, Nv, Nv/2+1); see tp.h.

    workspace: optional uint8 CUDA tensor of at least tp_workspace_bytes() bytes
    (allocated per call when omitted)."""
    return _forward("tp_project_3d_2d", 3, vol, rot, shift, N, interp, oversampling, radius, out,
                    stream, workspace)


def tp_project_3d_2d_save(vol, rot, shift=None, *, N=None, interp="cubic", oversampling=1.0,
                          radius=-1.0, out=None, dout=None, workspace=None, stream=None):
    """tp_project_3d_2d that also returns dout (B, P, N, N/2+1, 3) complex:
    phase * dS/dp_a per pixel, for tp_project_3d_2d_backward_saved; see tp.h."""
    _need(vol, "vol", torch.complex64, 4)
    Bv, Nv = vol.shape[0], vol.shape[1]
    Bp, P, Bs = _poses(rot, shift, 3)
    N = Nv if N is None else int(N)
    B = _batch(Bv, Bp, Bs)
    shape = (B, P, N, N // 2 + 1)
    if out is None:
        out = torch.empty(shape, dtype=torch.complex64, device=vol.device)
    if dout is None:
        dout = torch.empty(shape + (3,), dtype=torch.complex64, device=vol.device)
    _need(out, "out", torch.complex64, 4)
    _need(dout, "dout", torch.complex64, 5)
    if tuple(out.shape) != shape or tuple(dout.shape) != shape + (3,):
        raise ValueError(f"out must be {shape} and dout {shape + (3,)}")
    ws, nbytes = _workspace(workspace, Bv, B, P, Nv, N, interp, vol.device)
    _call("tp_project_3d_2d_save", _ptr(vol), Bv, Nv, _ptr(rot), Bp, P, _ptr(shift), Bs, N,
          _opts(interp, oversampling, radius), _ptr(out), _ptr(dout), _ptr(ws), nbytes,
          _stream(stream))
    return out, dout


def tp_project_3d_2d_l2(vol, rot, shift, target, *, N=None, interp="cubic", oversampling=1.0,
                        radius=-1.0, out=None, grad_out=None, grad_rot=None, grad_shift=None,
                        want_rot=True, want_shift=True, workspace=None, stream=None):
    """The forward fused with L = sum |out - target|^2; returns (out, grad_out,
    grad_rot, grad_shift) with grad_out = 2 (out - target) written and the
    rotation / shift gradients accumulated (None where not requested); see tp.h."""
    _need(vol, "vol", torch.complex64, 4)
    Bv, Nv = vol.shape[0], vol.shape[1]
    Bp, P, Bs = _poses(rot, shift, 3)
    N = Nv if N is None else int(N)
    B = _batch(Bv, Bp, Bs)
    shape = (B, P, N, N // 2 + 1)
    _need(target, "target", torch.complex64, 4)
    if tuple(target.shape) != shape:
        raise ValueError(f"target must be {shape}")
    if out is None:
        out = torch.empty(shape, dtype=torch.complex64, device=vol.device)
    if grad_out is None:
        grad_out = torch.empty(shape, dtype=torch.complex64, device=vol.device)
    for t, name in ((out, "out"), (grad_out, "grad_out")):
        _need(t, name, torch.complex64, 4)
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must be {shape}")
    if want_rot and grad_rot is None:
        grad_rot = torch.zeros_like(rot)
    if want_shift and shift is not None and grad_shift is None:
        grad_shift = torch.zeros_like(shift)
    if grad_rot is not None:
        _need(grad_rot, "grad_rot", torch.float32, 4)
        if grad_rot.shape != rot.shape:
            raise ValueError("grad_rot must have rot's shape")
    if grad_shift is not None:
        _need(grad_shift, "grad_shift", torch.float32, 3)
        if shift is None or grad_shift.shape != shift.shape:
            raise ValueError("grad_shift must have shift's shape")
    ws, nbytes = _workspace(workspace, Bv, B, P, Nv, N, interp, vol.device)
    _call("tp_project_3d_2d_l2", _ptr(vol), Bv, Nv, _ptr(rot), Bp, P, _ptr(shift), Bs, N,
          _opts(interp, oversampling, radius), _ptr(target), _ptr(out), _ptr(grad_out),
          _ptr(grad_rot), _ptr(grad_shift), _ptr(ws), nbytes, _stream(stream))
    return out, grad_out, grad_rot, grad_shift


def tp_project_3d_2d_backward_saved(grad_out, out, dout, rot, shift=None, *, interp="cubic",
                                    oversampling=1.0, radius=-1.0, grad_rot=None,
                                    grad_shift=None, want_rot=True, want_shift=True, stream=None):
    """dL/dR and dL/dshift (accumulated) from a tp_project_3d_2d_save forward's
    out and dout; rot and shift only give the gradients' shapes and batches."""
    _need(grad_out, "grad_out", torch.complex64, 4)
    _need(out, "out", torch.complex64, 4)
    _need(dout, "dout", torch.complex64, 5)
    B, P, N = grad_out.shape[0], grad_out.shape[1], grad_out.shape[2]
    if tuple(out.shape) != tuple(grad_out.shape) or tuple(dout.shape) != tuple(grad_out.shape) + (3,):
        raise ValueError("grad_out, out and dout (with a trailing 3) must have the same shape")
    Bp, Pr, Bs = _poses(rot, shift, 3)
    if Pr != P:
        raise ValueError("rot must have grad_out's P")
    if want_rot and grad_rot is None:
        grad_rot = torch.zeros_like(rot)
    if want_shift and shift is not None and grad_shift is None:
        grad_shift = torch.zeros_like(shift)
    if grad_rot is not None:
        _need(grad_rot, "grad_rot", torch.float32, 4)
        if grad_rot.shape != rot.shape:
            raise ValueError("grad_rot must have rot's shape")
    if grad_shift is not None:
        _need(grad_shift, "grad_shift", torch.float32, 3)
        if shift is None or grad_shift.shape != shift.shape:
            raise ValueError("grad_shift must have shift's shape")
    _call("tp_project_3d_2d_backward_saved", _ptr(grad_out), _ptr(out), _ptr(dout), B, P, N, Bp, Bs,
          _opts(interp, oversampling, radius), _ptr(grad_rot), _ptr(grad_shift), _stream(stream))
    return grad_rot, grad_shift


def tp_project_3d_2d_noalloc(vol, rot, shift=None, *, N=None, interp="cubic", oversampling=1.0,
                             radius=-1.0, out=None, stream=None):
    """tp_project_3d_2d for callers that cannot allocate device scratch.

    The library keeps the scratch in a fixed array of its own instead of a
    caller workspace; include/tp.h gives its size limit and the rule that such
    calls must not overlap on the GPU.  Pass `out` to avoid the one output
    allocation this wrapper would otherwise make.
    """
    _need(vol, "vol", torch.complex64, 4)
    Bv, Nv = vol.shape[0], vol.shape[1]
    Bp, P, Bs = _poses(rot, shift, 3)
    N = Nv if N is None else int(N)
    B = _batch(Bv, Bp, Bs)
    if out is None:
        out = torch.empty((B, P, N, N // 2 + 1), dtype=torch.complex64, device=vol.device)
    _need(out, "out", torch.complex64, 4)
    if tuple(out.shape) != (B, P, N, N // 2 + 1):
        raise ValueError(f"out must be {(B, P, N, N // 2 + 1)}")
    _call("tp_project_3d_2d_noalloc", _ptr(vol), Bv, Nv, _ptr(rot), Bp, P, _ptr(shift), Bs, N,
          _opts(interp, oversampling, radius), _ptr(out), _stream(stream))
    return out


def tp_project_2d_2d(img, rot, shift=None, *, N=None, interp="cubic", oversampling=1.0,
                     radius=-1.0, out=None, stream=None):
    """Rotated / shifted spectra (B, P, N, N/2+1) of img (Bi, Ni, Ni/2+1); see tp.h."""
    return _forward("tp_project_2d_2d", 2, img, rot, shift, N, interp, oversampling, radius, out,
                    stream)


def tp_project_3d_2d_backward(grad_out, vol, rot, shift=None, *, interp="cubic",
                              oversampling=1.0, radius=-1.0, grad_vol=None, grad_rot=None,
                              grad_shift=None, want_vol=True, want_rot=True, want_shift=True,
                              workspace=None, stream=None, hermitian_x0=False):
    """(grad_vol, grad_rot, grad_shift), accumulated into the given tensors; see tp.h.

    hermitian_x0: symmetrise the kx = 0 plane of grad_vol (TP_FLAG_HERMITIAN_X0)."""
    return _backward("tp_project_3d_2d_backward", 3, grad_out, vol, rot, shift, interp,
                     oversampling, radius, grad_vol, grad_rot, grad_shift, want_vol, want_rot,
                     want_shift, stream, workspace, hermitian_x0)


def tp_project_2d_2d_backward(grad_out, img, rot, shift=None, *, interp="cubic",
                              oversampling=1.0, radius=-1.0, grad_img=None, grad_rot=None,
                              grad_shift=None, want_img=True, want_rot=True, want_shift=True,
                              stream=None, hermitian_x0=False):
    """(grad_img, grad_rot, grad_shift), accumulated into the given tensors; see tp.h.

    hermitian_x0: symmetrise the kx = 0 column of grad_img (TP_FLAG_HERMITIAN_X0)."""
    return _backward("tp_project_2d_2d_backward", 2, grad_out, img, rot, shift, interp,
                     oversampling, radius, grad_img, grad_rot, grad_shift, want_img, want_rot,
                     want_shift, stream, None, hermitian_x0)


def tp_backproject_2d_3d(proj, rot, shift=None, weights=None, *, Nv=None, Bv=1, interp="cubic",
                         oversampling=1.0, radius=-1.0, data_vol=None, weight_vol=None,
                         want_weights=True, workspace=None, stream=None, hermitian_x0=False):
    """Scatter proj (B, P, N, N/2+1) into (data_vol, weight_vol) of box Nv (+=); see tp.h.

    hermitian_x0: symmetrise the kx = 0 planes afterwards (TP_FLAG_HERMITIAN_X0)."""
    _need(proj, "proj", torch.complex64, 4)
    B, P, N = proj.shape[0], proj.shape[1], proj.shape[2]
    Bp, Pr, Bs = _poses(rot, shift, 3)
    if Pr != P:
        raise ValueError("rot must have the projections' P")
    Nv = N if Nv is None else int(Nv)
    shape = (Bv, Nv, Nv, Nv // 2 + 1)
    if weights is not None:
        _need(weights, "weights", torch.float32, 4)
        if weights.shape != proj.shape:
            raise ValueError("weights must have proj's shape")
    if data_vol is None:
        data_vol = torch.zeros(shape, dtype=torch.complex64, device=proj.device)
    if want_weights and weight_vol is None:
        weight_vol = torch.zeros(shape, dtype=torch.float32, device=proj.device)
    _need(data_vol, "data_vol", torch.complex64, 4)
    if tuple(data_vol.shape) != shape:
        raise ValueError(f"data_vol must be {shape}")
    if weight_vol is not None:
        _need(weight_vol, "weight_vol", torch.float32, 4)
        if tuple(weight_vol.shape) != shape:
            raise ValueError(f"weight_vol must be {shape}")
    ws, nbytes = _workspace(workspace, Bv, B, P, Nv, N, interp, proj.device)
    _call("tp_backproject_2d_3d", _ptr(proj), _ptr(weights), B, P, N, _ptr(rot), Bp, _ptr(shift),
          Bs, Bv, Nv, _opts(interp, oversampling, radius, hermitian_x0), _ptr(data_vol),
          _ptr(weight_vol),
          _ptr(ws), nbytes, _stream(stream))
    return data_vol, weight_vol


def tp_hermitian_x0(spec=None, weight=None, *, dim=3, stream=None):
    """Symmetrise the kx = 0 plane (dim 3) or column (dim 2) in place; see tp.h.

    spec: complex64 (B, N, N, N/2+1) or (B, N, N/2+1); weight: float32 of the
    same shape; either may be None.  Returns (spec, weight)."""
    ref = spec if spec is not None else weight
    if ref is None:
        raise ValueError("spec or weight is required")
    if dim not in (2, 3):
        raise ValueError("dim must be 2 or 3")
    if spec is not None:
        _need(spec, "spec", torch.complex64, dim + 1)
    if weight is not None:
        _need(weight, "weight", torch.float32, dim + 1)
        if spec is not None and weight.shape != spec.shape:
            raise ValueError("weight must have spec's shape")
    _call("tp_hermitian_x0", _ptr(spec), _ptr(weight), ref.shape[0], ref.shape[1], dim,
          _stream(stream))
    return spec, weight


def tp_backproject_backward_scratch_bytes(Bv, B, P, N, Nv, with_weight_grad=True):
    """Scratch bytes tp_backproject_2d_3d_backward needs (see include/tp.h)."""
    return int(_fn("tp_backproject_backward_scratch_bytes")(int(Bv), int(B), int(P), int(N), int(Nv),
                                                            1 if with_weight_grad else 0))


def tp_backproject_2d_3d_backward(grad_data_vol, proj, rot, shift=None, weights=None,
                                  grad_weight_vol=None, *, interp="cubic", oversampling=1.0,
                                  radius=-1.0, grad_proj=None, grad_weights=None, grad_rot=None,
                                  grad_shift=None, want_proj=True, want_weights=True,
                                  want_rot=True, want_shift=True, scratch=None, workspace=None,
                                  stream=None):
    """Gradients of tp_backproject_2d_3d: (grad_proj, grad_weights, grad_rot, grad_shift).

    grad_proj and grad_weights are written; grad_rot and grad_shift are
    accumulated into the given tensors (zeros when omitted); see tp.h."""
    _need(grad_data_vol, "grad_data_vol", torch.complex64, 4)
    _need(proj, "proj", torch.complex64, 4)
    Bv, Nv = grad_data_vol.shape[0], grad_data_vol.shape[1]
    B, P, N = proj.shape[0], proj.shape[1], proj.shape[2]
    Bp, Pr, Bs = _poses(rot, shift, 3)
    if Pr != P:
        raise ValueError("rot must have the projections' P")
    if weights is not None:
        _need(weights, "weights", torch.float32, 4)
        if weights.shape != proj.shape:
            raise ValueError("weights must have proj's shape")
    if grad_weight_vol is not None:
        _need(grad_weight_vol, "grad_weight_vol", torch.float32, 4)
        if grad_weight_vol.shape != grad_data_vol.shape:
            raise ValueError("grad_weight_vol must have grad_data_vol's shape")
    dev = proj.device
    if want_proj and grad_proj is None:
        grad_proj = torch.empty_like(proj)
    if want_weights and grad_weight_vol is not None and grad_weights is None:
        grad_weights = torch.empty(proj.shape, dtype=torch.float32, device=dev)
    if want_rot and grad_rot is None:
        grad_rot = torch.zeros_like(rot)
    if want_shift and shift is not None and grad_shift is None:
        grad_shift = torch.zeros_like(shift)
    for t, name, dt in ((grad_proj, "grad_proj", torch.complex64),
                        (grad_weights, "grad_weights", torch.float32)):
        if t is not None:
            _need(t, name, dt, 4)
            if t.shape != proj.shape:
                raise ValueError(f"{name} must have proj's shape")
    if grad_rot is not None:
        _need(grad_rot, "grad_rot", torch.float32, 4)
        if grad_rot.shape != rot.shape:
            raise ValueError("grad_rot must have rot's shape")
    if grad_shift is not None:
        _need(grad_shift, "grad_shift", torch.float32, 3)
        if shift is None or grad_shift.shape != shift.shape:
            raise ValueError("grad_shift must have shift's shape")
    weight_terms = grad_weight_vol is not None and (grad_weights is not None or grad_rot is not None)
    need = tp_backproject_backward_scratch_bytes(Bv, B, P, N, Nv, weight_terms)
    if scratch is None:
        scratch = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if scratch.device.type != "cuda" or not scratch.is_contiguous():
        raise ValueError("scratch must be a contiguous CUDA tensor")
    ws, nbytes = _workspace(workspace, Bv, B, P, Nv, N, interp, dev)
    _call("tp_backproject_2d_3d_backward", _ptr(grad_data_vol), _ptr(grad_weight_vol), _ptr(proj),
          _ptr(weights), B, P, N, _ptr(rot), Bp, _ptr(shift), Bs, Bv, Nv,
          _opts(interp, oversampling, radius), _ptr(grad_proj), _ptr(grad_weights), _ptr(grad_rot),
          _ptr(grad_shift), _ptr(scratch), scratch.numel() * scratch.element_size(), _ptr(ws),
          nbytes, _stream(stream))
    return grad_proj, grad_weights, grad_rot, grad_shift
