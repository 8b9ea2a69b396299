"""torch.autograd wrappers over the C ABI, for drop-in use in PyTorch models.

The operators are the differentiable projections of "torch-projectors: A
High-Performance Differentiable Projection Library for PyTorch" [de §2
"Differentiable Backpropagation"; it §2 "Operazioni Supportate"]: every
forward and backward step runs in this library's kernels; these classes only
route tensors and gradients.  Complex gradients follow PyTorch's convention
(dL/dRe + i dL/dIm), which is the one the C ABI implements.

  y = project_3d_2d(vol, rot, shift)       # autograd through vol, rot, shift
  y = project_2d_2d(img, rot, shift)

The 3D forward saves D = phase * dS/dp when rot or shift need gradients, so
that their backward is a streaming pass (tp_project_3d_2d_backward_saved);
the volume gradient is the brick scatter of the upstream gradient.

hermitian_x0=True symmetrises the kx = 0 axis of the volume (image)
gradient (TP_FLAG_HERMITIAN_X0): the gradient with respect to a spectrum
constrained to be that of a real object.  The forward is unchanged.
"""
from __future__ import annotations

import torch

from . import (tp_project_2d_2d, tp_project_2d_2d_backward, tp_project_3d_2d,
               tp_project_3d_2d_backward, tp_project_3d_2d_backward_saved,
               tp_project_3d_2d_save, tp_workspace_bytes)


class _Project3D(torch.autograd.Function):
    @staticmethod
    def forward(ctx, vol, rot, shift, N, interp, oversampling, radius, hermitian_x0):
        kw = dict(N=N, interp=interp, oversampling=oversampling, radius=radius)
        need_pose = rot.requires_grad or (shift is not None and shift.requires_grad)
        # One workspace per call: the backward finds the forward's binning in it.
        B = max(vol.shape[0], rot.shape[0], shift.shape[0] if shift is not None else 1)
        ws = torch.empty(max(1, tp_workspace_bytes(vol.shape[0], B, rot.shape[1], vol.shape[1],
                                                   interp, N)), dtype=torch.uint8, device=vol.device)
        ws[:256].zero_()   # a recycled block may hold an old binning's key
        if need_pose:
            out, dout = tp_project_3d_2d_save(vol, rot, shift, workspace=ws, **kw)
        else:
            out, dout = tp_project_3d_2d(vol, rot, shift, workspace=ws, **kw), None
        ctx.save_for_backward(vol, rot, shift, out, dout, ws)
        ctx.opts = dict(interp=interp, oversampling=oversampling, radius=radius)
        ctx.hermitian_x0 = hermitian_x0
        return out

    @staticmethod
    def backward(ctx, grad_out):
        vol, rot, shift, out, dout, ws = ctx.saved_tensors
        grad_out = grad_out.contiguous()
        want_vol, want_rot, want_shift = ctx.needs_input_grad[:3]
        want_shift = want_shift and shift is not None
        gv = gr = gs = None
        if want_rot or want_shift:
            gr, gs = tp_project_3d_2d_backward_saved(grad_out, out, dout, rot, shift,
                                                     want_rot=want_rot, want_shift=want_shift,
                                                     **ctx.opts)
        if want_vol:
            # The workspace still holds the forward's binning of these poses.
            gv, _, _ = tp_project_3d_2d_backward(grad_out, vol, rot, shift, want_rot=False,
                                                 want_shift=False, workspace=ws,
                                                 hermitian_x0=ctx.hermitian_x0, **ctx.opts)
        return gv, gr, gs, None, None, None, None, None


class _Project2D(torch.autograd.Function):
    @staticmethod
    def forward(ctx, img, rot, shift, N, interp, oversampling, radius, hermitian_x0):
        out = tp_project_2d_2d(img, rot, shift, N=N, interp=interp, oversampling=oversampling,
                               radius=radius)
        ctx.save_for_backward(img, rot, shift)
        ctx.opts = dict(interp=interp, oversampling=oversampling, radius=radius,
                        hermitian_x0=hermitian_x0)
        return out

    @staticmethod
    def backward(ctx, grad_out):
        img, rot, shift = ctx.saved_tensors
        want_img, want_rot, want_shift = ctx.needs_input_grad[:3]
        gi, gr, gs = tp_project_2d_2d_backward(grad_out.contiguous(), img, rot, shift,
                                               want_img=want_img, want_rot=want_rot,
                                               want_shift=want_shift and shift is not None,
                                               **ctx.opts)
        return (gi if want_img else None, gr if want_rot else None,
                gs if want_shift else None, None, None, None, None, None)


def project_3d_2d(vol, rot, shift=None, *, N=None, interp="cubic", oversampling=1.0,
                  radius=-1.0, hermitian_x0=False):
    """Differentiable central slices (B, P, N, N/2+1) of vol (Bv, Nv, Nv, Nv/2+1)."""
    return _Project3D.apply(vol, rot, shift, N, interp, oversampling, radius, hermitian_x0)


def project_2d_2d(img, rot, shift=None, *, N=None, interp="cubic", oversampling=1.0,
                  radius=-1.0, hermitian_x0=False):
    """Differentiable rotated / shifted copies (B, P, N, N/2+1) of img (Bi, Ni, Ni/2+1)."""
    return _Project2D.apply(img, rot, shift, N, interp, oversampling, radius, hermitian_x0)
