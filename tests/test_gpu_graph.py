"""GPU: a whole differentiable step captured in a CUDA graph and replayed.

The library allocates nothing and enqueues everything on the caller's
stream, so a step (forward with saved derivatives, loss gradient, pose
gradients, volume gradient) can be captured once and replayed with new
inputs written into the captured tensors.  The replay must equal the eager
calls on the same inputs, including new poses (the binning re-runs inside
the graph) and poses equal to the previous replay's (it is kept).
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tp():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import backprojection_tp_project_gather_b300 as m
    return m


def crandn(rng, shape):
    return (rng.standard_normal(shape) + 1j * rng.standard_normal(shape)).astype(np.complex64)


def test_step_in_a_cuda_graph(tp):
    rng = np.random.default_rng(81)
    M = N = 32
    P = 6
    kw = dict(interp="cubic", oversampling=1.0, radius=-1.0)
    dev = torch.device("cuda")

    def inputs(seed):
        r = np.random.default_rng(seed)
        return (torch.from_numpy(crandn(r, (1, M, M, M // 2 + 1))).to(dev),
                torch.from_numpy(synth.random_rotations(P, r)[None]).to(dev),
                torch.from_numpy(r.uniform(-3, 3, (1, P, 2)).astype(np.float32)).to(dev),
                torch.from_numpy(crandn(r, (1, P, N, N // 2 + 1))).to(dev))

    vol, rot, shift, target = (t.clone() for t in inputs(1))
    y = torch.empty_like(target)
    D = torch.empty(tuple(target.shape) + (3,), dtype=torch.complex64, device=dev)
    g = torch.empty_like(target)
    gv, gr, gs = torch.zeros_like(vol), torch.zeros_like(rot), torch.zeros_like(shift)
    ws = torch.zeros(tp.tp_workspace_bytes(1, 1, P, M, "cubic"), dtype=torch.uint8, device=dev)

    def step():
        tp.tp_project_3d_2d_save(vol, rot, shift, out=y, dout=D, workspace=ws, **kw)
        torch.sub(y, target, out=g)
        g.mul_(2.0)
        gv.zero_()
        gr.zero_()
        gs.zero_()
        tp.tp_project_3d_2d_backward_saved(g, y, D, rot, shift, grad_rot=gr, grad_shift=gs, **kw)
        tp.tp_project_3d_2d_backward(g, vol, rot, shift, grad_vol=gv, want_rot=False,
                                     want_shift=False, workspace=ws, **kw)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                                   # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    def eager(v, r, t, tg):
        yy, dd = tp.tp_project_3d_2d_save(v, r, t, **kw)
        gg = 2 * (yy - tg)
        ggv, _, _ = tp.tp_project_3d_2d_backward(gg, v, r, t, want_rot=False, want_shift=False,
                                                 **kw)
        ggr, ggs = tp.tp_project_3d_2d_backward_saved(gg, yy, dd, r, t, **kw)
        return yy, ggv, ggr, ggs

    for seed in (2, 3, 3):                       # new inputs, then the same poses again
        new = inputs(seed)
        for dst, src in zip((vol, rot, shift, target), new):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        ref = eager(*new)
        for got, want in zip((y, gv, gr, gs), ref):
            a, b = got.cpu().numpy(), want.cpu().numpy()
            assert np.linalg.norm(a - b) <= 1e-5 * np.linalg.norm(b), seed
