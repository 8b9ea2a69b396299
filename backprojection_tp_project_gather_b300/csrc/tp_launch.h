// tp_launch.h -- internal launchers behind the C ABI (not exported).
#pragma once

#include <cuda_runtime.h>

#include "../../include/tp.h"
#include "tp_device.cuh"

namespace tp {

// Record the calling thread's failure message (read back by tp_last_error)
// and return st; every entry point reports its failures through this.
tp_status fail(tp_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));

// 2D operators (the 3D ones are the brick kernels below).
// Forward 2D -> 2D projection into out (overwritten) (tp_gather.cu).
cudaError_t launch_project_2d(bool cubic, const Params &q, float2 *out, cudaStream_t st);

// dL/dR (rows 0 and 1) and dL/dshift of the 2D forward, accumulated with
// atomics (tp_gather.cu).
cudaError_t launch_pose_grad_2d(bool cubic, const Params &q, const float2 *grad_out,
                                float *grad_rot, float *grad_shift, cudaStream_t st);

// The same two operators with the whole Friedel-completed source plane staged
// in shared memory (tp_plane2d.cu), for source box M and output box N whose
// plane (and phase tables) fit a block's shared memory (plane2d_fits).
bool plane2d_fits(int M, int N);
cudaError_t launch_plane2d_project(bool cubic, const Params &q, float2 *out, cudaStream_t st);
cudaError_t launch_plane2d_pose_grad(bool cubic, const Params &q, const float2 *grad_out,
                                     float *grad_rot, float *grad_shift, cudaStream_t st);


// Adjoint scatter of img (same layout as a forward output) into the 2D
// spectrum dst (+=) (tp_scatter.cu).  q.src / q.Bsrc describe the
// DESTINATION spectrum here (its batch and box).
cudaError_t launch_scatter_2d(bool cubic, const Params &q, const float2 *img, float2 *dst,
                              cudaStream_t st);

// 3D brick-binned kernels (tp_brick.cu): forward, pose gradients and
// scatter.  ws is the caller's workspace of brick_workspace_bytes() bytes.
// With kBinNew the launch bins its poses first (pose geometry, brick masks,
// work units; masks and units are kept when the workspace already holds the
// binning of identical poses and sizes); with kBinSameCall it uses the
// binning an earlier launch of the same call made.  With dout the forward
// also writes D_a = phase * dS/dp_a, three complex values per output pixel.
enum BinMode { kBinNew = 0, kBinSameCall = 1 };
size_t brick_workspace_bytes(const Params &q, bool cubic);   // every 3D operator
size_t brick_binning_bytes(const Params &q, bool cubic);     // the forward and pose gradients
long long brick_parts(const Params &q, bool cubic);          // list keys of one volume
// tp_workspace_bytes with or without the cubic scatter's sample lists.
size_t workspace_bytes(int Bv, int B, int P, int Nv, int N, tp_options opts, bool lists);
cudaError_t launch_brick_project(bool cubic, const Params &q, float2 *out, float2 *dout, void *ws,
                                 BinMode mode, cudaStream_t st);
// The forward fused with an L2 data term (always bins its poses): writes out
// and grad_out = 2 (out - target), and accumulates the rotation and shift
// gradients of sum |out - target|^2 (either may be null).
cudaError_t launch_brick_project_l2(bool cubic, const Params &q, const float2 *target, float2 *out,
                                    float2 *grad_out, float *grad_rot, float *grad_shift, void *ws,
                                    cudaStream_t st);
cudaError_t launch_brick_pose_grad(bool cubic, const Params &q, const float2 *grad_out,
                                   float *grad_rot, float *grad_shift, void *ws, BinMode mode,
                                   cudaStream_t st);
cudaError_t launch_brick_scatter(bool cubic, const Params &q, const float2 *img, const float *omega,
                                 float2 *dst, float *wdst, void *ws, BinMode mode, cudaStream_t st);

// dL/dR (rows 0 and 1) and dL/dshift of the 3D forward from its output y and
// saved derivatives D (tp_saved.cu), accumulated with atomics.
cudaError_t launch_pose_grad_saved(const Params &q, const float2 *grad_out, const float2 *y,
                                   const float2 *D, float *grad_rot, float *grad_shift,
                                   cudaStream_t st);

// Weight-spectrum gradients of the backprojection (tp_bpgrad.cu): dst = src
// + 0i for n elements, and grad_weights = Re y (written) plus grad_rot +=
// omega Re D_a s k_i from the unshifted projection y, D of the weight
// spectrum's gradient.
cudaError_t launch_real_to_complex(const float *src, float2 *dst, long long n, cudaStream_t st);
cudaError_t launch_weight_grads(const Params &q, const float *omega, const float2 *y,
                                const float2 *D, float *grad_weights, float *grad_rot,
                                cudaStream_t st);

// The symmetrised kx = 0 plane (dim 3) or column (dim 2) of B stored
// half-spectra of box M, complex V and / or real W (tp_hermitian.cu), in place.
cudaError_t launch_hermitian_x0(float2 *V, float *W, int B, int M, int dim, cudaStream_t st,
                                unsigned *dbg);

}  // namespace tp
