// tp_launch.h -- internal launchers behind the C ABI (not exported).
#pragma once

#include <cuda_runtime.h>

#include "tp_device.cuh"

namespace tp {

// Forward projection into out (overwritten).  dim = 2 or 3.
cudaError_t launch_project(int dim, bool cubic, const Params &q, float2 *out, cudaStream_t st);

// dL/dR (rows 0 and 1) and dL/dshift, accumulated with atomics.
cudaError_t launch_pose_grad(int dim, bool cubic, const Params &q, const float2 *grad_out,
                             float *grad_rot, float *grad_shift, cudaStream_t st);

// Adjoint scatter of img (same layout as a forward output) into dst (+=),
// and of w * omega into wdst (+=) when wdst is not null.  q.src / q.Bsrc
// describe the DESTINATION spectrum here (its batch and box).
cudaError_t launch_scatter(int dim, bool cubic, const Params &q, const float2 *img,
                           const float *omega, float2 *dst, float *wdst, cudaStream_t st);

}  // namespace tp
