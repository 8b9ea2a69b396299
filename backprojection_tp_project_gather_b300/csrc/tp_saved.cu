// tp_saved.cu -- rotation and shift gradients of the 3D forward projection
// from the values its forward pass saved.
//
// The forward maps output pixel k = (kx, ky) to the sample position
// p = s R^T k (k_z = 0) and writes y = phase * S(p).  With the saved
// D_a = phase * dS/dp_a (tp_project_3d_2d_save) the chain rule gives, per
// pixel with upstream gradient g (the real adjoint, as in the backward pass
// that recomputes S):
//   dL/dp_a       = Re(conj(g) D_a)
//   dL/dR[i][a]  += s k_i dL/dp_a           (i = 0, 1; row 2 stays 0)
//   dL/dshift_a  += (2 pi k_a / N) Im(conj(g) y)
// These are the analytic rotation and shift gradients of "torch-projectors: A
// High-Performance Differentiable Projection Library for PyTorch" [de §3 item 4;
// ar §2], with the inverse rotation of [ko §2 "Forward Projection"] and the
// shift phase exp(-2 pi i (kx sx + ky sy) / N) of [de §2 "Interpolation"].
// This is a streaming reduction over (g, y, D): one block per output image,
// one warp per row, the in-radius pixels only (y and D are zero outside).
#include <cuda_runtime.h>

#include "tp_launch.h"

namespace tp {

namespace {

constexpr int kSavedWarps = 8;
constexpr int kSavedThreads = 32 * kSavedWarps;

__global__ void __launch_bounds__(kSavedThreads) k_pose_grad_saved(Params q,
                                                                   const float2 *__restrict__ g,
                                                                   const float2 *__restrict__ y,
                                                                   const float2 *__restrict__ D,
                                                                   float *__restrict__ grad_rot,
                                                                   float *__restrict__ grad_shift) {
    __shared__ float part[kSavedWarps][8];
    const int bp = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = q.N >> 1;
    const float tau = 6.283185307179586f * q.invN;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int iy = warp; iy < q.N; iy += kSavedWarps) {
        const int ky = row_freq(iy, q.N);
        const int rr = q.r2max - ky * ky;
        if (rr < 0) continue;
        const int xcut = min(half, (int)floorf(sqrtf((float)rr)));
        const size_t r0 = (size_t)bp * q.plane + (size_t)iy * q.Xo;
        if (!TP_CHECK(q.dbg, r0 + half < (size_t)q.B * q.P * q.plane, 10)) continue;
        // Four pixels per lane per pass: all their loads are issued before
        // any of them is used, to keep enough bytes in flight.
        for (int x0 = 0; x0 <= xcut; x0 += 4 * 32) {
            float2 gv[4], yv[4], dv[4][3];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int kx = x0 + u * 32 + lane;
                const size_t e = r0 + min(kx, xcut);
                gv[u] = kx <= xcut ? __ldg(g + e) : make_float2(0.f, 0.f);
                yv[u] = __ldg(y + e);
#pragma unroll
                for (int a = 0; a < 3; ++a) dv[u][a] = __ldg(D + 3 * e + a);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int kx = x0 + u * 32 + lane;   // gv is 0 beyond xcut
                const float skx = q.s * (float)kx, sky = q.s * (float)ky;
#pragma unroll
                for (int a = 0; a < 3; ++a) {
                    const float dl = gv[u].x * dv[u][a].x + gv[u].y * dv[u][a].y;   // Re(conj(g) D_a)
                    acc[a] = fmaf(skx, dl, acc[a]);
                    acc[3 + a] = fmaf(sky, dl, acc[3 + a]);
                }
                const float qv = tau * (gv[u].x * yv[u].y - gv[u].y * yv[u].x);   // (2 pi / N) Im(conj(g) y)
                acc[6] = fmaf((float)kx, qv, acc[6]);
                acc[7] = fmaf((float)ky, qv, acc[7]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float t = acc[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) part[warp][i] = t;
    }
    __syncthreads();
    if (warp != 0) return;
    float t = lane < 8 ? part[0][lane] : 0.f;
#pragma unroll
    for (int w = 1; w < kSavedWarps; ++w) t += lane < 8 ? part[w][lane] : 0.f;
    const int b = bp / q.P, pi = bp - b * q.P;
    if (lane < 6 && grad_rot) {
        const int ridx = ((q.Bp == 1) ? 0 : b) * q.P + pi;
        if (t != 0.f && TP_CHECK(q.dbg, ridx < q.Bp * q.P, 9))
            atomicAdd(grad_rot + (size_t)ridx * 9 + lane, t);
    } else if (lane >= 6 && lane < 8 && grad_shift) {
        const int sidx = ((q.Bs == 1) ? 0 : b) * q.P + pi;
        if (t != 0.f && TP_CHECK(q.dbg, sidx < q.Bs * q.P, 9))
            atomicAdd(grad_shift + 2 * (size_t)sidx + (lane - 6), t);
    }
}

}  // namespace

cudaError_t launch_pose_grad_saved(const Params &q, const float2 *grad_out, const float2 *y,
                                   const float2 *D, float *grad_rot, float *grad_shift,
                                   cudaStream_t st) {
    const long long images = (long long)q.B * q.P;
    if (images == 0 || (!grad_rot && !grad_shift)) return cudaSuccess;
    k_pose_grad_saved<<<(unsigned)images, kSavedThreads, 0, st>>>(q, grad_out, y, D, grad_rot,
                                                                   grad_shift);
    return cudaGetLastError();
}

}  // namespace tp
