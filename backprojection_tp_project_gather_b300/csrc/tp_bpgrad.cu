// tp_bpgrad.cu -- the weight-spectrum part of the gradients of the 3D
// backprojection (tp_backproject_2d_3d_backward).
//
// The backprojection adds, per image pixel k and tap n, w_n(p_k) * omega_k to
// the real weight spectrum [de §2 "Dual-Volumen-Ansatz"; it §2 "accumulo di
// pesi"], with omega the image weights (1 when none are given) and no phase.
// For an upstream gradient GW of that spectrum:
//   dL/domega_k  = sum_n GW[n] w_n(p_k)           = Re of the unshifted
//                  projection of GW at pixel k
//   dL/dp_a     += omega_k sum_n GW[n] dw_n/dp_a   = omega_k Re D_a(GW)
// with D_a the saved derivative of that projection (tp_brick.cu), and
// dL/dR[i][a] += s k_i dL/dp_a as for the forward (p = s R^T k,
// [ko §2 "Forward Projection"]).  The data-spectrum part reuses the forward
// with saved derivatives and the saved-path pose gradient (tp_saved.cu).
#include <cuda_runtime.h>

#include "tp_launch.h"

namespace tp {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;

__global__ void __launch_bounds__(256) k_real_to_complex(const float *__restrict__ src,
                                                         float2 *__restrict__ dst, long long n) {
    for (long long i = (long long)blockIdx.x * 256 + threadIdx.x; i < n;
         i += (long long)gridDim.x * 256)
        dst[i] = make_float2(__ldg(src + i), 0.f);
}

// One block per output image, one warp per row: grad_weights gets Re y over
// the whole image (zero outside the radius, where y is zero), and the
// in-radius pixels add omega Re D_a s k_i to grad_rot.
__global__ void __launch_bounds__(kThreads) k_weight_grads(Params q, const float *__restrict__ omega,
                                                           const float2 *__restrict__ y,
                                                           const float2 *__restrict__ D,
                                                           float *__restrict__ grad_weights,
                                                           float *__restrict__ grad_rot) {
    __shared__ float part[kWarps][6];
    const int bp = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = q.N >> 1;
    float acc[6];
#pragma unroll
    for (int i = 0; i < 6; ++i) acc[i] = 0.f;
    for (int iy = warp; iy < q.N; iy += kWarps) {
        const int ky = row_freq(iy, q.N);
        const int rr = q.r2max - ky * ky;
        const int xcut = rr < 0 ? -1 : min(half, (int)floorf(sqrtf((float)rr)));
        const size_t r0 = (size_t)bp * q.plane + (size_t)iy * q.Xo;
        if (!TP_CHECK(q.dbg, r0 + half < (size_t)q.B * q.P * q.plane, 10)) continue;
        if (grad_weights)
            for (int kx = lane; kx <= half; kx += 32) grad_weights[r0 + kx] = __ldg(&y[r0 + kx].x);
        if (!grad_rot) continue;
        for (int kx = lane; kx <= xcut; kx += 32) {
            const size_t e = r0 + kx;
            const float om = omega ? __ldg(omega + e) : 1.0f;
            const float skx = q.s * (float)kx, sky = q.s * (float)ky;
#pragma unroll
            for (int a = 0; a < 3; ++a) {
                const float dl = om * __ldg(&D[3 * e + a].x);
                acc[a] = fmaf(skx, dl, acc[a]);
                acc[3 + a] = fmaf(sky, dl, acc[3 + a]);
            }
        }
    }
    if (!grad_rot) return;
#pragma unroll
    for (int i = 0; i < 6; ++i) {
        float t = acc[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0) part[warp][i] = t;
    }
    __syncthreads();
    if (warp != 0 || lane >= 6) return;
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t += part[w][lane];
    const int b = bp / q.P, pi = bp - b * q.P;
    const int ridx = ((q.Bp == 1) ? 0 : b) * q.P + pi;
    if (t != 0.f && TP_CHECK(q.dbg, ridx < q.Bp * q.P, 9)) atomicAdd(grad_rot + (size_t)ridx * 9 + lane, t);
}

}  // namespace

cudaError_t launch_real_to_complex(const float *src, float2 *dst, long long n, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    long long blocks = (n + 255) / 256;
    if (blocks > 148LL * 64) blocks = 148LL * 64;
    k_real_to_complex<<<(unsigned)blocks, 256, 0, st>>>(src, dst, n);
    return cudaGetLastError();
}

cudaError_t launch_weight_grads(const Params &q, const float *omega, const float2 *y,
                                const float2 *D, float *grad_weights, float *grad_rot,
                                cudaStream_t st) {
    const long long images = (long long)q.B * q.P;
    if (images == 0 || (!grad_weights && !grad_rot)) return cudaSuccess;
    k_weight_grads<<<(unsigned)images, kThreads, 0, st>>>(q, omega, y, D, grad_weights, grad_rot);
    return cudaGetLastError();
}

}  // namespace tp
