// tp_scatter.cu -- scatter-side kernels: backprojection of data and weights
// and the spectrum gradient (the adjoint of the forward projection).
//
// One thread per input Fourier sample; each in-radius sample spreads
// w * conj(phase) * y over its stencil with vector atomics (float2 RED into
// the complex spectrum, f32 RED into the weight spectrum).  Friedel taps
// (n_x < 0) add the conjugate at -n, which makes this the exact real adjoint
// of the gather in tp_gather.cu.
//
// Method: "torch-projectors: A High-Performance Differentiable Projection
// Library for PyTorch", backprojection [it §2 "Operazioni Supportate";
// ko §2 "Backward Projection"] with the dual data/weight volume
// [de §2 "Dual-Volumen-Ansatz"]; the pages name global atomics as the cost
// of the scatter [it §4 "Backward Pass"].
#include "tp_device.cuh"
#include "tp_launch.h"

namespace tp {

namespace {

constexpr int kThreads = kSampleBlock;

template <int D, bool CUBIC>
__global__ void __launch_bounds__(kThreads) k_scatter(Params q, const float2 *__restrict__ img,
                                                      const float *__restrict__ omega,
                                                      float2 *__restrict__ dst,
                                                      float *__restrict__ wdst) {
    using St = Stencil<CUBIC>;
    constexpr int T = St::TAPS;
    const int bp = blockIdx.x / q.tiles;
    const int rem = (blockIdx.x - bp * q.tiles) * kThreads + threadIdx.x;
    if (rem >= q.plane) return;
    const int b = bp / q.P;
    const int pi = bp - b * q.P;
    const int iy = rem / q.Xo;
    const int kx = rem - iy * q.Xo;
    const int ky = row_freq(iy, q.N);
    if (kx * kx + ky * ky > q.r2max) return;
    const Pose<D> ps = load_pose<D>(q, b, pi);
    const size_t sidx = (size_t)bp * q.plane + rem;
    float2 c = __ldg(img + sidx);
    if (q.shift) c = cmul_conj_a(shift_phase(kx, ky, ps.sx, ps.sy, q.fN, q.invN), c);
    const float om = omega ? __ldg(omega + sidx) : 1.0f;

    float p[D];
#pragma unroll
    for (int j = 0; j < D; ++j) p[j] = fmaf(ps.a[j], (float)kx, ps.b[j] * (float)ky);
    int x0[D];
    float w[D][4];
#pragma unroll
    for (int a = 0; a < D; ++a) {
        float t;
        x0[a] = split_coord(p[a], t);
        St::weights(t, w[a]);
    }
    const size_t boff = (q.Bsrc == 1) ? 0 : (size_t)b * q.src_stride;
    float2 *V = dst + boff;
    float *W = wdst ? wdst + boff : nullptr;
    const int half = q.M >> 1;
    const int M = q.M, X = q.Xs;
    constexpr int TZ = (D == 3) ? T : 1;
#pragma unroll
    for (int jz = 0; jz < TZ; ++jz) {
#pragma unroll
        for (int jy = 0; jy < T; ++jy) {
#pragma unroll
            for (int jx = 0; jx < T; ++jx) {
                int nx = x0[0] - St::LO + jx;
                int ny = x0[1] - St::LO + jy;
                int nz = 0;
                if constexpr (D == 3) nz = x0[2] - St::LO + jz;
                const bool cj = nx < 0;
                if (cj) {
                    nx = -nx;
                    ny = -ny;
                    nz = -nz;
                }
                if (nx > half || !row_ok(ny, half)) continue;
                size_t e = (size_t)wrap_row(ny, M) * X + nx;
                float wt = w[0][jx] * w[1][jy];
                if constexpr (D == 3) {
                    if (!row_ok(nz, half)) continue;
                    e += (size_t)wrap_row(nz, M) * M * X;
                    wt *= w[2][jz];
                }
                if (!TP_CHECK(q.dbg, e < (size_t)(D == 3 ? M : 1) * M * X, 6)) continue;
                atomicAdd(V + e, make_float2(wt * c.x, cj ? -wt * c.y : wt * c.y));
                if (W) atomicAdd(W + e, wt * om);
            }
        }
    }
}

template <int D, bool CUBIC>
cudaError_t launch_scatter_t(const Params &q, const float2 *img, const float *omega, float2 *dst,
                             float *wdst, cudaStream_t st) {
    const long long blocks = (long long)q.B * q.P * q.tiles;
    k_scatter<D, CUBIC><<<(unsigned)blocks, kThreads, 0, st>>>(q, img, omega, dst, wdst);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scatter(int dim, bool cubic, const Params &q, const float2 *img,
                           const float *omega, float2 *dst, float *wdst, cudaStream_t st) {
    if (dim == 3)
        return cubic ? launch_scatter_t<3, true>(q, img, omega, dst, wdst, st)
                     : launch_scatter_t<3, false>(q, img, omega, dst, wdst, st);
    return cubic ? launch_scatter_t<2, true>(q, img, omega, dst, wdst, st)
                 : launch_scatter_t<2, false>(q, img, omega, dst, wdst, st);
}

}  // namespace tp
