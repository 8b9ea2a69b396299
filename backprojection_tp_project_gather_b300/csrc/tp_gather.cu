// tp_gather.cu -- gather-side kernels of the 2D operators: the 2D->2D
// forward (rotation and shift) and its rotation / shift gradients.  The
// sampling code is written for D = 2 or 3 axes; the 3D operators use the
// brick kernels of tp_brick.cu, so only D = 2 is instantiated.
//
// One thread per output Fourier sample.  A thread block covers a run of
// consecutive samples of ONE pose (rows of the output plane), so the pose is
// uniform per block, neighbouring threads sample neighbouring points of the
// rotated plane and the stencils of a warp overlap in L1.  The source
// spectrum is read with __ldg through L1/L2 (a box-256 volume is 67.6 MB and
// stays resident in the 126 MB L2); each output sample is written once.
//
// Method: "torch-projectors: A High-Performance Differentiable Projection
// Library for PyTorch", forward projection [it §2 "Operazioni Supportate";
// ko §2 "Forward Projection"] and analytic gradients [de §3 item 4; ar §2].
#include "tp_device.cuh"
#include "tp_launch.h"

namespace tp {

namespace {

constexpr int kThreads = kSampleBlock;

// Sum of w * v over the stencil, and optionally of the derivative weights.
// ND = number of axes (2 or 3).  Coordinates are (x, y[, z]).
template <int D, bool CUBIC, bool DERIV>
struct Gather {
    using St = Stencil<CUBIC>;
    static constexpr int T = St::TAPS;

    // Fast path: every tap lies inside the stored range on the same side of
    // kx = 0.  base[] is the lowest tap coordinate in storage space and
    // w/d are the per-axis weights in ascending storage order.
    __device__ __forceinline__ static void run_fast(const float2 *__restrict__ src, int M, int X,
                                                    const int *base, float (*w)[4], float (*d)[4],
                                                    float2 &S, float2 *dS, unsigned *dbg) {
        const long long nsrc = (long long)(D == 3 ? M : 1) * M * X;
        if constexpr (D == 3) {
#pragma unroll
            for (int jz = 0; jz < T; ++jz) {
                const int zi = wrap_row(base[2] + jz, M);
                float2 ay = make_float2(0.f, 0.f), ayx = ay, ayy = ay;
#pragma unroll
                for (int jy = 0; jy < T; ++jy) {
                    const int yi = wrap_row(base[1] + jy, M);
                    const float2 *row = src + ((size_t)zi * M + yi) * X + base[0];
                    float2 r0 = make_float2(0.f, 0.f), r1 = r0;
#pragma unroll
                    for (int jx = 0; jx < T; ++jx) {
                        const long long at = (row - src) + jx;
                        if (!TP_CHECK(dbg, at >= 0 && at < nsrc, 0)) continue;
                        const float2 v = __ldg(row + jx);
                        cfma(w[0][jx], v, r0);
                        if (DERIV) cfma(d[0][jx], v, r1);
                    }
                    cfma(w[1][jy], r0, ay);
                    if (DERIV) {
                        cfma(w[1][jy], r1, ayx);
                        cfma(d[1][jy], r0, ayy);
                    }
                }
                cfma(w[2][jz], ay, S);
                if (DERIV) {
                    cfma(w[2][jz], ayx, dS[0]);
                    cfma(w[2][jz], ayy, dS[1]);
                    cfma(d[2][jz], ay, dS[2]);
                }
            }
        } else {
#pragma unroll
            for (int jy = 0; jy < T; ++jy) {
                const int yi = wrap_row(base[1] + jy, M);
                const float2 *row = src + (size_t)yi * X + base[0];
                float2 r0 = make_float2(0.f, 0.f), r1 = r0;
#pragma unroll
                for (int jx = 0; jx < T; ++jx) {
                    const long long at = (row - src) + jx;
                    if (!TP_CHECK(dbg, at >= 0 && at < nsrc, 0)) continue;
                    const float2 v = __ldg(row + jx);
                    cfma(w[0][jx], v, r0);
                    if (DERIV) cfma(d[0][jx], v, r1);
                }
                cfma(w[1][jy], r0, S);
                if (DERIV) {
                    cfma(w[1][jy], r1, dS[0]);
                    cfma(d[1][jy], r0, dS[1]);
                }
            }
        }
    }

    // General path: per-tap Friedel reflection and range checks.
    __device__ __forceinline__ static void run_general(const float2 *__restrict__ src, int M, int X,
                                                       const int *x0, float (*w)[4], float (*d)[4],
                                                       float2 &S, float2 *dS, unsigned *dbg) {
        const int half = M >> 1;
        const int TZ = (D == 3) ? T : 1;
        for (int jz = 0; jz < TZ; ++jz) {
            for (int jy = 0; jy < T; ++jy) {
#pragma unroll
                for (int jx = 0; jx < T; ++jx) {
                    int nx = x0[0] - St::LO + jx;
                    int ny = x0[1] - St::LO + jy;
                    int nz = (D == 3) ? x0[2] - St::LO + jz : 0;
                    const bool cj = nx < 0;
                    if (cj) {
                        nx = -nx;
                        ny = -ny;
                        nz = -nz;
                    }
                    if (nx > half || !row_ok(ny, half) || (D == 3 && !row_ok(nz, half))) continue;
                    size_t e = (size_t)wrap_row(ny, M) * X + nx;
                    if (D == 3) e += (size_t)wrap_row(nz, M) * M * X;
                    if (!TP_CHECK(dbg, e < (size_t)(D == 3 ? M : 1) * M * X, 0)) continue;
                    float2 v = __ldg(src + e);
                    if (cj) v.y = -v.y;
                    const float wz = (D == 3) ? w[2][jz] : 1.0f;
                    const float wyz = w[1][jy] * wz;
                    cfma(w[0][jx] * wyz, v, S);
                    if (DERIV) {
                        cfma(d[0][jx] * wyz, v, dS[0]);
                        cfma(w[0][jx] * d[1][jy] * wz, v, dS[1]);
                        if constexpr (D == 3) cfma(w[0][jx] * w[1][jy] * d[2][jz], v, dS[2]);
                    }
                }
            }
        }
    }

    // Interpolated value at p (and its gradient when DERIV).
    __device__ __forceinline__ static void sample(const float2 *__restrict__ src, int M, int X,
                                                  const float *p, float2 &S, float2 *dS,
                                                  unsigned *dbg) {
        const int half = M >> 1;
        int x0[D];
        float w[D][4], d[D][4];
#pragma unroll
        for (int a = 0; a < D; ++a) {
            float t;
            x0[a] = split_coord(p[a], t);
            St::weights(t, w[a]);
            if (DERIV) St::derivs(t, d[a]);
        }
        S = make_float2(0.f, 0.f);
        if (DERIV)
#pragma unroll
            for (int a = 0; a < D; ++a) dS[a] = make_float2(0.f, 0.f);

        // All taps direct and stored?
        bool direct = (x0[0] - St::LO >= 0) && (x0[0] + St::HI <= half);
        // All taps Friedel-reflected and stored?
        bool friedel = (x0[0] + St::HI < 0) && (St::LO - x0[0] <= half);
#pragma unroll
        for (int a = 1; a < D; ++a) {
            direct = direct && (x0[a] - St::LO >= -half) && (x0[a] + St::HI < half);
            friedel = friedel && (-(x0[a] + St::HI) >= -half) && (St::LO - x0[a] < half);
        }
        if (direct) {
            int base[D];
#pragma unroll
            for (int a = 0; a < D; ++a) base[a] = x0[a] - St::LO;
            run_fast(src, M, X, base, w, d, S, dS, dbg);
        } else if (friedel) {
            // Tap n = x0 - LO + j reads conj(V[-n]); in storage order the
            // reflected taps run from -(x0 + HI) upwards with weights reversed.
            int base[D];
            float wr[D][4], dr[D][4];
#pragma unroll
            for (int a = 0; a < D; ++a) {
                base[a] = -(x0[a] + St::HI);
#pragma unroll
                for (int j = 0; j < T; ++j) {
                    wr[a][j] = w[a][T - 1 - j];
                    if (DERIV) dr[a][j] = d[a][T - 1 - j];
                }
            }
            run_fast(src, M, X, base, wr, dr, S, dS, dbg);
            S.y = -S.y;
            if (DERIV)
#pragma unroll
                for (int a = 0; a < D; ++a) dS[a].y = -dS[a].y;
        } else {
            run_general(src, M, X, x0, w, d, S, dS, dbg);
        }
    }
};

template <int D, bool CUBIC>
__global__ void __launch_bounds__(kThreads) k_project(Params q, float2 *__restrict__ out) {
    const int bp = blockIdx.x / q.tiles;
    const int rem = (blockIdx.x - bp * q.tiles) * kThreads + threadIdx.x;
    if (rem >= q.plane) return;
    const int b = bp / q.P;
    const int pi = bp - b * q.P;
    const int iy = rem / q.Xo;
    const int kx = rem - iy * q.Xo;
    const int ky = row_freq(iy, q.N);
    float2 *o = out + (size_t)bp * q.plane + rem;
    if (kx * kx + ky * ky > q.r2max) {
        *o = make_float2(0.f, 0.f);
        return;
    }
    const Pose<D> ps = load_pose<D>(q, b, pi);
    float p[D];
#pragma unroll
    for (int j = 0; j < D; ++j) p[j] = fmaf(ps.a[j], (float)kx, ps.b[j] * (float)ky);
    const float2 *src = q.src + (q.Bsrc == 1 ? 0 : (size_t)b * q.src_stride);
    float2 S;
    Gather<D, CUBIC, false>::sample(src, q.M, q.Xs, p, S, nullptr, q.dbg);
    if (q.shift) S = cmul(shift_phase(kx, ky, ps.sx, ps.sy, q.fN, q.invN), S);
    *o = S;
}

// dL/dR and dL/dshift.  Each block reduces its samples (all of one pose)
// and adds the partial sums into grad_rot / grad_shift with atomics.
template <int D, bool CUBIC>
__global__ void __launch_bounds__(kThreads) k_pose_grad(Params q, const float2 *__restrict__ g_out,
                                                        float *__restrict__ grad_rot,
                                                        float *__restrict__ grad_shift) {
    constexpr int NR = 2 * D;       // rows 0 and 1 of dL/dR (k_z = 0 leaves row 2 at zero)
    constexpr int NV = NR + 2;      // plus the two shift components
    const int bp = blockIdx.x / q.tiles;
    const int rem = (blockIdx.x - bp * q.tiles) * kThreads + threadIdx.x;
    const int b = bp / q.P;
    const int pi = bp - b * q.P;
    const Pose<D> ps = load_pose<D>(q, b, pi);
    float acc[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) acc[i] = 0.f;

    if (rem < q.plane) {
        const int iy = rem / q.Xo;
        const int kx = rem - iy * q.Xo;
        const int ky = row_freq(iy, q.N);
        if (kx * kx + ky * ky <= q.r2max) {
            float p[D];
#pragma unroll
            for (int j = 0; j < D; ++j) p[j] = fmaf(ps.a[j], (float)kx, ps.b[j] * (float)ky);
            const float2 *src = q.src + (q.Bsrc == 1 ? 0 : (size_t)b * q.src_stride);
            float2 S, dS[D];
            Gather<D, CUBIC, true>::sample(src, q.M, q.Xs, p, S, dS, q.dbg);
            const float2 g = __ldg(g_out + (size_t)bp * q.plane + rem);
            float2 ph = make_float2(1.f, 0.f);
            if (q.shift) ph = shift_phase(kx, ky, ps.sx, ps.sy, q.fN, q.invN);
            const float2 gp = cmul_conj_a(ph, g);   // conj(phase) * g
            // dL/dp_j = Re(conj(g) phase dS_j) = Re(conj(conj(phase) g) dS_j)
#pragma unroll
            for (int j = 0; j < D; ++j) {
                const float dl = gp.x * dS[j].x + gp.y * dS[j].y;
                acc[j] = q.s * (float)kx * dl;
                acc[D + j] = q.s * (float)ky * dl;
            }
            // dL/dt_a = (2 pi k_a / N) (g.re y.im - g.im y.re), y = phase * S
            const float2 y = cmul(ph, S);
            const float qv = 2.0f * 3.14159265358979f * q.invN * (g.x * y.y - g.y * y.x);
            acc[NR] = (float)kx * qv;
            acc[NR + 1] = (float)ky * qv;
        }
    }
    // Block reduction: warp shuffles, then one partial per warp in shared memory.
    __shared__ float red[kThreads / 32][NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        float v = acc[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        acc[i] = v;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0)
#pragma unroll
        for (int i = 0; i < NV; ++i) red[warp][i] = acc[i];
    __syncthreads();
    if (threadIdx.x < NV) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) v += red[w][threadIdx.x];
        const int i = threadIdx.x;
        if (!TP_CHECK(q.dbg, ps.ridx < q.Bp * q.P && ps.sidx < q.Bs * q.P, 9)) return;
        if (i < NR) {
            if (grad_rot) atomicAdd(grad_rot + (size_t)ps.ridx * D * D + i, v);
        } else if (grad_shift) {
            atomicAdd(grad_shift + 2 * (size_t)ps.sidx + (i - NR), v);
        }
    }
}

template <int D, bool CUBIC>
cudaError_t launch_project_t(const Params &q, float2 *out, cudaStream_t st) {
    const long long blocks = (long long)q.B * q.P * q.tiles;
    k_project<D, CUBIC><<<(unsigned)blocks, kThreads, 0, st>>>(q, out);
    return cudaGetLastError();
}

template <int D, bool CUBIC>
cudaError_t launch_pose_grad_t(const Params &q, const float2 *g, float *grot, float *gshift,
                               cudaStream_t st) {
    const long long blocks = (long long)q.B * q.P * q.tiles;
    k_pose_grad<D, CUBIC><<<(unsigned)blocks, kThreads, 0, st>>>(q, g, grot, gshift);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_project_2d(bool cubic, const Params &q, float2 *out, cudaStream_t st) {
    return cubic ? launch_project_t<2, true>(q, out, st) : launch_project_t<2, false>(q, out, st);
}

cudaError_t launch_pose_grad_2d(bool cubic, const Params &q, const float2 *g, float *grot,
                                float *gshift, cudaStream_t st) {
    return cubic ? launch_pose_grad_t<2, true>(q, g, grot, gshift, st)
                 : launch_pose_grad_t<2, false>(q, g, grot, gshift, st);
}

}  // namespace tp
