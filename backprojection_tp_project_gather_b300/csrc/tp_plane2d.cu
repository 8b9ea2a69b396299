// tp_plane2d.cu -- the 2D -> 2D forward projection and its rotation / shift
// gradients with the whole source plane staged in shared memory.
//
// A 2D half-spectrum of box M (M x (M/2+1) complex) is small enough that a
// thread block can hold its Friedel-completed "virtual" plane -- F(n) = V[n]
// for n_x >= 0, conj(V[-n]) for n_x < 0, zero outside the stored range
// [ar §2 "التمرير الأمامي"; ko §2 "Friedel 대칭성 처리"] -- over the stored
// columns and a strip of the Friedel side.  Every sample then reads its taps
// from shared memory on one branch-free path.
//
//  - Half plane.  The plane covers columns n_x in [-4, WX - 4) (WX the next
//    multiple of 4 of M/2 + 8) and rows n_y in [Y0, Y0 + WY) (Y0 = -(M/2 + 4),
//    WY the next multiple of 4 of M + 8), so a stencil (taps floor(p) - LO ..
//    floor(p) + HI) with p_x >= -2 that leaves the region lies wholly outside
//    the stored range and reads zero.  A sample with p_x < -2 is taken at -p:
//    all its taps lie at n_x <= -1, where F(n) = conj(F(-n)) holds by
//    construction, and the stencil weights are even, so S(p) = conj(S(-p))
//    and dS/dp(p) = -conj(dS/dp(-p)) exactly; its mirror's taps all lie at
//    n_x >= 1, away from the stored n_x = 0 column, which need not be
//    Hermitian.
//  - Layout.  The plane is cut into 4 x 4 tiles of 16 complex words (one
//    128-byte row of banks): element (x, y) sits in bank pair
//    (x mod 4) + 4 (y mod 4).  For cubic, lane L visits its 16 taps in its own
//    order -- at step (sx, sy) the tap in bank pair ((sx + L) mod 4) +
//    4 ((sy + L / 4) mod 4) -- so the 16 lanes of a half-warp never share a
//    bank pair and every 64-bit load takes the minimum two wavefronts.
//  - Staging.  A block holds two planes.  Each stored element of a source is
//    copied straight to its place in the tiled plane with an 8-byte
//    cp.async; once it landed, the three Friedel columns n_x = -1, -2, -3 are
//    filled from the plane itself.  Every other word is zero for every source
//    and is cleared once, at the start.  The copy of the block's NEXT source
//    image goes into the other plane before the current one is used, so it
//    lands while the block computes.
//  - Work.  The poses of each source image are cut into items; a persistent
//    block takes a contiguous range of items (consecutive items mostly share
//    their source, which then stays staged).  Threads take output pixels in
//    row order (coalesced reads of the upstream gradient and writes of the
//    output); pixels outside the radius are written as zeros by the forward.
//  - Phase.  The shift phase is separable, exp(-2 pi i (kx sx + ky sy) / N) =
//    exp(-2 pi i kx sx / N) exp(-2 pi i ky sy / N): per pose the block
//    tabulates both factors in shared memory (N/2 + 1 and N values, each from
//    the exactly period-reduced cycle count), and a pixel multiplies two
//    table entries instead of evaluating a sine and a cosine.
//
// The forward gives out = phase * S(p); with GRAD the same gather also forms
// the derivative weights and reduces, per pose, dL/dR[i][a] = s k_i dL/dp_a and
// dL/dshift_a (the analytic gradients of [de §3 item 4; ar §2]) over the block,
// adding them to grad_rot / grad_shift with one atomic per entry.  (The
// image gradient stays on the tiled scatter of tp_scatter.cu: accumulating
// into a shared plane measured slower there, with warps that own bands of
// rows stalled on the busiest band and with shared-memory atomics.)
//
// Method: "torch-projectors: A High-Performance Differentiable Projection
// Library for PyTorch", 2D -> 2D forward and its gradients [it §2 "Operazioni
// Supportate"; de §2 "Unterstützte Operationen" items 1 and 4].
#include <cstdint>

#include "tp_device.cuh"
#include "tp_launch.h"
#include "tp_tiles.cuh"

namespace tp {

namespace {

constexpr int kPlaneThreads = 512;
constexpr int kPlaneWarps = kPlaneThreads / 32;

// Geometry of the staged half plane of a box-M source.
constexpr int kPlaneX0 = -4;      // virtual column of local column 0
constexpr float kMirror = -2.0f;  // samples with p_x below this are taken at -p

struct PlaneGeo {
    int M, half, Xs;   // source box, M/2, M/2 + 1
    int Y0;            // virtual row of local row 0
    int WX, WY;        // local extents, multiples of 4
    int TWX;           // tiles per row (WX / 4)
    int words;         // complex words of one plane (WX * WY)
    int raw_words;     // complex words of one stored source image (M * Xs)
};

__host__ __device__ inline PlaneGeo plane_geo(int M) {
    PlaneGeo g;
    g.M = M;
    g.half = M / 2;
    g.Xs = M / 2 + 1;
    g.Y0 = -(M / 2 + 4);
    g.WX = ((M / 2 + 8) + 3) & ~3;
    g.WY = ((M + 8) + 3) & ~3;
    g.TWX = g.WX / 4;
    g.words = g.WX * g.WY;
    g.raw_words = M * g.Xs;
    return g;
}


// Shared memory of a launch: two planes and the phase tables (16-byte
// aligned: the plane words are a multiple of 16).
__host__ __device__ inline size_t plane_smem_bytes(int M, int N) {
    const PlaneGeo g = plane_geo(M);
    return sizeof(float2) * (2 * (size_t)g.words + (size_t)table_words(N));
}

// Tiled index of local element (lx, ly).
__device__ __forceinline__ int tidx(const PlaneGeo &g, int lx, int ly) {
    return ((ly >> 2) * g.TWX + (lx >> 2)) * 16 + (lx & 3) + 4 * (ly & 3);
}

// Quotient and remainder of e by d (e < 2^24, inv = 1/d rounded) without an
// integer division: the float quotient is off by at most one.
__device__ __forceinline__ int divmod(int e, int d, float inv, int &rem) {
    int quo = (int)((float)e * inv);
    int r = e - quo * d;
    if (r < 0) {
        --quo;
        r += d;
    } else if (r >= d) {
        ++quo;
        r -= d;
    }
    rem = r;
    return quo;
}

// Issue the copy of one stored source image (raw_words complex words at src,
// row-major M x Xs) into plane: element (r, x) goes to virtual (x, y) with
// y = r for r < M/2, r - M above.  One commit group.
__device__ __forceinline__ void issue_plane_copy(const PlaneGeo &g, const float2 *src,
                                                 float2 *plane, unsigned *dbg) {
    const unsigned sbase = (unsigned)__cvta_generic_to_shared(plane);
    int r, x;
    r = divmod(threadIdx.x, g.Xs, 1.0f / (float)g.Xs, x);
    const int dq = kPlaneThreads / g.Xs, dr = kPlaneThreads - dq * g.Xs;
    for (int e = threadIdx.x; e < g.raw_words; e += kPlaneThreads) {
        const int y = r < g.half ? r : r - g.M;
        const int at = tidx(g, x - kPlaneX0, y - g.Y0);
        if (TP_CHECK(dbg, at >= 0 && at < g.words, 1))
            asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(sbase + 8u * at),
                         "l"(src + e)
                         : "memory");
        x += dr;
        r += dq;
        if (x >= g.Xs) {
            x -= g.Xs;
            ++r;
        }
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

// The Friedel columns n_x = -1, -2, -3 of a landed plane: F(n) = conj(F(-n)),
// for the rows whose mirror -n_y is stored (-M/2 < n_y <= M/2); the other
// rows of these columns stay zero.
__device__ __forceinline__ void friedel_columns(const PlaneGeo &g, float2 *plane, unsigned *dbg) {
    for (int i = threadIdx.x; i < 3 * g.M; i += kPlaneThreads) {
        const int c = i / g.M;
        const int nx = -1 - c, ny = i - c * g.M - g.half + 1;   // ny in (-M/2, M/2]
        const int from = tidx(g, -nx - kPlaneX0, -ny - g.Y0), to = tidx(g, nx - kPlaneX0, ny - g.Y0);
        if (!TP_CHECK(dbg, from >= 0 && from < g.words && to >= 0 && to < g.words, 1)) continue;
        const float2 v = plane[from];
        plane[to] = make_float2(v.x, -v.y);
    }
}

// Weighted sum over the stencil of the sample at local tap origin (lx, ly)
// (the local coordinates of tap floor(p) - LO), with derivative weights when
// DERIV.  Cubic visits the taps in the lane-rotated order described above.
//
// At step sx a lane reads the tap whose x is (sx + lane) mod 4 (its
// residue rho); within [lx, lx + 3] that is x = 4 ((lx + 3 - rho) >> 2) + rho,
// so the tiled x offset is 16 ((lx + 3 - rho) >> 2) + rho, and likewise in y
// with the residue (sy + lane / 4) mod 4.  The residues are the lane's own
// and are passed in precomputed.
struct LaneRes {
    int rx[4], ry[4];   // tap residues of the steps
};

__device__ __forceinline__ LaneRes lane_residues() {
    LaneRes r;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        r.rx[i] = (i + lane) & 3;
        r.ry[i] = (i + (lane >> 2)) & 3;
    }
    return r;
}

template <bool CUBIC, bool DERIV>
__device__ __forceinline__ void gather_plane(const PlaneGeo &g, const LaneRes &res,
                                             const float2 *plane, int lx, int ly,
                                             const float (&w)[2][4], const float (&d)[2][4],
                                             float2 &S, float2 (&dS)[2], unsigned *dbg) {
    S = make_float2(0.f, 0.f);
    dS[0] = dS[1] = S;
    const int total = g.words;
    if constexpr (CUBIC) {
        const int lane = threadIdx.x & 31;
        const int cx = (lane - lx) & 3, cy = ((lane >> 2) - ly) & 3;
        float wx[4], wy[4], dx[4], dy[4];
        rot4(w[0], cx, wx);   // the separable weights follow the tap order
        rot4(w[1], cy, wy);
        if (DERIV) {
            rot4(d[0], cx, dx);
            rot4(d[1], cy, dy);
        }
        int ox[4], oy[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            ox[i] = ((lx + 3 - res.rx[i]) >> 2) * 16 + res.rx[i];
            oy[i] = ((ly + 3 - res.ry[i]) >> 2) * (16 * g.TWX) + 4 * res.ry[i];
        }
#pragma unroll
        for (int sy = 0; sy < 4; ++sy) {
            float2 r0 = make_float2(0.f, 0.f), r1 = r0;
#pragma unroll
            for (int sx = 0; sx < 4; ++sx) {
                const int at = oy[sy] + ox[sx];
                if (!TP_CHECK(dbg, at >= 0 && at < total, 2)) continue;
                const float2 v = plane[at];
                cfma(wx[sx], v, r0);
                if (DERIV) cfma(dx[sx], v, r1);
            }
            cfma(wy[sy], r0, S);
            if (DERIV) {
                cfma(wy[sy], r1, dS[0]);
                cfma(dy[sy], r0, dS[1]);
            }
        }
    } else {
#pragma unroll
        for (int jy = 0; jy < 2; ++jy) {
            float2 r0 = make_float2(0.f, 0.f), r1 = r0;
#pragma unroll
            for (int jx = 0; jx < 2; ++jx) {
                const int at = tidx(g, lx + jx, ly + jy);
                if (!TP_CHECK(dbg, at >= 0 && at < total, 2)) continue;
                const float2 v = plane[at];
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

// Work items: item i covers source v = i / per_src and the poses
// [c * chunk, min((c + 1) * chunk, pps)) of that source's pose list, c = i % per_src.
struct Items {
    int per_src;   // items per source image
    int chunk;     // poses per item
    int pps;       // poses per source: B * P when the source is shared, else P
    int count;     // Bsrc * per_src
};

// Output-image index of pose j of source v's pose list.
__device__ __forceinline__ int image_of(const Params &q, int v, int j) {
    return (q.Bsrc == 1) ? j : v * q.P + j;
}

// Stencil of the pixel (kx, ky) of pose ps: local tap origin and weights,
// at -p when p_x < kMirror (mir; the caller conjugates what it gathers).
// Returns false when the stencil leaves the staged region, i.e. lies wholly
// outside the stored range.
template <bool CUBIC, bool DERIV>
__device__ __forceinline__ bool stencil_at(const PlaneGeo &g, const Pose<2> &ps, int kx, int ky,
                                           int &lx, int &ly, bool &mir, float (&w)[2][4],
                                           float (&d)[2][4]) {
    using St = Stencil<CUBIC>;
    float t;
    float px = fmaf(ps.a[0], (float)kx, ps.b[0] * (float)ky);
    float py = fmaf(ps.a[1], (float)kx, ps.b[1] * (float)ky);
    mir = px < kMirror;
    if (mir) {
        px = -px;
        py = -py;
    }
    lx = split_coord(px, t) - St::LO - kPlaneX0;
    St::weights(t, w[0]);
    if (DERIV) St::derivs(t, d[0]);
    ly = split_coord(py, t) - St::LO - g.Y0;
    St::weights(t, w[1]);
    if (DERIV) St::derivs(t, d[1]);
    constexpr int span = St::LO + St::HI + 1;
    return (unsigned)lx <= (unsigned)(g.WX - span) && (unsigned)ly <= (unsigned)(g.WY - span);
}

template <bool CUBIC, bool GRAD>
__global__ void __launch_bounds__(kPlaneThreads, 1)
    k_plane2d(Params q, Items it, float2 *__restrict__ out,
              const float2 *__restrict__ g_out, float *__restrict__ grad_rot,
              float *__restrict__ grad_shift) {
    extern __shared__ float4 s_plane4[];
    __shared__ float s_red[kPlaneWarps][6];
    const PlaneGeo g = plane_geo(q.M);
    float2 *planes = reinterpret_cast<float2 *>(s_plane4);   // two planes
    float2 *phx = planes + 2 * (size_t)g.words;
    float2 *phy = phx + q.Xo;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int first = (int)((long long)it.count * blockIdx.x / gridDim.x);
    const int last = (int)((long long)it.count * (blockIdx.x + 1) / gridDim.x);
    if (first >= last) return;
    // The words no copy writes are zero for every source: clear both planes once.
    for (int i = threadIdx.x; i < g.words; i += kPlaneThreads)   // 2 planes = g.words float4
        s_plane4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    const int npix = q.N * q.Xo;
    const LaneRes res = lane_residues();
    // Pixel e = threadIdx.x + k * kPlaneThreads as (row, column), advanced
    // without a division: the stride is dq rows and dr columns.
    int iy0, kx0;
    iy0 = divmod(threadIdx.x, q.Xo, 1.0f / (float)q.Xo, kx0);
    const int dq = kPlaneThreads / q.Xo, dr = kPlaneThreads - dq * q.Xo;
    int staged = -1;   // source held in plane `cur`
    int cur = 0;       // plane receiving (then holding) the next source
    issue_plane_copy(g, q.src + (size_t)(first / it.per_src) * q.src_stride, planes, q.dbg);
    const float2 *plane = planes;
    for (int i = first; i < last; ++i) {
        const int v = i / it.per_src;
        if (v != staged) {
            // Sources come in increasing order and the copy in flight is
            // always the next one's, into plane `cur`.
            asm volatile("cp.async.wait_group 0;\n" ::: "memory");
            __syncthreads();   // landed for every thread; the other plane is no longer read
            friedel_columns(g, planes + (size_t)cur * g.words, q.dbg);
            plane = planes + (size_t)cur * g.words;
            staged = v;
            __syncthreads();   // plane complete
            // Prefetch the next different source into the other plane.
            for (int k = i + 1; k < last; ++k)
                if (k / it.per_src != v) {
                    cur ^= 1;
                    issue_plane_copy(g, q.src + (size_t)(k / it.per_src) * q.src_stride,
                                     planes + (size_t)cur * g.words, q.dbg);
                    break;
                }
        }
        const int c = i - v * it.per_src;
        const int j1 = min((c + 1) * it.chunk, it.pps);
        for (int j = c * it.chunk; j < j1; ++j) {
            const int bp = image_of(q, v, j);
            const int b = bp / q.P, pi = bp - b * q.P;
            const Pose<2> ps = load_pose<2>(q, b, pi);
            if (q.shift) {
                __syncthreads();   // the previous pose's tables are no longer read
                phase_tables(q, ps.sx, ps.sy, phx, phy);
                __syncthreads();
            }
            float acc[6];
#pragma unroll
            for (int k = 0; k < 6; ++k) acc[k] = 0.f;
            const size_t ob = (size_t)bp * q.plane;
            int iy = iy0, kx = kx0;
            for (int e = threadIdx.x; e < npix; e += kPlaneThreads) {
                const int ry = iy, rx = kx;
                kx += dr;
                iy += dq;
                if (kx >= q.Xo) {
                    kx -= q.Xo;
                    ++iy;
                }
                const int ky = row_freq(ry, q.N);
                if (rx * rx + ky * ky > q.r2max) {
                    if (!GRAD) out[ob + e] = make_float2(0.f, 0.f);
                    continue;
                }
                float2 gv = make_float2(0.f, 0.f);
                if (GRAD) gv = __ldg(g_out + ob + e);   // in flight during the gather
                float w[2][4], d[2][4];
                int lx, ly;
                bool mir;
                float2 S = make_float2(0.f, 0.f), dS[2] = {S, S};
                if (stencil_at<CUBIC, GRAD>(g, ps, rx, ky, lx, ly, mir, w, d)) {
                    gather_plane<CUBIC, GRAD>(g, res, plane, lx, ly, w, d, S, dS, q.dbg);
                    if (mir) {   // S(p) = conj(S(-p)), dS/dp(p) = -conj(dS/dp(-p))
                        S.y = -S.y;
                        dS[0].x = -dS[0].x;
                        dS[1].x = -dS[1].x;
                    }
                }
                const float2 ph = q.shift ? cmul(phx[rx], phy[ry]) : make_float2(1.f, 0.f);
                if (!GRAD) {
                    out[ob + e] = cmul(ph, S);
                } else {
                    const float2 gq = cmul_conj_a(ph, gv);   // conj(phase) * g
#pragma unroll
                    for (int a = 0; a < 2; ++a) {
                        const float dl = gq.x * dS[a].x + gq.y * dS[a].y;   // dL/dp_a
                        acc[a] = fmaf(q.s * (float)rx, dl, acc[a]);
                        acc[2 + a] = fmaf(q.s * (float)ky, dl, acc[2 + a]);
                    }
                    const float2 y = cmul(ph, S);
                    const float qv = 6.283185307179586f * q.invN * (gv.x * y.y - gv.y * y.x);
                    acc[4] = fmaf((float)rx, qv, acc[4]);
                    acc[5] = fmaf((float)ky, qv, acc[5]);
                }
            }
            if (GRAD) {
#pragma unroll
                for (int k = 0; k < 6; ++k) {
                    float x = acc[k];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                    if (lane == 0) s_red[warp][k] = x;
                }
                __syncthreads();
                if (threadIdx.x < 6) {
                    float x = 0.f;
#pragma unroll
                    for (int w2 = 0; w2 < kPlaneWarps; ++w2) x += s_red[w2][threadIdx.x];
                    const int k = threadIdx.x;
                    if (TP_CHECK(q.dbg, ps.ridx < q.Bp * q.P && ps.sidx < q.Bs * q.P, 9)) {
                        if (k < 4) {
                            if (grad_rot && x != 0.f) atomicAdd(grad_rot + (size_t)ps.ridx * 4 + k, x);
                        } else if (grad_shift && x != 0.f) {
                            atomicAdd(grad_shift + 2 * (size_t)ps.sidx + (k - 4), x);
                        }
                    }
                }
                __syncthreads();   // s_red is reused by the next pose
            }
        }
    }
    // Leave no copy in flight (a prefetch is only issued for an item that follows).
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

int sm_count() {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

Items make_items(const Params &q, int blocks_target) {
    Items it;
    it.pps = (q.Bsrc == 1) ? q.B * q.P : q.P;
    // About two items per block, never an item smaller than one pose.
    const long long want = 2LL * blocks_target;
    const long long per_src = (want + q.Bsrc - 1) / q.Bsrc;
    it.chunk = (int)((it.pps + per_src - 1) / per_src);
    if (it.chunk < 1) it.chunk = 1;
    it.per_src = (it.pps + it.chunk - 1) / it.chunk;
    it.count = q.Bsrc * it.per_src;
    return it;
}

template <bool CUBIC, bool GRAD>
cudaError_t plane_launch(const Params &q, float2 *out, const float2 *g, float *grot, float *gshift,
                         cudaStream_t st) {
    if ((long long)q.B * q.P == 0) return cudaSuccess;
    const size_t smem = plane_smem_bytes(q.M, q.N);
    auto kern = k_plane2d<CUBIC, GRAD>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int sms = sm_count();
    const Items it = make_items(q, sms);
    const int blocks = it.count < sms ? it.count : sms;
    kern<<<blocks, kPlaneThreads, smem, st>>>(q, it, out, g, grot, gshift);
    return cudaGetLastError();
}

}  // namespace

bool plane2d_fits(int M, int N) {
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return false;
    // The static reduction array and a margin for the runtime's own use.
    return plane_smem_bytes(M, N) + 1024 <= (size_t)optin;
}

cudaError_t launch_plane2d_project(bool cubic, const Params &q, float2 *out, cudaStream_t st) {
    return cubic ? plane_launch<true, false>(q, out, nullptr, nullptr, nullptr, st)
                 : plane_launch<false, false>(q, out, nullptr, nullptr, nullptr, st);
}

cudaError_t launch_plane2d_pose_grad(bool cubic, const Params &q, const float2 *grad_out,
                                     float *grad_rot, float *grad_shift, cudaStream_t st) {
    if (!grad_rot && !grad_shift) return cudaSuccess;
    return cubic ? plane_launch<true, true>(q, nullptr, grad_out, grad_rot, grad_shift, st)
                 : plane_launch<false, true>(q, nullptr, grad_out, grad_rot, grad_shift, st);
}

}  // namespace tp
