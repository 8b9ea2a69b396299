// tp_device.cuh -- device-side building blocks shared by the gather and
// scatter kernels: launch parameters, interpolation stencils, half-spectrum
// addressing and the shift phase.
//
// Method: "torch-projectors: A High-Performance Differentiable Projection
// Library for PyTorch" (summary pages; [it §2] = Italian page, technical
// summary section 2, and so on).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tp {

// Threads per block of the per-sample kernels (gather, pose gradient,
// scatter); the host sizes Params::tiles with it.
constexpr int kSampleBlock = 256;

// Everything a projection kernel needs, passed by value.
struct Params {
    const float2 *src;     // source spectrum (volume or image), batch-major
    long long src_stride;  // complex elements per source batch element
    int Bsrc;              // source batch (1 = shared)
    int M;                 // source box
    int Xs;                // M/2 + 1
    const float *rot;      // (Bp, P, D, D) row-major
    int Bp;
    const float *shift;    // (Bs, P, 2) or nullptr
    int Bs;
    int P;                 // poses per batch element
    int B;                 // batch
    int N;                 // output box
    int Xo;                // N/2 + 1
    int plane;             // N * Xo
    int tiles;             // thread blocks per output plane
    float s;               // oversampling factor
    float fN;              // N as a float
    float invN;            // 1 / N
    int r2max;             // pixels with kx^2 + ky^2 > r2max are outside the radius
    unsigned mplane, mxo;  // floor(2^32 / plane), floor(2^32 / Xo): see udiv
    unsigned *dbg;         // bounds-check word of a TP_DEBUG_BOUNDS build, else null
};

// Bounds checks of the debug build (nvcc -DTP_DEBUG_BOUNDS): TP_CHECK(dbg,
// cond, bit) is cond, and when cond is false it also sets bit `bit` of the
// word *dbg, so that the access it guards is skipped and the host can read
// which kind of index went out of range (tp_debug_bounds_word).  In the
// normal build it is the constant true and cond is not evaluated (only named
// in a sizeof, so that the variables it alone uses stay referenced).  Bits:
// 0 source spectrum read (staging or direct gather), 1 staging destination,
// 2 staged gather taps, 3 output rows,
// 4 scatter tile, 5 weight tile, 6 fold target, 7 image read, 8 workspace
// lists (units, masks, poses), 9 rotation / shift gradient rows, 10 saved
// derivative or weight-gradient rows.
#ifdef TP_DEBUG_BOUNDS
__device__ __forceinline__ bool flag_bound(unsigned *dbg, int bit) {
    if (dbg) atomicOr(dbg, 1u << bit);
    return false;
}
#define TP_CHECK(dbg, cond, bit) ((cond) || ::tp::flag_bound((dbg), (bit)))
#else
#define TP_CHECK(dbg, cond, bit) (sizeof(cond) > 0)
#endif

// ---------------------------------------------------------------------------
// Stencils [it §2 "Interpolazione"; ko §2 "보간법"; ar §2].
//
// Catmull-Rom is Keys' cubic convolution kernel with a = -1/2.  For a
// sample at x0 + t (t in [0, 1)) its four taps x0-1 .. x0+2 sit at distances
// 1+t, t, 1-t, 2-t; expanding the kernel's two branches there gives the
// polynomials below (and their derivatives in t, which equal d/dp).
template <bool CUBIC>
struct Stencil;

template <>
struct Stencil<true> {
    static constexpr int TAPS = 4;
    static constexpr int LO = 1;   // first tap is x0 - LO
    static constexpr int HI = 2;   // last tap is x0 + HI
    __device__ __forceinline__ static void weights(float t, float w[4]) {
        const float u = 1.0f - t;
        w[0] = -0.5f * t * u * u;
        w[1] = (1.5f * t - 2.5f) * t * t + 1.0f;
        w[2] = (1.5f * u - 2.5f) * u * u + 1.0f;
        w[3] = -0.5f * u * t * t;
    }
    __device__ __forceinline__ static void derivs(float t, float d[4]) {
        const float u = 1.0f - t;
        d[0] = -0.5f * u * (1.0f - 3.0f * t);
        d[1] = (4.5f * t - 5.0f) * t;
        d[2] = -(4.5f * u - 5.0f) * u;
        d[3] = -0.5f * t * (2.0f - 3.0f * t);
    }
};

// Multilinear: taps x0, x0+1 with weights 1-t, t.  The derivative is the
// one of the branch on [x0, x0+1), also at integer positions.
template <>
struct Stencil<false> {
    static constexpr int TAPS = 2;
    static constexpr int LO = 0;
    static constexpr int HI = 1;
    __device__ __forceinline__ static void weights(float t, float w[2]) {
        w[0] = 1.0f - t;
        w[1] = t;
    }
    __device__ __forceinline__ static void derivs(float, float d[2]) {
        d[0] = -1.0f;
        d[1] = 1.0f;
    }
};

// Sample coordinate split into tap origin x0 = floor(p) and fraction t.  p is
// first clamped to +-2^20 so that a huge or non-finite coordinate (any
// matrix is accepted) cannot overflow the tap arithmetic; such a coordinate
// lies far outside every stored spectrum, so all of its taps read zero.
__device__ __forceinline__ int split_coord(float p, float &t) {
    const float pc = fminf(fmaxf(p, -1048576.0f), 1048576.0f);
    const float f = floorf(pc);
    t = pc - f;
    return (int)f;
}

// n / d for n < 2^31 and d >= 2, given m = floor(2^32 / d): umulhi(n, m) is
// n / d or one less (m underestimates 2^32 / d by less than one, n by less
// than 2^32), and one comparison of the remainder corrects it.
__device__ __forceinline__ unsigned udiv(unsigned n, unsigned d, unsigned m) {
    unsigned qt = __umulhi(n, m);
    if (n - qt * d >= d) ++qt;
    return qt;
}

// Row of frequency f (valid for -M/2 <= f < M/2) in rfftn order.
__device__ __forceinline__ int wrap_row(int f, int M) { return f < 0 ? f + M : f; }

__device__ __forceinline__ bool row_ok(int f, int half) { return f >= -half && f < half; }

// Frequency of output row iy.
__device__ __forceinline__ int row_freq(int iy, int N) { return iy < (N >> 1) ? iy : iy - N; }

// exp(-2 pi i (kx sx + ky sy) / N) [de §2 "Interpolation"; ar §2].
//
// The phase is formed from the fractional part of the cycle count k * sh / N
// with one rounding error: k * sh is split exactly into hi + lo (fmaf returns
// the rounding error of the product), whole periods of N are removed from hi
// exactly (q * N is an integer and the remainder is representable), and only
// the remainder, at most about N/2 in size, is divided by N.  This keeps
// shifts of hundreds of pixels at high frequency accurate in fp32.
__device__ __forceinline__ float frac_cycles(int k, float sh, float N, float invN) {
    const float kf = (float)k;
    const float hi = kf * sh;
    const float lo = fmaf(kf, sh, -hi);
    const float qn = rintf(hi * invN);
    const float r = fmaf(-qn, N, hi);
    return (r + lo) * invN;
}

__device__ __forceinline__ float2 shift_phase(int kx, int ky, float sx, float sy, float N,
                                              float invN) {
    const float c = frac_cycles(kx, sx, N, invN) + frac_cycles(ky, sy, N, invN);
    float sn, cs;
    sincospif(-2.0f * c, &sn, &cs);
    return make_float2(cs, sn);
}

__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
    return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}

__device__ __forceinline__ float2 cmul_conj_a(float2 a, float2 b) {  // conj(a) * b
    return make_float2(a.x * b.x + a.y * b.y, a.x * b.y - a.y * b.x);
}

// acc += w v for a real weight and a complex value: one packed two-lane FMA
// (both lanes fused, so the result equals two fmaf calls bit for bit).
__device__ __forceinline__ void cfma(float w, float2 v, float2 &acc) {
    acc = __ffma2_rn(make_float2(w, w), v, acc);
}

// Do any two of the G samples of a spreading round share a tile word?  Lane
// group g (lanes g * lanes .. g * lanes + lanes - 1) holds its sample's tile
// coordinates packed one per byte (x | y << 8 | z << 16), or kFarAway when
// it has no sample; two stencils of `taps` taps per axis meet iff the
// coordinates differ by less than `taps` on every axis.  The groups'
// coordinates are exchanged with shuffles, which cost far less than a warp
// match on the tap words.  Call with the whole warp.
constexpr int kFarAway = 0x00404040;

template <int G, int AXES>
__device__ __forceinline__ bool stencils_meet(int mine, int lanes, int taps) {
    bool meet = false;
#pragma unroll
    for (int k = 1; k < G; ++k) {
        const int other = __shfl_xor_sync(0xffffffffu, mine, k * lanes);
        bool all = mine != kFarAway;
#pragma unroll
        for (int a = 0; a < AXES; ++a) {
            const int d = ((mine >> (8 * a)) & 0xff) - ((other >> (8 * a)) & 0xff);
            all = all && d < taps && d > -taps;
        }
        meet = meet || all;
    }
    return __any_sync(0xffffffffu, meet);
}

// Per-pose geometry, loaded once per thread block.
template <int D>
struct Pose {
    float a[D];   // s * R[0][:]  (p = a*kx + b*ky)
    float b[D];   // s * R[1][:]
    float sx, sy;
    int ridx;     // index of the pose in rot  (for gradients)
    int sidx;     // index of the pose in shift
};

template <int D>
__device__ __forceinline__ Pose<D> load_pose(const Params &q, int b, int pi) {
    Pose<D> ps;
    ps.ridx = ((q.Bp == 1) ? 0 : b) * q.P + pi;
    const float *R = q.rot + (size_t)ps.ridx * D * D;
#pragma unroll
    for (int j = 0; j < D; ++j) {
        ps.a[j] = q.s * __ldg(R + j);
        ps.b[j] = q.s * __ldg(R + D + j);
    }
    ps.sidx = ((q.Bs == 1) ? 0 : b) * q.P + pi;
    if (q.shift) {
        ps.sx = __ldg(q.shift + 2 * (size_t)ps.sidx);
        ps.sy = __ldg(q.shift + 2 * (size_t)ps.sidx + 1);
    } else {
        ps.sx = ps.sy = 0.0f;
    }
    return ps;
}

}  // namespace tp
