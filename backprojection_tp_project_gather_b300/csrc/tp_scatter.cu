// tp_scatter.cu -- the scatter side of the 2D operators: the image gradient
// of the 2D -> 2D projection (its real adjoint applied to an upstream
// gradient).  Each in-radius sample spreads w * conj(phase) * g over its
// stencil; Friedel taps (n_x < 0) add the conjugate at -n, which makes this
// the exact real adjoint of the gather in tp_gather.cu.  The 3D scatters are
// the brick kernels of tp_brick.cu.
//
// Method: "torch-projectors: A High-Performance Differentiable Projection
// Library for PyTorch", 2D -> 2D backward [de §2 item 4; it §2 "Operazioni
// Supportate"]; the pages name global atomics as the cost of the scatter
// [it §4 "Backward Pass"], which the tiles below avoid.
#include "tp_device.cuh"
#include "tp_launch.h"
#include "tp_tiles.cuh"

namespace tp {

namespace {

// ---------------------------------------------------------------------------
// 2D image gradient without per-tap global atomics.
//
// The 2D half-spectrum is viewed as the Friedel-completed virtual plane
// (F(n) = V[n] for n_x >= 0, conj(V[-n]) for n_x < 0, zero outside the
// stored range) and cut into kTile x kTile tiles.  A sample belongs to the
// tile that holds floor(p), so its stencil lies in the tile plus a halo of
// LO + HI.  kSplit blocks per output image, each with an interleaved quarter
// of its tiles; a block's warps take their tiles from a counter in shared
// memory.  A warp enumerates the image's pixels
// whose sample position falls in its tile (rows from the inverse of
// [a b], each row's qx interval from the two slab constraints, a warp
// prefix sum packing the candidates into 32-lane rounds) and spreads the
// owned ones into a private tile with plain read-add-write.  Cubic: each lane
// spreads its own sample's 16 taps in a lane-rotated order that keeps the 16
// lanes of a half-warp on 16 different words; each half-warp has a tile of its
// own, so both spread at once, and the fold adds the two.  Linear: owned
// samples are queued and tap lanes (jx, jy) spread
// several samples per round, one at a time in a round where two of their
// stencils meet (stencils_meet).  The tile is then added to the stored
// half-spectrum with one vector atomic per touched word (Friedel positions
// conjugated at -n).  With a shift (and N <= kMaxTableN) the block first
// tabulates the two separable factors of the pose's phase, and a sample
// multiplies two entries instead of evaluating a sine and a cosine.
constexpr int kTile = 16;
constexpr int kMaxTableN = 1024;
constexpr int kTileWarps = 4;
constexpr int kSplit = 4;   // blocks per image: shorter blocks, a smaller last wave
constexpr float kTileMargin = 0.01f;

// The warp's tile.  Cubic: 20 x 20 words in 4 x 4 tiles of 16 complex words,
// so word (x, y) sits in bank pair (x mod 4) + 4 (y mod 4), one tile per
// half-warp.  Linear: row-major 17 x 18 (x pitch 18).
template <bool CUBIC>
struct Tile2 {
    using St = Stencil<CUBIC>;
    static constexpr int S = kTile + St::LO + St::HI;  // staged edge (19 or 17)
    static constexpr int PX = CUBIC ? 20 : 18;          // x extent (pitch)
    static constexpr int ELEMS = (CUBIC ? 20 : S) * PX;
    static constexpr int LANES = St::TAPS * St::TAPS;   // lanes per linear sample
    // Linear spreads eight samples per round, drawn R slots apart, whose 2 x 2
    // stencils rarely meet; a round in which two of them do is spread one
    // sample at a time.
    static constexpr int SPS = 32 / LANES;
    static constexpr int COPIES = CUBIC ? 2 : 1;          // tiles per warp
    static constexpr size_t TILE_BYTES = sizeof(float2) * ELEMS * COPIES;
    static constexpr size_t QUEUE_BYTES = CUBIC ? 0 : sizeof(float) * 32 * 9 + sizeof(float4) * 32;
    static constexpr size_t WARP_BYTES = TILE_BYTES + QUEUE_BYTES;
    static_assert(TILE_BYTES % 16 == 0, "16-byte aligned queue");
    __device__ __forceinline__ static int index(int x, int y) {
        if (CUBIC) return ((y >> 2) * (PX / 4) + (x >> 2)) * 16 + (x & 3) + 4 * (y & 3);
        return y * PX + x;
    }
};

// Linear: queued samples of a warp.
struct Queue2 {
    float w[32][9];   // per sample: wx (4), wy (4), unused
    float4 rec[32];   // per sample: conj(phase) * g (re, im), tile x | y << 8, first tap
};

template <bool CUBIC>
__global__ void __launch_bounds__(32 * kTileWarps) k_scatter2d_tiles(Params q,
                                                                    const float2 *__restrict__ img,
                                                                    float2 *__restrict__ dst,
                                                                    bool tables) {
    using T = Tile2<CUBIC>;
    using St = Stencil<CUBIC>;
    extern __shared__ float4 s_t2[];
    __shared__ int s_next;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    char *mine = reinterpret_cast<char *>(s_t2) + warp * T::WARP_BYTES;
    float2 *acc = reinterpret_cast<float2 *>(mine);
    Queue2 &Q = *reinterpret_cast<Queue2 *>(mine + T::TILE_BYTES);   // linear only
    const int grp = lane / T::LANES, jx = lane % St::TAPS, jy = (lane / St::TAPS) % St::TAPS;
    const int toff = jx + T::PX * jy;
    // Cubic: this lane's tap residues per step (see the spreading below).
    int rx[4], ry[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        rx[i] = (i + lane) & 3;
        ry[i] = (i + (lane >> 2)) & 3;
    }

    // kSplit blocks per image, block s taking the image's tiles s, s + kSplit, ...
    const int bp = blockIdx.x / kSplit, sub = blockIdx.x - bp * kSplit;
    const int b = bp / q.P, pi = bp - b * q.P;
    const Pose<2> ps = load_pose<2>(q, b, pi);
    const float a0 = ps.a[0], a1 = ps.a[1], b0 = ps.b[0], b1 = ps.b[1];   // p = a qx + b qy
    const float det = a0 * b1 - a1 * b0;
    const float aa = a0 * a0 + a1 * a1, bb = b0 * b0 + b1 * b1, ab = a0 * b0 + a1 * b1;
    const bool degenerate = !(fabsf(det) > 1e-6f * (aa + bb)) || !(aa > 0.f);
    const float id = degenerate ? 0.f : 1.0f / det;
    const float u0 = -a1 * id, u1 = a0 * id;   // qy = u . p
    const float v0 = b1 * id, v1 = -b0 * id;   // qx = v . p
    const float ia0 = fabsf(a0) > 1e-6f ? 1.0f / a0 : 0.f, ia1 = fabsf(a1) > 1e-6f ? 1.0f / a1 : 0.f;
    const float hs = 0.5f * (aa + bb), hd = 0.5f * (aa - bb);
    const float reach = sqrtf((hs + sqrtf(hd * hd + ab * ab)) * (float)q.r2max) * 1.001f + 0.01f;
    const int half = q.M >> 1, nhalf = q.N >> 1;
    const int rmax = (int)floorf(sqrtf((float)q.r2max));
    // Tiles whose floor(p) positions can have a tap in the stored range.
    const int tlo = (int)floorf((float)(-half - St::HI) / kTile);
    const int thi = (int)floorf((float)(half + St::LO) / kTile);
    const int nt = thi - tlo + 1;
    const float2 *gimg = img + (size_t)bp * q.plane;
    float2 *V = dst + (q.Bsrc == 1 ? (size_t)0 : (size_t)b * q.src_stride);
    const float sx = ps.sx, sy = ps.sy;
    float2 *phx = reinterpret_cast<float2 *>(reinterpret_cast<char *>(s_t2) + kTileWarps * T::WARP_BYTES);
    float2 *phy = phx + q.Xo;
    if (tables) phase_tables(q, sx, sy, phx, phy);   // read after the barrier below

    for (int e = lane; e < T::ELEMS * T::COPIES; e += 32) acc[e] = make_float2(0.f, 0.f);
    float2 *const mytile = acc + (T::COPIES == 2 ? (lane >> 4) * T::ELEMS : 0);   // this half-warp's tile
    if (threadIdx.x == 0) s_next = 0;
    __syncthreads();
    for (;;) {
        int t = 0;
        if (lane == 0) t = atomicAdd(&s_next, 1);
        t = __shfl_sync(0xffffffffu, t, 0) * kSplit + sub;
        if (t >= nt * nt) break;
        const int ox = (tlo + t % nt) * kTile, oy = (tlo + t / nt) * kTile;
        const float lo0 = (float)ox - kTileMargin, hi0 = (float)(ox + kTile) + kTileMargin;
        const float lo1 = (float)oy - kTileMargin, hi1 = (float)(oy + kTile) + kTileMargin;
        const float c0 = 0.5f * (lo0 + hi0), c1 = 0.5f * (lo1 + hi1), h = 0.5f * (hi0 - lo0);
        {   // can an in-radius sample of this pose land in the tile?
            const float e0 = fmaxf(fabsf(c0) - h, 0.f), e1 = fmaxf(fabsf(c1) - h, 0.f);
            if (e0 * e0 + e1 * e1 > reach * reach) continue;
            if (!degenerate && v0 * c0 + v1 * c1 + h * (fabsf(v0) + fabsf(v1)) < -0.01f) continue;
        }
        int qy0, qy1;
        if (degenerate) {
            qy0 = -nhalf;
            qy1 = nhalf - 1;
        } else {
            const float m = u0 * c0 + u1 * c1, e = h * (fabsf(u0) + fabsf(u1));
            qy0 = max((int)ceilf(fmaxf(m - e - 0.01f, -1e7f)), -nhalf);
            qy1 = min((int)floorf(fminf(m + e + 0.01f, 1e7f)), nhalf - 1);
        }
        qy0 = max(qy0, -rmax);
        qy1 = min(qy1, rmax);
        bool touched = false;
        for (int base = qy0; base <= qy1; base += 32) {
            const int qy = base + lane;
            int xs = 0, cnt = 0;
            if (qy <= qy1) {
                float xl = 0.f, xh = (float)nhalf;
                bool empty = false;
                const float bd0 = (float)qy * b0, bd1 = (float)qy * b1;
                if (ia0 != 0.f) {
                    const float t1 = (lo0 - bd0) * ia0, t2 = (hi0 - bd0) * ia0;
                    xl = fmaxf(xl, fminf(t1, t2));
                    xh = fminf(xh, fmaxf(t1, t2));
                } else if (bd0 < lo0 || bd0 > hi0) {
                    empty = true;
                }
                if (ia1 != 0.f) {
                    const float t1 = (lo1 - bd1) * ia1, t2 = (hi1 - bd1) * ia1;
                    xl = fmaxf(xl, fminf(t1, t2));
                    xh = fminf(xh, fmaxf(t1, t2));
                } else if (bd1 < lo1 || bd1 > hi1) {
                    empty = true;
                }
                const int rr = q.r2max - qy * qy;
                if (rr < 0) empty = true;
                xh = fminf(xh, floorf(sqrtf((float)max(rr, 0))));
                if (!empty && xl <= xh) {
                    xs = (int)ceilf(xl);
                    cnt = max(0, (int)floorf(xh) - xs + 1);
                }
            }
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int x = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += x;
            }
            const int total = __shfl_sync(0xffffffffu, incl, 31);
            const int excl = incl - cnt;
            for (int i0 = 0; i0 < total; i0 += 32) {
                const int i = i0 + lane;
                int r = 0;
#pragma unroll
                for (int step = 16; step > 0; step >>= 1) {
                    const int x = __shfl_sync(0xffffffffu, incl, r + step - 1);
                    if (x <= i) r += step;
                }
                r = min(r, 31);
                const int qx = __shfl_sync(0xffffffffu, xs, r) + (i - __shfl_sync(0xffffffffu, excl, r));
                const int qyr = base + r;
                // Ownership: floor(p) inside the tile.
                float w[2][4];
                int l0 = 0, l1 = 0;
                bool own = i < total;
                if (own) {
                    float tt;
                    l0 = split_coord(fmaf(a0, (float)qx, b0 * (float)qyr), tt) - ox;
                    St::weights(tt, w[0]);
                    l1 = split_coord(fmaf(a1, (float)qx, b1 * (float)qyr), tt) - oy;
                    St::weights(tt, w[1]);
                    own = (unsigned)l0 < (unsigned)kTile && (unsigned)l1 < (unsigned)kTile;
                }
                const unsigned mask = __ballot_sync(0xffffffffu, own);
                if constexpr (CUBIC) {
                    // Each lane spreads its own sample's 16 taps into its
                    // half-warp's tile.  At step (sx, sy) lane L takes the tap
                    // whose x is (sx + L) mod 4 and y (sy + L / 4) mod 4: the 16
                    // lanes of a half-warp touch 16 different bank pairs, hence 16
                    // different words, so the plain read-add-write never races;
                    // the warp synchronises between steps because the stencils of
                    // different lanes' samples meet at different steps.
                    touched = touched || mask != 0u;
                    if (mask == 0u) continue;
                    float2 cy[4];
                    int tox[4], toy[4];
                    float wx[4];
                    if (own) {
                        const int iy = qyr < 0 ? qyr + q.N : qyr;
                        const bool in = TP_CHECK(q.dbg, iy >= 0 && iy < q.N && qx >= 0 && qx < q.Xo, 7);
                        float2 cv = in ? __ldg(gimg + iy * q.Xo + qx) : make_float2(0.f, 0.f);
                        if (q.shift && in)
                            cv = cmul_conj_a(tables ? cmul(phx[qx], phy[iy])
                                                    : shift_phase(qx, qyr, sx, sy, q.fN, q.invN),
                                             cv);
                        float wy[4];
                        rot4(w[0], (lane - l0) & 3, wx);
                        rot4(w[1], ((lane >> 2) - l1) & 3, wy);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            // the tap of residue r within [l, l + 3] is 4 ((l + 3 - r) >> 2) + r
                            tox[i] = ((l0 + 3 - rx[i]) >> 2) * 16 + rx[i];
                            toy[i] = ((l1 + 3 - ry[i]) >> 2) * (16 * (T::PX / 4)) + 4 * ry[i];
                            cy[i] = make_float2(wy[i] * cv.x, wy[i] * cv.y);
                        }
                    }
#pragma unroll
                    for (int sy2 = 0; sy2 < 4; ++sy2) {
#pragma unroll
                        for (int sx2 = 0; sx2 < 4; ++sx2) {
                            const int at = toy[sy2] + tox[sx2];
                            if (own && TP_CHECK(q.dbg, at >= 0 && at < T::ELEMS, 4)) {
                                float2 a = mytile[at];
                                cfma(wx[sx2], cy[sy2], a);
                                mytile[at] = a;
                            }
                            __syncwarp();
                        }
                    }
                    continue;
                }
                if (own) {
                    const int slot = __popc(mask & ((1u << lane) - 1u));
                    const int iy = qyr < 0 ? qyr + q.N : qyr;
                    const bool in = TP_CHECK(q.dbg, iy >= 0 && iy < q.N && qx >= 0 && qx < q.Xo, 7);
                    float2 cv = in ? __ldg(gimg + iy * q.Xo + qx) : make_float2(0.f, 0.f);
                    if (q.shift && in)
                        cv = cmul_conj_a(tables ? cmul(phx[qx], phy[iy])
                                                : shift_phase(qx, qyr, sx, sy, q.fN, q.invN),
                                         cv);
                    float *wq = Q.w[slot];
#pragma unroll
                    for (int j = 0; j < St::TAPS; ++j) {
                        wq[j] = w[0][j];
                        wq[4 + j] = w[1][j];
                    }
                    Q.rec[slot] = make_float4(cv.x, cv.y, __int_as_float(l0 | (l1 << 8)),
                                              __int_as_float(l1 * T::PX + l0));
                }
                __syncwarp();
                const int nq = __popc(mask);
                touched = touched || nq > 0;
                const int R = (nq + T::SPS - 1) / T::SPS;
                for (int rd = 0; rd < R; ++rd) {
                    const int sq = rd + R * grp;
                    const bool act = sq < nq;
                    float wt = 0.f;
                    float4 cur = make_float4(0.f, 0.f, 0.f, 0.f);
                    int idx = -1 - lane;   // unique for idle lanes
                    if (act) {
                        wt = Q.w[sq][jx] * Q.w[sq][4 + jy];
                        cur = Q.rec[sq];
                        idx = __float_as_int(cur.w) + toff;
                    }
                    bool clash = false;
                    if (T::SPS > 1)
                        clash = stencils_meet<T::SPS, 2>(act ? __float_as_int(cur.z) : kFarAway,
                                                         T::LANES, St::TAPS);
                    for (int k = 0; k < T::SPS; ++k) {
                        if (act && (!clash || grp == k) &&
                            TP_CHECK(q.dbg, idx >= 0 && idx < T::ELEMS, 4)) {
                            float2 a = acc[idx];
                            cfma(wt, make_float2(cur.x, cur.y), a);
                            acc[idx] = a;
                        }
                        __syncwarp();
                        if (!clash) break;
                    }
                }
                __syncwarp();
            }
        }
        if (!touched) continue;
        // Add the tile to the stored half-spectrum and clear it.
        const int x0 = ox - St::LO, y0 = oy - St::LO;
        for (int e = lane; e < T::S * T::S; e += 32) {
            const int lx = e % T::S, ly = e / T::S;
            const int k = T::index(lx, ly);
            float2 cv = acc[k];
            if (T::COPIES == 2) {   // the two half-warps' tiles
                const float2 c2 = acc[k + T::ELEMS];
                cv = make_float2(cv.x + c2.x, cv.y + c2.y);
                acc[k + T::ELEMS] = make_float2(0.f, 0.f);
            }
            if (cv.x == 0.f && cv.y == 0.f) continue;
            acc[k] = make_float2(0.f, 0.f);
            int nx = x0 + lx, ny = y0 + ly;
            const bool cj = nx < 0;
            if (cj) {
                nx = -nx;
                ny = -ny;
            }
            if (nx > half || !row_ok(ny, half)) continue;
            const size_t at = (size_t)wrap_row(ny, q.M) * q.Xs + nx;
            if (!TP_CHECK(q.dbg, at < (size_t)q.M * q.Xs, 6)) continue;
            atomicAdd(V + at, make_float2(cv.x, cj ? -cv.y : cv.y));
        }
        __syncwarp();
    }
}

template <bool CUBIC>
cudaError_t launch_scatter2d_tiles(const Params &q, const float2 *img, float2 *dst, cudaStream_t st) {
    using T = Tile2<CUBIC>;
    const long long images = (long long)q.B * q.P;
    if (images == 0) return cudaSuccess;
    const bool tables = q.shift && q.N <= kMaxTableN;
    const size_t smem = kTileWarps * T::WARP_BYTES + (tables ? sizeof(float2) * table_words(q.N) : 0);
    auto kern = k_scatter2d_tiles<CUBIC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(images * kSplit), 32 * kTileWarps, smem, st>>>(q, img, dst, tables);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scatter_2d(bool cubic, const Params &q, const float2 *img, float2 *dst,
                              cudaStream_t st) {
    return cubic ? launch_scatter2d_tiles<true>(q, img, dst, st)
                 : launch_scatter2d_tiles<false>(q, img, dst, st);
}

}  // namespace tp
