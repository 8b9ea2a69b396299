// tp_brick.cu -- brick-binned kernels for the 3D operators (forward central
// slices, rotation/shift gradients, backprojection / spectrum gradient).
//
// Design.  The 3D half-spectrum is viewed as a "virtual" full spectrum
// F(n) = V[n] for n_x >= 0 and conj(V[-n]) for n_x < 0 (zero outside the
// stored range): exactly the per-tap Friedel rule of the method
// [ar §2 "التمرير الأمامي"; ko §2 "Friedel 대칭성 처리"].  It is tiled
// into bricks of kBS^3 voxels.  Every output pixel q whose sample position
// p(q) = s R^T q has floor(p) inside a brick belongs to that brick, so each
// pixel has exactly one owner and its whole stencil (taps floor(p)-LO ..
// floor(p)+HI) lies in the brick plus a halo of LO+HI voxels.
//
//  - gather (forward, pose gradients): a block stages brick+halo of F in
//    shared memory, then every owned sample reads its 8 or 64 taps from
//    shared memory with one branch-free code path (for cubic in a tiled
//    layout and a per-lane tap order free of bank conflicts);
//  - scatter (backprojection, spectrum gradient): every warp owns a private
//    tile for one part of a brick (an x and y half and a z quarter) plus the
//    stencil halo, spreads its samples into it with plain read-add-write,
//    and adds the tile to the stored half-spectrum once per work item
//    (Friedel positions conjugated at -n), with vector atomics because halos
//    of neighbouring parts and other work items overlap.  The scatters read their samples from lists
//    of the output pixels sorted by brick part (a counting sort over the
//    pixels).
//
// Binning.  Three small passes precede every operator: one thread per pose
// computes the pose's geometry (into the caller's workspace, where a later
// call on the same poses finds and keeps it); a lane per brick marks which
// of a 32-pose chunk's poses can reach the brick (the plane spanned by
// a = s R[0], b = s R[1] must meet it, the half-plane qx >= 0 must touch it
// and it must lie within the pose's reach) and counts them per brick; one
// block per volume then turns the counts into a compact list of work units
// -- a brick and a range of chunks holding about kUnitHits reaching poses,
// so busy bricks near the origin are split and empty bricks vanish.  The
// gathers take units from a global counter in brick order, busiest first.  For one (pose, box) pair the
// owned pixels form a convex polygon in k-space: its rows come from the
// pseudo-inverse of [a b] and each row's qx interval from the three slab
// constraints; the enumeration is a small superset and the exact floor(p)
// test decides ownership.
//
// Method: "torch-projectors: A High-Performance Differentiable Projection
// Library for PyTorch", 3D->2D projection and 2D->3D backprojection
// [it §2 "Operazioni Supportate"; de §2 "Unterstützte Operationen"] with the
// weight spectrum [de §2 "Dual-Volumen-Ansatz"].
#include <algorithm>
#include <cstddef>

#include "tp_device.cuh"
#include "tp_launch.h"

namespace tp {

namespace {

constexpr int kBS = 16;          // brick edge (voxels)
constexpr int kWarps = 8;        // warps per block
constexpr int kThreads = 32 * kWarps;
constexpr int kGroup = 4;        // 32-pose chunks per batch of a work unit
constexpr int kUnitPoses = 32 * kGroup;
constexpr int kUnitHits = 128;   // reaching poses per work unit (load-balance target)
constexpr float kMargin = 0.01f; // enumeration margin in voxel units

// Brick + halo in shared memory.  Linear: row-major with pitches 20 x 20.
// Cubic: each z layer is a 5 x 5 grid of 4 x 4 (x, y) tiles of 16 complex
// words (one full row of 32 banks), so element (x, y) sits in bank pair
// (x mod 4) + 4 (y mod 4) whatever the tile; see gather_smem.
template <bool CUBIC>
struct Halo {
    using St = Stencil<CUBIC>;
    static constexpr int S = kBS + St::LO + St::HI;  // staged edge (19 or 17)
    static constexpr int PX = 20;                     // pitches (the cubic tiles cover 20 x 20)
    static constexpr int PY = 20;
    static constexpr int ELEMS = PX * PY * S;
    __device__ __forceinline__ static int index(int x, int y, int z) {
        if (CUBIC) return z * (PX * PY) + ((y >> 2) * (PX / 4) + (x >> 2)) * 16 + (x & 3) + 4 * (y & 3);
        return (z * PY + y) * PX + x;
    }
};

// Per-pose geometry, computed once per call.
struct PoseGeo {
    float a[3], b[3];   // p = a*qx + b*qy
    float ia[3];        // 1/a_d (0 when |a_d| is negligible)
    float u[3];         // qy = u . p for p on the plane
    float v[3];         // qx = v . p for p on the plane
    float n[3];         // a x b, the plane normal (unnormalised)
    float reach;        // largest |p| of an in-radius sample
    float sx, sy;
    int ridx, sidx;     // pose position in rot / shift
    int bp;             // output image index (b * P + p)
    int degenerate;     // a and b (nearly) parallel: no pseudo-inverse
};
constexpr int kGeoWords = sizeof(PoseGeo) / 4;
// In the workspace a pose's geometry is a record of kGeoVec 16-byte words
// (the PoseGeo words, then zeros), so one warp-uniform record load is
// kGeoVec 128-bit loads.
constexpr int kGeoVec = (kGeoWords + 3) / 4;
constexpr int kGeoReach = offsetof(PoseGeo, reach) / 4;   // word of reach in the record

// What the brick-mask pass needs of a pose, with the plane's extents over a
// brick precomputed: the brick half-size is kBS/2 plus the margin on every
// axis, so |n|.h and |v|.h are per-pose constants.
struct ReachGeo {
    float4 n;   // plane normal, then |n| . h
    float4 v;   // qx-direction v, then |v| . h
    float4 r;   // reach^2, degenerate (1 / 0), unused, unused
};

// Scratch layout inside the caller's workspace.
// Identity of a binning: the sizes it was computed for.  Together with the
// pose geometry it determines the masks and work units completely.
constexpr int kKeyWords = 12;
struct BinKey {
    unsigned w[kKeyWords];
};

struct Scratch {
    unsigned *key;        // BinKey of the binning held in the workspace
    unsigned *changed;    // set by k_pose_geometry when key or geometry differ
    unsigned *lflag;      // [0] the sample lists fit the binning held, [1] this call builds them
    unsigned *counters;   // [5][Bsrc]: work counters of the three main kernels, unit counts,
                          // item counts of the sample lists
    int4 *geo;            // B*P pose records of kGeoVec words
    float4 *pose8;        // B*P poses: (a0, a1, a2, b0), (b1, b2, sx, sy)
    ReachGeo *reach;      // B*P poses, for the brick-mask pass
    unsigned *masks;      // [Bsrc][bricks][chunks] pose bitmasks
    int *hits;            // [Bsrc][bricks] reaching poses per brick
    int4 *units;          // [Bsrc][bricks * chunks] work units (brick, first chunk, end chunk)
    // Sample lists (cubic scatter only; null in a forward-only workspace).
    unsigned *lcount;     // [Bsrc][bricks * kParts] samples per brick part, then fill cursors
    int2 *lbrick;         // [Bsrc][bricks] samples and items, then their sums before
    int4 *litems;         // [Bsrc][itemcap] items: (first entry, count, brick, part box)
    unsigned *llist;      // B*P*plane entries: output pixel index (b * P + p) * plane + row * Xo + kx
    unsigned *lrank;      // B*P*plane: each in-radius pixel's place in its key's list
    int2 *lblock;         // [Bsrc][brick blocks] the sums of k_list_sums' blocks
    int nchunks;          // 32-pose chunks per volume
    int itemcap;          // items per volume and kind
};

__device__ __forceinline__ void pose_geo(const Params &q, int b, int pi, PoseGeo &g) {
    const Pose<3> ps = load_pose<3>(q, b, pi);
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        g.a[d] = ps.a[d];
        g.b[d] = ps.b[d];
        g.ia[d] = fabsf(ps.a[d]) > 1e-6f ? 1.0f / ps.a[d] : 0.0f;
    }
    g.n[0] = g.a[1] * g.b[2] - g.a[2] * g.b[1];
    g.n[1] = g.a[2] * g.b[0] - g.a[0] * g.b[2];
    g.n[2] = g.a[0] * g.b[1] - g.a[1] * g.b[0];
    const float aa = g.a[0] * g.a[0] + g.a[1] * g.a[1] + g.a[2] * g.a[2];
    const float bb = g.b[0] * g.b[0] + g.b[1] * g.b[1] + g.b[2] * g.b[2];
    const float ab = g.a[0] * g.b[0] + g.a[1] * g.b[1] + g.a[2] * g.b[2];
    const float det = aa * bb - ab * ab;
    const bool degenerate = !(det > 1e-6f * aa * bb) || !(aa > 0.f);
    const float id = degenerate ? 0.f : 1.0f / det;
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        g.u[d] = (aa * g.b[d] - ab * g.a[d]) * id;
        g.v[d] = (bb * g.a[d] - ab * g.b[d]) * id;
    }
    // |p| <= sigma_max([a b]) |q| and |q|^2 <= r2max for in-radius pixels.
    const float hs = 0.5f * (aa + bb), hd = 0.5f * (aa - bb);
    const float smax2 = hs + sqrtf(hd * hd + ab * ab);
    g.reach = sqrtf(smax2 * (float)q.r2max) * 1.001f + 0.01f;
    g.sx = ps.sx;
    g.sy = ps.sy;
    g.ridx = ps.ridx;
    g.sidx = ps.sidx;
    g.bp = b * q.P + pi;
    g.degenerate = degenerate;
}

struct BrickBox {
    int o[3];           // brick origin (virtual spectrum coordinates)
    float lo[3], hi[3]; // box with margin
};

// Brick placement: index i in [0, 2S) of an axis maps centre-out to the
// brick coordinate 0, -1, 1, -2, ... so low brick indices are the busiest
// (central) bricks and are handed out first.
__device__ __forceinline__ int brick_coord(int i) { return (i & 1) ? -((i + 1) >> 1) : (i >> 1); }

__device__ __forceinline__ BrickBox brick_box(int linear, int nb) {
    BrickBox bx;
    const int ix = linear % nb, iy = (linear / nb) % nb, iz = linear / (nb * nb);
    bx.o[0] = brick_coord(ix) * kBS;
    bx.o[1] = brick_coord(iy) * kBS;
    bx.o[2] = brick_coord(iz) * kBS;
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        bx.lo[d] = (float)bx.o[d] - kMargin;
        bx.hi[d] = (float)(bx.o[d] + kBS) + kMargin;
    }
    return bx;
}

// Calls f(qx, qy, active) on every lane for groups of 32 candidate pixels:
// a superset of the image pixels (inside the radius) whose sample position
// lies in the box; active is false on lanes without a candidate.  Must be
// called by a whole warp with warp-uniform arguments (f may use warp
// collectives).
template <class F>
__device__ __forceinline__ void for_pixels_in_box(const PoseGeo &g, const BrickBox &bx, int N,
                                                  int r2max, F &&f) {
    const int lane = threadIdx.x & 31;
    const float *lo = bx.lo, *hi = bx.hi;
    int qy0, qy1;
    if (g.degenerate) {
        qy0 = -(N >> 1);
        qy1 = (N >> 1) - 1;
    } else {
        float m = 0.f, e = 0.f;
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            m += g.u[d] * 0.5f * (lo[d] + hi[d]);
            e += fabsf(g.u[d]) * 0.5f * (hi[d] - lo[d]);
        }
        const float lo_y = fmaxf(m - e - 0.01f, -1e7f), hi_y = fminf(m + e + 0.01f, 1e7f);
        qy0 = max((int)ceilf(lo_y), -(N >> 1));
        qy1 = min((int)floorf(hi_y), (N >> 1) - 1);
    }
    const int rmax = (int)floorf(sqrtf((float)r2max));
    qy0 = max(qy0, -rmax);
    qy1 = min(qy1, rmax);
    for (int base = qy0; base <= qy1; base += 32) {
        const int qy = base + lane;
        int xs = 0, cnt = 0;
        if (qy <= qy1) {
            float xl = 0.f, xh = (float)(N >> 1);
            bool empty = false;
#pragma unroll
            for (int d = 0; d < 3; ++d) {
                const float bd = (float)qy * g.b[d];
                if (g.ia[d] != 0.f) {
                    const float t1 = (lo[d] - bd) * g.ia[d], t2 = (hi[d] - bd) * g.ia[d];
                    xl = fmaxf(xl, fminf(t1, t2));
                    xh = fminf(xh, fmaxf(t1, t2));
                } else if (bd < lo[d] || bd > hi[d]) {
                    empty = true;
                }
            }
            const int rr = r2max - qy * qy;
            if (rr < 0) empty = true;
            xh = fminf(xh, floorf(sqrtf((float)max(rr, 0))));
            if (!empty && xl <= xh) {
                xs = (int)ceilf(xl);
                cnt = max(0, (int)floorf(xh) - xs + 1);
            }
        }
        // Inclusive scan of the row counts across the warp.
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        const int excl = incl - cnt;
        for (int i0 = 0; i0 < total; i0 += 32) {
            const int i = i0 + lane;
            // Row holding candidate i: the first lane whose inclusive count exceeds i.
            int r = 0;
#pragma unroll
            for (int step = 16; step > 0; step >>= 1) {
                const int t = __shfl_sync(0xffffffffu, incl, r + step - 1);
                if (t <= i) r += step;
            }
            r = min(r, 31);
            const int rx = __shfl_sync(0xffffffffu, xs, r);
            const int re = __shfl_sync(0xffffffffu, excl, r);
            f(rx + (i - re), base + r, i < total);
        }
    }
}

__device__ __forceinline__ int poses_of_volume(const Params &q) {
    return (q.Bsrc == 1) ? q.B * q.P : q.P;
}

// Output-image index of pose i of the pose list of spectrum v.
__device__ __forceinline__ int pose_id(const Params &q, int v, int i) {
    return (q.Bsrc == 1) ? i : v * q.P + i;
}

// ---------------------------------------------------------------------------
// Binning passes.
// Pose geometry, and whether the binning held in the workspace still fits:
// *sc.changed (cleared before the launch) is set when the key or any pose's
// geometry differs bit for bit from what is stored, and the masks and units
// are then recomputed; otherwise the two passes after this one return at
// once.  The work counters of the main kernels are cleared either way.
__global__ void __launch_bounds__(256) k_pose_geometry(Params q, int nbr, Scratch sc, BinKey key) {
    const int id = blockIdx.x * 256 + threadIdx.x;
    const int stride = gridDim.x * 256;
    for (int k = id; k < 3 * q.Bsrc; k += stride) sc.counters[k] = 0u;
    for (long long k = id; k < (long long)q.Bsrc * nbr; k += stride) sc.hits[k] = 0;
    if (id == 0) {
        bool same = true;
#pragma unroll
        for (int i = 0; i < kKeyWords; ++i) same = same && sc.key[i] == key.w[i];
        if (!same) {
#pragma unroll
            for (int i = 0; i < kKeyWords; ++i) sc.key[i] = key.w[i];
            atomicOr(sc.changed, 1u);
            sc.lflag[0] = 0u;
        }
    }
    if (id >= q.B * q.P) return;
    const int b = id / q.P, pi = id - b * q.P;
    PoseGeo g;
    pose_geo(q, b, pi, g);
    sc.pose8[2 * id] = make_float4(g.a[0], g.a[1], g.a[2], g.b[0]);
    sc.pose8[2 * id + 1] = make_float4(g.b[1], g.b[2], g.sx, g.sy);
    {
        const float h = 0.5f * (float)kBS + kMargin;
        ReachGeo rg;
        rg.n = make_float4(g.n[0], g.n[1], g.n[2],
                           h * (fabsf(g.n[0]) + fabsf(g.n[1]) + fabsf(g.n[2])));
        rg.v = make_float4(g.v[0], g.v[1], g.v[2],
                           h * (fabsf(g.v[0]) + fabsf(g.v[1]) + fabsf(g.v[2])));
        rg.r = make_float4(g.reach * g.reach, g.degenerate ? 1.f : 0.f, 0.f, 0.f);
        sc.reach[id] = rg;
    }
    int now[4 * kGeoVec];
    const int *gw = reinterpret_cast<const int *>(&g);
#pragma unroll
    for (int k = 0; k < 4 * kGeoVec; ++k) now[k] = k < kGeoWords ? gw[k] : 0;
    int4 *rec = sc.geo + (size_t)kGeoVec * id;
    bool same = true;
#pragma unroll
    for (int j = 0; j < kGeoVec; ++j) {
        const int4 h = rec[j];
        same = same && h.x == now[4 * j] && h.y == now[4 * j + 1] && h.z == now[4 * j + 2] &&
               h.w == now[4 * j + 3];
    }
    if (!same) {
#pragma unroll
        for (int j = 0; j < kGeoVec; ++j)
            rec[j] = make_int4(now[4 * j], now[4 * j + 1], now[4 * j + 2], now[4 * j + 3]);
        atomicOr(sc.changed, 1u);
        sc.lflag[0] = 0u;
    }
}

// Pose pid's record (kGeoVec 128-bit loads) as a PoseGeo.
__device__ __forceinline__ PoseGeo load_geo(const int4 *geo, int pid) {
    const int4 *rec = geo + (size_t)kGeoVec * pid;
    int w[4 * kGeoVec];
#pragma unroll
    for (int j = 0; j < kGeoVec; ++j) {
        const int4 v = __ldg(rec + j);
        w[4 * j] = v.x;
        w[4 * j + 1] = v.y;
        w[4 * j + 2] = v.z;
        w[4 * j + 3] = v.w;
    }
    PoseGeo g;
    int *dst = reinterpret_cast<int *>(&g);
#pragma unroll
    for (int k = 0; k < kGeoWords; ++k) dst[k] = w[k];
    return g;
}

__device__ __forceinline__ float geo_reach(const int4 *geo, int pid) {
    return __ldg(reinterpret_cast<const float *>(geo + (size_t)kGeoVec * pid) + kGeoReach);
}

// Bit l of mask (volume, brick, chunk) = pose 32*chunk + l of the volume's
// list can reach the brick: the box must come within the pose's reach of the
// origin, the plane must meet it and the half-plane qx >= 0 must reach it
// (with the per-pose constants of ReachGeo); the brick's count grows by the
// number of set bits.
// A lane owns one brick and runs through the chunk's 32 poses, whose
// records every lane of the warp reads at once.
__global__ void __launch_bounds__(256) k_brick_masks(Params q, int nb, Scratch sc) {
    if (*sc.changed == 0u) return;
    // The chunk's 32 reach records, each lane loading one, so that their
    // loads are in flight together.
    __shared__ ReachGeo s_rg[8][32];
    ReachGeo *const rgs = s_rg[threadIdx.x >> 5];
    const int nbr = nb * nb * nb;
    const int nchunks = sc.nchunks;
    const int groups = (nbr + 31) / 32;
    const long long total = (long long)q.Bsrc * nchunks * groups;
    const int Pv = poses_of_volume(q);
    const int lane = threadIdx.x & 31;
    const float h = 0.5f * (float)kBS + kMargin;
    for (long long w = ((long long)blockIdx.x * 256 + threadIdx.x) >> 5; w < total;
         w += ((long long)gridDim.x * 256) >> 5) {
        const int grp = (int)(w % groups);
        const long long r = w / groups;
        const int c = (int)(r % nchunks), v = (int)(r / nchunks);
        const int j = grp * 32 + lane;
        const BrickBox bx = brick_box(min(j, nbr - 1), nb);
        float cen[3], e2 = 0.f;
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            cen[d] = 0.5f * (bx.lo[d] + bx.hi[d]);
            const float e = fmaxf(fabsf(cen[d]) - h, 0.f);
            e2 += e * e;
        }
        const int np = min(32, Pv - c * 32);
        __syncwarp();   // the previous chunk's records have been read
        if (lane < np) {
            const int pid = pose_id(q, v, c * 32 + lane);
            if (TP_CHECK(q.dbg, pid >= 0 && pid < q.B * q.P, 8)) {
                const ReachGeo *rg = sc.reach + pid;
                rgs[lane].n = __ldg(&rg->n);
                rgs[lane].v = __ldg(&rg->v);
                rgs[lane].r = __ldg(&rg->r);
            } else {
                rgs[lane].r = make_float4(-1.f, 0.f, 0.f, 0.f);   // reaches nothing
            }
        }
        __syncwarp();
        unsigned m = 0u;
        for (int k = 0; k < np; ++k) {
            const float4 rr = rgs[k].r;
            if (e2 > rr.x) continue;
            bool hit = rr.y != 0.f;   // degenerate poses reach every brick within reach
            if (!hit) {
                const float4 nn = rgs[k].n, vv = rgs[k].v;
                const float cn = nn.x * cen[0] + nn.y * cen[1] + nn.z * cen[2];
                const float cv = vv.x * cen[0] + vv.y * cen[1] + vv.z * cen[2];
                hit = fabsf(cn) <= nn.w * 1.0001f + 1e-6f && cv + vv.w >= -0.01f;
            }
            m |= (hit ? 1u : 0u) << k;
        }
        if (j < nbr) {
            const size_t vj = (size_t)v * nbr + j;
            if (!TP_CHECK(q.dbg, vj < (size_t)q.Bsrc * nbr && c < nchunks, 8)) continue;
            sc.masks[vj * nchunks + c] = m;
            if (m) atomicAdd(sc.hits + vj, __popc(m));
        }
    }
}

// One block per volume: split every brick with reaching poses into
// ceil(hits / kUnitHits) units over equal chunk ranges, and list the units
// in brick order (a block-wide exclusive scan gives each brick its slots).
constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) k_plan_units(int nbr, Scratch sc, unsigned *dbg) {
    if (*sc.changed == 0u) return;
    __shared__ int warp_sum[kPlanThreads / 32];
    const int v = blockIdx.x;
    const int nch = sc.nchunks;
    const int per = (nbr + kPlanThreads - 1) / kPlanThreads;
    const int j0 = threadIdx.x * per, j1 = min(nbr, j0 + per);
    const int *hits = sc.hits + (size_t)v * nbr;
    int mine = 0;
    for (int j = j0; j < j1; ++j) {
        const int h = hits[j];
        mine += h ? min(nch, (h + kUnitHits - 1) / kUnitHits) : 0;
    }
    // Block-wide exclusive scan of the per-thread unit counts.
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int x = warp_sum[lane];
        int y = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, y, o);
            if (lane >= o) y += t;
        }
        warp_sum[lane] = y - x;   // exclusive prefix of the warp totals
        if (lane == 31) sc.counters[3 * gridDim.x + v] = (unsigned)y;
    }
    __syncthreads();
    int at = warp_sum[warp] + incl - mine;
    int4 *out = sc.units + (size_t)v * nbr * nch;
    for (int j = j0; j < j1; ++j) {
        const int h = hits[j];
        if (!h) continue;
        const int n = min(nch, (h + kUnitHits - 1) / kUnitHits);
        for (int i = 0; i < n; ++i, ++at)
            if (TP_CHECK(dbg, at < nbr * nch, 8))
                out[at] = make_int4(j, (int)((long long)nch * i / n), (int)((long long)nch * (i + 1) / n), 0);
    }
}

// ---------------------------------------------------------------------------
// Shared pieces of the main kernels.

// A batch of the block's current work unit: the poses that reach its
// brick, with their geometry copied into shared memory.
struct UnitTable {
    PoseGeo pose[kUnitPoses];
    float key[kUnitPoses];             // plane-to-brick-centre distance, relative: small = many samples
    unsigned short order[kUnitPoses];  // entries of pose[] by increasing key
    unsigned mask[32];   // masks of the batch's chunks
    int base[32];        // table offset of each chunk's first pose
    int nhit;            // entries of pose[]
    int nchunk;          // chunks in the batch
    int next;            // work counter for the warps
    int unit;            // unit index handed out by the global counter
};

// Take the next unit of volume v from the global counter (block-wide).
// Returns false when the volume's units are exhausted.
__device__ __forceinline__ bool next_unit(const Params &q, const Scratch &sc, int slot, int v,
                                          int nbr, UnitTable &t, int4 &rec) {
    const int nvol = gridDim.z;
    if (threadIdx.x == 0) t.unit = (int)atomicAdd(sc.counters + slot * nvol + v, 1u);
    __syncthreads();
    const int u = t.unit;
    __syncthreads();   // everyone has read t.unit before the next request
    if (u >= (int)__ldg(sc.counters + 3 * nvol + v)) return false;
    if (!TP_CHECK(q.dbg, u >= 0 && u < nbr * sc.nchunks, 8)) return false;
    rec = __ldg(sc.units + (size_t)v * nbr * sc.nchunks + u);
    return TP_CHECK(q.dbg, rec.x >= 0 && rec.x < nbr && rec.y >= 0 && rec.y <= rec.z &&
                               rec.z <= sc.nchunks, 8);
}

// Load the reaching poses of the unit's chunks, from chunk c on, into the
// table (block-wide): as many whole chunks (at most 32) as fit into its
// kUnitPoses entries.  Returns the first chunk not loaded; t.nhit holds the
// number of poses loaded.  The warps take the poses in t.order: the planes
// nearest the brick's centre (the largest sections, the most samples) first,
// so that the poses left when the first warps run out of work are small ones.
__device__ __forceinline__ int load_batch(const Params &q, const Scratch &sc, int nbr, int v,
                                          int brick, const BrickBox &bx, int c, int c1,
                                          UnitTable &t) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned *masks = sc.masks + ((size_t)v * nbr + brick) * sc.nchunks;
    if (warp == 0) {
        const unsigned m = (c + lane < c1) ? __ldg(masks + c + lane) : 0u;
        const int n = __popc(m);
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += x;
        }
        // Chunks 0..k-1 fit (a single chunk always does: 32 <= kUnitPoses).
        const int k = max(1, __popc(__ballot_sync(0xffffffffu, incl <= kUnitPoses)));
        t.mask[lane] = m;
        t.base[lane] = incl - n;
        if (lane == k - 1) t.nhit = incl;
        if (lane == 0) {
            t.nchunk = min(k, c1 - c);
            t.next = 0;
        }
    }
    __syncthreads();
    const int nchunk = t.nchunk;
    for (int i = warp; i < nchunk; i += kWarps) {
        const unsigned m = t.mask[i];
        if ((m >> lane) & 1u) {
            const int at = t.base[i] + __popc(m & ((1u << lane) - 1u));
            const int pid = pose_id(q, v, (c + i) * 32 + lane);
            if (!TP_CHECK(q.dbg, at < kUnitPoses && pid >= 0 && pid < q.B * q.P, 8)) continue;
            const PoseGeo g = load_geo(sc.geo, pid);
            const int *src = reinterpret_cast<const int *>(&g);
            int *dst = reinterpret_cast<int *>(&t.pose[at]);
#pragma unroll
            for (int k = 0; k < kGeoWords; ++k) dst[k] = src[k];
            float cn = 0.f, sn = 0.f;
#pragma unroll
            for (int d = 0; d < 3; ++d) {
                cn += g.n[d] * 0.5f * (bx.lo[d] + bx.hi[d]);
                sn += fabsf(g.n[d]);
            }
            t.key[at] = fabsf(cn) / fmaxf(sn, 1e-30f);
        }
    }
    __syncthreads();
    const int nhit = t.nhit;
    for (int i = threadIdx.x; i < nhit; i += kThreads) {
        const float ki = t.key[i];
        int rank = 0;
        for (int j = 0; j < nhit; ++j) {
            const float kj = t.key[j];
            rank += (kj < ki || (kj == ki && j < i)) ? 1 : 0;
        }
        t.order[rank] = (unsigned short)i;
    }
    __syncthreads();
    return c + nchunk;
}

// Next listed pose for the calling warp (its entry of t.pose), or -1 when
// the list is exhausted.
__device__ __forceinline__ int next_pose(UnitTable &t) {
    int k = 0;
    if ((threadIdx.x & 31) == 0) k = atomicAdd(&t.next, 1);
    k = __shfl_sync(0xffffffffu, k, 0);
    return k < t.nhit ? (int)t.order[k] : -1;
}

__device__ __forceinline__ bool stored(int x, int y, int z, int half) {
    return x >= 0 && x <= half && y >= -half && y < half && z >= -half && z < half;
}

// Stage brick + halo of the virtual spectrum into shared memory.  Every
// element is one 8-byte cp.async (zero-filled outside the stored range, with
// an L2 evict-last hint), so all copies of the block are in flight at once.
// A thread keeps the same
// (x, y) positions of the S x S layer in every z layer: whether its column
// lies on the Friedel side (n_x < 0, read from -n), its source column and
// its y row are fixed per brick, and each layer only adds the z row.  The
// thread then conjugates its own Friedel-side elements once its copies have
// landed.  Offsets within one stored spectrum fit 32 bits (the entry points
// refuse larger spectra).
template <bool CUBIC>
__device__ __forceinline__ void stage(const float2 *__restrict__ V, int M, int X, const BrickBox &bx,
                                      float2 *s, unsigned *dbg) {
    using H = Halo<CUBIC>;
    constexpr int L = H::S * H::S;                      // elements of one z layer
    constexpr int SLOTS = (L + kThreads - 1) / kThreads;
    const int half = M >> 1;
    const int x0 = bx.o[0] - Stencil<CUBIC>::LO, y0 = bx.o[1] - Stencil<CUBIC>::LO,
              z0 = bx.o[2] - Stencil<CUBIC>::LO;
    const int MX = M * X;
    const unsigned sbase = (unsigned)__cvta_generic_to_shared(s);
    // The spectrum is read by many bricks' stagings; ask L2 to keep it over
    // the output images, which stream past it (written evict-first).
    unsigned long long keep;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(keep));
    int at_xy[SLOTS], yoff[SLOTS];
    bool live[SLOTS], cj[SLOTS], okxy[SLOTS];
#pragma unroll
    for (int k = 0; k < SLOTS; ++k) {
        const int j = threadIdx.x + k * kThreads;
        live[k] = j < L;
        const int lx = j % H::S, ly = j / H::S;
        const int nx = x0 + lx, ny = y0 + ly;
        cj[k] = nx < 0;
        const int col = cj[k] ? -nx : nx, ys = cj[k] ? -ny : ny;
        okxy[k] = live[k] && col <= half && row_ok(ys, half);
        yoff[k] = wrap_row(ys, M) * X + col;
        at_xy[k] = H::index(lx, ly, 0);
    }
    for (int lz = 0; lz < H::S; ++lz) {
        const int nz = z0 + lz;
#pragma unroll
        for (int k = 0; k < SLOTS; ++k) {
            if (!live[k]) continue;
            const int zs = cj[k] ? -nz : nz;
            const bool ok = okxy[k] && row_ok(zs, half);
            const int off = ok ? wrap_row(zs, M) * MX + yoff[k] : 0;
            const int at = at_xy[k] + lz * (H::PX * H::PY);
            if (!TP_CHECK(dbg, off >= 0 && off < M * MX, 0)) continue;
            if (!TP_CHECK(dbg, at >= 0 && at < H::ELEMS, 1)) continue;
            asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 8, %2, %3;\n" ::"r"(
                             sbase + 8u * at),
                         "l"(V + off), "r"(ok ? 8 : 0), "l"(keep)
                         : "memory");
        }
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    // The Friedel side holds conj(V[-n]): negate the imaginary parts this
    // thread copied (zero-filled ones included, as the sign of zero is moot).
#pragma unroll
    for (int k = 0; k < SLOTS; ++k) {
        if (!live[k] || !cj[k]) continue;
        for (int lz = 0; lz < H::S; ++lz) {
            const int at = at_xy[k] + lz * (H::PX * H::PY);
            if (!TP_CHECK(dbg, at >= 0 && at < H::ELEMS, 1)) continue;
            s[at].y = -s[at].y;
        }
    }
}

// Weighted sum over the stencil from staged shared memory (and derivatives).
//
// Cubic: the 16 (x, y) taps of a layer cover all 16 bank pairs (the tile
// layout of Halo<true>), and each lane visits them in its own order: at
// step (sx, sy) lane L reads the tap in bank pair ((sx + L) mod 4) +
// 4 ((sy + L / 4) mod 4).  The 16 lanes of a half-warp then never share a
// bank pair, so every 64-bit load of the warp takes the minimum two
// wavefronts.  The order rotates the x and y taps independently, so the
// separable weights are rotated once per sample (rot4) and the row sums stay.
__device__ __forceinline__ void rot4(const float (&v)[4], int c, float (&r)[4]) {
    float t[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) t[i] = (c & 1) ? v[(i + 1) & 3] : v[i];
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = (c & 2) ? t[(i + 2) & 3] : t[i];
}

template <bool CUBIC, bool DERIV>
__device__ __forceinline__ void gather_smem(const float2 *s, const int *l, float (*w)[4],
                                            float (*d)[4], float2 &S, float2 *dS, unsigned *dbg) {
    using H = Halo<CUBIC>;
    constexpr int T = Stencil<CUBIC>::TAPS;
    S = make_float2(0.f, 0.f);
    if (DERIV)
#pragma unroll
        for (int a = 0; a < 3; ++a) dS[a] = make_float2(0.f, 0.f);
    if (CUBIC) {
        const int lane = threadIdx.x & 31;
        const int cx = (lane - l[0]) & 3, cy = ((lane >> 2) - l[1]) & 3;
        float wx[4], wy[4], dx[4], dy[4];
        rot4(w[0], cx, wx);
        rot4(w[1], cy, wy);
        if (DERIV) {
            rot4(d[0], cx, dx);
            rot4(d[1], cy, dy);
        }
        int ox[4], oy[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int x = l[0] + ((i + cx) & 3), y = l[1] + ((i + cy) & 3);
            ox[i] = (x >> 2) * 16 + (x & 3);
            oy[i] = (y >> 2) * (16 * H::PX / 4) + 4 * (y & 3);
        }
        // The 16 (x, y) tap offsets are formed once; the four z layers add
        // constants to them.
        const float2 *base = s + l[2] * (H::PX * H::PY);
        int oxy[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) oxy[i] = oy[i >> 2] + ox[i & 3];
#pragma unroll
        for (int jz = 0; jz < 4; ++jz) {
            float2 ay = make_float2(0.f, 0.f), ayx = ay, ayy = ay;
#pragma unroll
            for (int sy = 0; sy < 4; ++sy) {
                float2 r0 = make_float2(0.f, 0.f), r1 = r0;
#pragma unroll
                for (int sx = 0; sx < 4; ++sx) {
                    const int off = oxy[4 * sy + sx] + jz * (H::PX * H::PY);
                    const long long at = (base - s) + off;
                    if (!TP_CHECK(dbg, at >= 0 && at < H::ELEMS, 2)) continue;
                    const float2 val = base[off];
                    cfma(wx[sx], val, r0);
                    if (DERIV) cfma(dx[sx], val, r1);
                }
                cfma(wy[sy], r0, ay);
                if (DERIV) {
                    cfma(wy[sy], r1, ayx);
                    cfma(dy[sy], r0, ayy);
                }
            }
            cfma(w[2][jz], ay, S);
            if (DERIV) {
                cfma(w[2][jz], ayx, dS[0]);
                cfma(w[2][jz], ayy, dS[1]);
                cfma(d[2][jz], ay, dS[2]);
            }
        }
        return;
    }
    const float2 *base = s + H::index(l[0], l[1], l[2]);
#pragma unroll
    for (int jz = 0; jz < T; ++jz) {
        float2 ay = make_float2(0.f, 0.f), ayx = ay, ayy = ay;
#pragma unroll
        for (int jy = 0; jy < T; ++jy) {
            const float2 *row = base + (jz * H::PY + jy) * H::PX;
            float2 r0 = make_float2(0.f, 0.f), r1 = r0;
#pragma unroll
            for (int jx = 0; jx < T; ++jx) {
                const long long at = (row - s) + jx;
                if (!TP_CHECK(dbg, at >= 0 && at < H::ELEMS, 2)) continue;
                const float2 val = row[jx];
                cfma(w[0][jx], val, r0);
                if (DERIV) cfma(d[0][jx], val, r1);
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
}

// Owned-sample set-up: position, ownership and stencil of pixel (qx, qy).
// The box is SIZE voxels wide in x and y and SIZEZ in z.
template <bool CUBIC, bool DERIV, int SIZE = kBS, int SIZEZ = SIZE>
__device__ __forceinline__ bool own_sample(const PoseGeo &g, const BrickBox &bx, int qx, int qy,
                                           int *l, float (*w)[4], float (*d)[4]) {
    bool own = true;
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        const float p = fmaf(g.a[a], (float)qx, g.b[a] * (float)qy);
        float t;
        const int x0 = split_coord(p, t);
        l[a] = x0 - bx.o[a];
        own = own && (unsigned)l[a] < (unsigned)(a == 2 ? SIZEZ : SIZE);
        Stencil<CUBIC>::weights(t, w[a]);
        if (DERIV) Stencil<CUBIC>::derivs(t, d[a]);
    }
    return own;
}

// ---------------------------------------------------------------------------
// The fused L2 data term of the forward (tp_project_3d_2d_l2): the target
// images, the residual gradient written beside the output, and the rotation
// and shift gradients it accumulates.
struct L2Args {
    const float2 *target;   // (B, P, N, N/2+1)
    float2 *gout;           // g = 2 (out - target), same shape
    float *grad_rot;        // (Bp, P, 3, 3) +=, or null
    float *grad_shift;      // (Bs, P, 2) +=, or null
};

// Zeros for the pixels no brick owns: outside the radius (a warp writes the
// tail of an output row beyond the radius), and, for poses whose reach
// exceeds the brick grid of half-width G, in-radius pixels with floor(p)
// outside it (all their taps lie outside the stored range).  dout, when
// given, receives the matching zeros (three complex values per pixel), and
// with an L2 term gout receives -2 target there.  The rows are shared out
// over the nwarps warps of the grid.
__device__ __forceinline__ void zero_unowned(const Params &q, int G, const int4 *__restrict__ geo,
                                             float2 *__restrict__ out, float2 *__restrict__ dout,
                                             const L2Args *l2, long long warp, long long nwarps) {
    const long long rows = (long long)q.B * q.P * q.N;
    const int lane = threadIdx.x & 31;
    const int half = q.N >> 1;
    const float2 zero = make_float2(0.f, 0.f);
    const size_t nout = (size_t)q.B * q.P * q.plane;
    for (long long row = warp; row < rows; row += nwarps) {
        const int bp = (int)(row / q.N), iy = (int)(row - (long long)bp * q.N);
        const int ky = row_freq(iy, q.N);
        const int rr = q.r2max - ky * ky;
        const int xcut = rr < 0 ? -1 : min(half, (int)floorf(sqrtf((float)rr)));
        const size_t r0 = (size_t)bp * q.plane + (size_t)iy * q.Xo;
        if (!TP_CHECK(q.dbg, r0 + half < nout, 3)) continue;
        for (int x = xcut + 1 + lane; x <= half; x += 32) {
            __stcs(out + r0 + x, zero);
            if (l2) {
                const float2 t = __ldcs(l2->target + r0 + x);
                __stcs(l2->gout + r0 + x, make_float2(-2.f * t.x, -2.f * t.y));
            }
        }
        if (dout)
            for (int k = 3 * (xcut + 1) + lane; k < 3 * (half + 1); k += 32)
                __stcs(dout + 3 * r0 + k, zero);
        if (xcut >= 0 && geo_reach(geo, bp) >= (float)G - 0.5f) {
            const PoseGeo g = load_geo(geo, bp);
            for (int x = lane; x <= xcut; x += 32) {
                bool outside = false;
#pragma unroll
                for (int a = 0; a < 3; ++a) {
                    float t;
                    const int x0 = split_coord(fmaf(g.a[a], (float)x, g.b[a] * (float)ky), t);
                    outside = outside || x0 < -G || x0 >= G;
                }
                if (outside) {
                    __stcs(out + r0 + x, zero);
                    if (l2) {
                        const float2 t = __ldcs(l2->target + r0 + x);
                        __stcs(l2->gout + r0 + x, make_float2(-2.f * t.x, -2.f * t.y));
                    }
                    if (dout)
#pragma unroll
                        for (int a = 0; a < 3; ++a) __stcs(dout + 3 * (r0 + x) + a, zero);
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Forward projection, in one of three modes.  kPlain writes the output.
// kSave also gathers the stencil's derivative weights and writes
// D_a = phase * dS/dp_a (the derivative of the output with respect to the
// sample position) next to the output, three complex values per pixel.
// kL2 fuses an L2 data term L = sum |out - target|^2: it writes the output
// and the residual gradient g = 2 (out - target), and from the same
// derivative gather reduces, per warp and (pose, brick), the rotation and
// shift gradients of L (the sums of the recomputing backward) into
// grad_rot / grad_shift with one atomic per entry.
enum ProjectMode { kPlain = 0, kSave = 1, kL2 = 2 };

template <bool CUBIC, int MODE>
__global__ void __launch_bounds__(kThreads, MODE == kPlain ? 3 : 2)
    k_brick_project(Params q, int nb, Scratch sc, float2 *__restrict__ out,
                    float2 *__restrict__ dout, L2Args l2) {
    constexpr bool SAVE = MODE == kSave;
    constexpr bool L2 = MODE == kL2;
    constexpr bool DERIV = MODE != kPlain;
    extern __shared__ float2 s_vol[];
    __shared__ UnitTable s_tab;
    const int v = blockIdx.z, nbr = nb * nb * nb;
    // The zeros go out first: plain stores that overlap the gathers below.
    zero_unowned(q, (nb / 2) * kBS, sc.geo, out, dout, L2 ? &l2 : nullptr,
                 ((long long)(blockIdx.z * gridDim.x + blockIdx.x) * kThreads + threadIdx.x) >> 5,
                 (long long)gridDim.x * gridDim.z * kWarps);
    int4 rec;
    while (next_unit(q, sc, 0, v, nbr, s_tab, rec)) {
        const BrickBox bx = brick_box(rec.x, nb);
        stage<CUBIC>(q.src + (size_t)v * q.src_stride, q.M, q.Xs, bx, s_vol, q.dbg);
        for (int c0 = rec.y; c0 < rec.z;) {
            c0 = load_batch(q, sc, nbr, v, rec.x, bx, c0, rec.z, s_tab);
            for (int k; (k = next_pose(s_tab)) >= 0;) {
                const PoseGeo &g = s_tab.pose[k];
                const size_t ob = (size_t)g.bp * q.plane;
                const float sx = g.sx, sy = g.sy;
                float acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0.f;
                for_pixels_in_box(g, bx, q.N, q.r2max, [&](int qx, int qy, bool active) {
                    int l[3];
                    float w[3][4], d[3][4];
                    if (!active || !own_sample<CUBIC, DERIV>(g, bx, qx, qy, l, w, d)) return;
                    const int iy = qy < 0 ? qy + q.N : qy;
                    const size_t e = ob + (size_t)iy * q.Xo + qx;
                    if (!TP_CHECK(q.dbg, e < (size_t)q.B * q.P * q.plane && qx >= 0 && qx < q.Xo, 3))
                        return;
                    float2 t = make_float2(0.f, 0.f);
                    if (L2) t = __ldcs(l2.target + e);   // in flight during the gather
                    float2 S, dS[3];
                    gather_smem<CUBIC, DERIV>(s_vol, l, w, d, S, dS, q.dbg);
                    float2 ph = make_float2(1.f, 0.f);
                    if (q.shift) {
                        ph = shift_phase(qx, qy, sx, sy, q.fN, q.invN);
                        S = cmul(ph, S);
                        if (SAVE)
#pragma unroll
                            for (int a = 0; a < 3; ++a) dS[a] = cmul(ph, dS[a]);
                    }
                    __stcs(out + e, S);
                    if (SAVE)
#pragma unroll
                        for (int a = 0; a < 3; ++a) __stcs(dout + 3 * e + a, dS[a]);
                    if (L2) {
                        const float2 gv = make_float2(2.f * (S.x - t.x), 2.f * (S.y - t.y));
                        __stcs(l2.gout + e, gv);
                        // dL/dp_a = Re(conj(g) phase dS_a) with dS unphased here.
                        const float2 gq = cmul_conj_a(ph, gv);
#pragma unroll
                        for (int a = 0; a < 3; ++a) {
                            const float dl = gq.x * dS[a].x + gq.y * dS[a].y;
                            acc[a] = fmaf(q.s * (float)qx, dl, acc[a]);
                            acc[3 + a] = fmaf(q.s * (float)qy, dl, acc[3 + a]);
                        }
                        // Im(conj(g) y) = -2 Im(conj(t) y) exactly for g = 2 (y - t):
                        // the |y|^2 terms cancel, so form it from t and y alone
                        // (from g it would lose the digits where |y| >> |t|).
                        const float qv = -12.566370614359172f * q.invN * (t.x * S.y - t.y * S.x);
                        acc[6] = fmaf((float)qx, qv, acc[6]);
                        acc[7] = fmaf((float)qy, qv, acc[7]);
                    }
                });
                if (L2) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float t = acc[i];
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                        acc[i] = t;
                    }
                    if ((threadIdx.x & 31) == 0 &&
                        TP_CHECK(q.dbg, g.ridx >= 0 && g.ridx < q.Bp * q.P && g.sidx >= 0 &&
                                            g.sidx < q.Bs * q.P, 9)) {
                        if (l2.grad_rot)
#pragma unroll
                            for (int i = 0; i < 6; ++i)
                                if (acc[i] != 0.f) atomicAdd(l2.grad_rot + (size_t)g.ridx * 9 + i, acc[i]);
                        if (l2.grad_shift) {
                            if (acc[6] != 0.f) atomicAdd(l2.grad_shift + 2 * (size_t)g.sidx, acc[6]);
                            if (acc[7] != 0.f) atomicAdd(l2.grad_shift + 2 * (size_t)g.sidx + 1, acc[7]);
                        }
                    }
                }
            }
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------------------
// Rotation / shift gradients: per warp and (pose, brick), sums over the
// owned samples, reduced across the warp and added to grad_rot / grad_shift.
template <bool CUBIC>
__global__ void __launch_bounds__(kThreads, 2) k_brick_pose_grad(Params q, int nb, Scratch sc,
                                                                 const float2 *__restrict__ g_out,
                                                                 float *__restrict__ grad_rot,
                                                                 float *__restrict__ grad_shift) {
    extern __shared__ float2 s_vol[];
    __shared__ UnitTable s_tab;
    const int v = blockIdx.z, nbr = nb * nb * nb;
    int4 rec;
    while (next_unit(q, sc, 1, v, nbr, s_tab, rec)) {
        const BrickBox bx = brick_box(rec.x, nb);
        stage<CUBIC>(q.src + (size_t)v * q.src_stride, q.M, q.Xs, bx, s_vol, q.dbg);
        for (int c0 = rec.y; c0 < rec.z;) {
            c0 = load_batch(q, sc, nbr, v, rec.x, bx, c0, rec.z, s_tab);
            for (int k; (k = next_pose(s_tab)) >= 0;) {
                const PoseGeo &g = s_tab.pose[k];
                float acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0.f;
                const float2 *gp = g_out + (size_t)g.bp * q.plane;
                const float sx = g.sx, sy = g.sy;
                for_pixels_in_box(g, bx, q.N, q.r2max, [&](int qx, int qy, bool active) {
                    int l[3];
                    float w[3][4], d[3][4];
                    if (!active || !own_sample<CUBIC, true>(g, bx, qx, qy, l, w, d)) return;
                    float2 S, dS[3];
                    gather_smem<CUBIC, true>(s_vol, l, w, d, S, dS, q.dbg);
                    const int iy = qy < 0 ? qy + q.N : qy;
                    if (!TP_CHECK(q.dbg, iy >= 0 && iy < q.N && qx >= 0 && qx < q.Xo &&
                                             g.bp < q.B * q.P, 7))
                        return;
                    const float2 gv = __ldg(gp + iy * q.Xo + qx);
                    float2 ph = make_float2(1.f, 0.f);
                    if (q.shift) ph = shift_phase(qx, qy, sx, sy, q.fN, q.invN);
                    const float2 gq = cmul_conj_a(ph, gv);   // conj(phase) * g
#pragma unroll
                    for (int i = 0; i < 3; ++i) {
                        const float dl = gq.x * dS[i].x + gq.y * dS[i].y;   // dL/dp_i
                        acc[i] = fmaf(q.s * (float)qx, dl, acc[i]);
                        acc[3 + i] = fmaf(q.s * (float)qy, dl, acc[3 + i]);
                    }
                    const float2 y = cmul(ph, S);
                    const float qv = 6.283185307179586f * q.invN * (gv.x * y.y - gv.y * y.x);
                    acc[6] = fmaf((float)qx, qv, acc[6]);
                    acc[7] = fmaf((float)qy, qv, acc[7]);
                });
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float t = acc[i];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                    acc[i] = t;
                }
                if ((threadIdx.x & 31) == 0 &&
                    TP_CHECK(q.dbg, g.ridx >= 0 && g.ridx < q.Bp * q.P && g.sidx >= 0 &&
                                        g.sidx < q.Bs * q.P, 9)) {
                    if (grad_rot)
#pragma unroll
                        for (int i = 0; i < 6; ++i)
                            if (acc[i] != 0.f) atomicAdd(grad_rot + (size_t)g.ridx * 9 + i, acc[i]);
                    if (grad_shift) {
                        if (acc[6] != 0.f) atomicAdd(grad_shift + 2 * (size_t)g.sidx, acc[6]);
                        if (acc[7] != 0.f) atomicAdd(grad_shift + 2 * (size_t)g.sidx + 1, acc[7]);
                    }
                }
            }
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------------------
// Backprojection / spectrum gradient (adjoint of the forward projection).
//
// Both scatter kernels give every warp a private tile for one part of a
// brick plus the stencil's halo, so the spreading needs no atomics, and the
// tile is folded into the stored half-spectrum with vector global atomics
// (Friedel positions conjugated at -n) when the warp's work item is done.
// Both take their samples from lists of the output pixels sorted by brick
// part.

// Sample lists: every in-radius output pixel whose floor(p) lies in the
// brick grid, binned by brick part with a counting sort (count, scan, fill).
// A brick has kParts parts, its x and y halves times its four z quarters,
// numbered (z half, y half, x half, z quarter within the half), so the two
// parts of an octant are consecutive; a work item names its part's box by
// 4 z quarter + 2 y half + x half (part_box).  The lists depend on the poses alone, so a call keeps the
// ones held in the workspace when its binning is unchanged (k_pose_geometry
// clears lflag[0] whenever it is not).
constexpr int kParts = 16;
constexpr int kListChunk = 2048;   // most samples per scatter item

// Sample position of output pixel (qx, qy) of a pose: the ownership test of
// the forward (own_sample) uses the same expression, so both agree on floor(p).
__device__ __forceinline__ void pose8_position(const float4 &A, const float4 &Bv, int qx, int qy,
                                               float (&p)[3]) {
    p[0] = fmaf(A.x, (float)qx, A.w * (float)qy);
    p[1] = fmaf(A.y, (float)qx, Bv.x * (float)qy);
    p[2] = fmaf(A.z, (float)qx, Bv.y * (float)qy);
}

// Output pixel e = bp * plane + iy * Xo + qx as (bp, qx, qy).
__device__ __forceinline__ unsigned split_pixel(const Params &q, unsigned e, int &qx, int &qy) {
    const unsigned bp = udiv(e, (unsigned)q.plane, q.mplane);
    const unsigned pix = e - bp * (unsigned)q.plane;
    const unsigned iy = udiv(pix, (unsigned)q.Xo, q.mxo);
    qx = (int)(pix - iy * (unsigned)q.Xo);
    qy = row_freq((int)iy, q.N);
    return bp;
}

// List key (volume v, brick, part) of a sample at p: the sum of one table
// entry per axis (built by key_tables: brick index times its stride, plus
// the part bits of the axis), negative when floor(p) lies outside the brick
// grid on any axis (an entry of kKeyOut, whose sign bit is or-ed into the
// sum).  The keys stay below 2^31.  floor(p) + 1.5 * 2^23, rounded down, is
// exact for |p| < 2^22 and its bits are then floor(p) + 0x4B400000, the
// floor of split_coord; beyond 2^22 (and for infinities and NaN) the index
// leaves the table's range on the side of p, as split_coord's clamped floor
// leaves the grid.
constexpr int kKeyOut = (int)0x80000000u;   // table entry outside the grid

__device__ __forceinline__ int sample_key(const int *__restrict__ tab, int nb, int vkey,
                                          const float (&p)[3]) {
    const int span = 16 * nb;   // table entries per axis, for floor(p) in [-8 nb, 8 nb)
    const int bias = 0x4B400000 - 8 * nb - 1;
    int e[3];
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        const unsigned k = (unsigned)(__float_as_int(__fadd_rd(p[d], 12582912.0f)) - bias);
        e[d] = tab[d * (span + 2) + min(k, (unsigned)span + 1u)];   // 0 and span + 1: outside
    }
    const unsigned sum = (unsigned)vkey + (unsigned)e[0] + (unsigned)e[1] + (unsigned)e[2];
    return (int)(sum | ((unsigned)(e[0] | e[1] | e[2]) & 0x80000000u));
}

// Tables of sample_key for the grid of nb bricks per axis: axis 0 adds
// 16 i + 2 (x half), axis 1 16 nb i + 4 (y half), axis 2 16 nb^2 i +
// 8 (z half) + (z quarter within the half), i = the brick's index (see
// brick_coord) -- together brick * kParts + part, part = 8 (z half) +
// 4 (y half) + 2 (x half) + (z quarter within the half).
__device__ __forceinline__ void key_tables(int *tab, int nb) {
    const int span = 16 * nb;
    for (int t = threadIdx.x; t < 3 * (span + 2); t += blockDim.x) {
        const int d = t / (span + 2), k = t - d * (span + 2);
        int val = kKeyOut;
        if (k >= 1 && k <= span) {
            const int c = k - 1 - 8 * nb, bc = c >> 4, l = c & (kBS - 1);
            const int i = (bc << 1) ^ (bc >> 31);   // 2 bc, or -2 bc - 1
            const int stride = kParts * (d == 0 ? 1 : d == 1 ? nb : nb * nb);
            const int bits = d == 0 ? 2 * (l >> 3) : d == 1 ? 4 * (l >> 3) : 8 * (l >> 3) + ((l >> 2) & 1);
            val = i * stride + bits;
        }
        tab[t] = val;
    }
}

// Starts a list build when the lists held do not fit the binning.
__global__ void k_list_begin(Scratch sc) {
    if (threadIdx.x == 0) {
        sc.lflag[1] = sc.lflag[0] == 0u ? 1u : 0u;
        sc.lflag[0] = 1u;
    }
}

// The count pass over the output pixels (the counts were cleared before the
// launch).  A warp takes one image row and gathers, 32 in-radius pixels at a
// time, the lanes of each run of equal keys (a key that recurs after a gap
// starts another run): the run's first lane adds its length to the key's
// count with one atomic, whose result places the run in the key's list, and
// every pixel keeps its place for the fill (which recomputes the key).  The
// atomics of kListChunks chunks are issued before their results are used.
constexpr int kListChunks = 4;

// One image row of the list passes: its first pixel, last in-radius kx,
// the pose record and the key offset of its volume.  False when the row
// lies wholly outside the radius.
struct ListRow {
    unsigned e0;        // output index of the row's pixel kx = 0
    int xmax;           // last kx with kx^2 + ky^2 <= r2max
    float4 A;           // pose record (a, b0)
    float by[3];        // b qy, rounded first as in pose8_position
    int vkey;           // key offset of the row's volume
};

__device__ __forceinline__ bool list_row(const Params &q, const Scratch &sc, int nb, int row,
                                         ListRow &r) {
    const int bp = row / q.N, iy = row - bp * q.N;
    const int qy = row_freq(iy, q.N);
    const int rr = q.r2max - qy * qy;
    if (rr < 0) return false;
    // The last kx with kx^2 + ky^2 <= r2max (sqrtf corrected to the exact bound).
    int xmax = (int)sqrtf((float)rr);
    if ((xmax + 1) * (xmax + 1) <= rr) ++xmax;
    if (xmax * xmax > rr) --xmax;
    r.xmax = min(xmax, q.Xo - 1);
    r.e0 = (unsigned)bp * (unsigned)q.plane + (unsigned)iy * (unsigned)q.Xo;
    r.A = __ldg(sc.pose8 + 2 * bp);
    const float4 Bv = __ldg(sc.pose8 + 2 * bp + 1);
    r.vkey = (q.Bsrc == 1) ? 0 : (bp / q.P) * (nb * nb * nb * kParts);
    r.by[0] = r.A.w * (float)qy;
    r.by[1] = Bv.x * (float)qy;
    r.by[2] = Bv.y * (float)qy;
    return true;
}

// The key of pixel kx = f of the row (f a float holding kx).
__device__ __forceinline__ int row_key(const int *__restrict__ tab, int nb, const ListRow &r,
                                       float f) {
    const float p[3] = {fmaf(r.A.x, f, r.by[0]), fmaf(r.A.y, f, r.by[1]), fmaf(r.A.z, f, r.by[2])};
    return sample_key(tab, nb, r.vkey, p);
}

__global__ void __launch_bounds__(256) k_list_count(Params q, int nb, Scratch sc) {
    if (sc.lflag[1] == 0u) return;
    extern __shared__ int s_tab[];
    key_tables(s_tab, nb);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int rows = q.B * q.P * q.N;
    const unsigned upto = (2u << lane) - 1u;   // lanes 0 .. lane
    for (int row = (blockIdx.x * 256 + threadIdx.x) >> 5; row < rows; row += (gridDim.x * 256) >> 5) {
        ListRow R;
        if (!list_row(q, sc, nb, row, R)) continue;
        const int xmax = R.xmax;
        const unsigned e0 = R.e0;
        float fx = (float)lane;
        for (int xb = 0; xb <= xmax; xb += 32 * kListChunks, fx += 32.0f * kListChunks) {
            int key[kListChunks], leader[kListChunks];
            unsigned at[kListChunks];
#pragma unroll
            for (int k = 0; k < kListChunks; ++k) {
                const int qx = xb + 32 * k + lane;
                key[k] = -1;
                if (qx <= xmax) key[k] = row_key(s_tab, nb, R, fx + 32.0f * k);
                const int prev = __shfl_up_sync(0xffffffffu, key[k], 1);
                const unsigned starts = __ballot_sync(0xffffffffu, lane == 0 || key[k] != prev);
                leader[k] = 31 - __clz(starts & upto);
                const unsigned after = starts & ~upto;
                const int len = (after ? __ffs(after) - 1 : 32) - lane;   // meaningful on leaders
                at[k] = 0u;
                if (key[k] >= 0 && lane == leader[k]) at[k] = atomicAdd(sc.lcount + key[k], (unsigned)len);
            }
#pragma unroll
            for (int k = 0; k < kListChunks; ++k) {
                const unsigned rank = __shfl_sync(0xffffffffu, at[k], leader[k]) + (unsigned)(lane - leader[k]);
                const int qx = xb + 32 * k + lane;
                if (qx <= xmax && key[k] >= 0) sc.lrank[e0 + qx] = rank;
            }
        }
    }
}

// The fill pass (the counts are the parts' first entries now): every
// in-radius pixel with a key -- recomputed exactly as the count pass formed
// it -- is written at its key's first entry plus its place.  A warp takes one
// image row, 32 pixels at a time.
__global__ void __launch_bounds__(256) k_list_fill(Params q, int nb, Scratch sc) {
    if (sc.lflag[1] == 0u) return;
    extern __shared__ int s_tab[];
    key_tables(s_tab, nb);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int rows = q.B * q.P * q.N;
    const unsigned entries = (unsigned)q.B * (unsigned)q.P * (unsigned)q.plane;
    for (int row = (blockIdx.x * 256 + threadIdx.x) >> 5; row < rows; row += (gridDim.x * 256) >> 5) {
        ListRow R;
        if (!list_row(q, sc, nb, row, R)) continue;
        const int xmax = R.xmax;
        const unsigned e0 = R.e0;
        // kListChunks chunks at a time: their loads are all in flight before
        // the first store.
        float fx = (float)lane;
        for (int xb = lane; xb <= xmax; xb += 32 * kListChunks, fx += 32.0f * kListChunks) {
            int key[kListChunks];
            unsigned rank[kListChunks], first[kListChunks];
#pragma unroll
            for (int k = 0; k < kListChunks; ++k) {
                key[k] = xb + 32 * k <= xmax ? row_key(s_tab, nb, R, fx + 32.0f * k) : -1;
                rank[k] = key[k] >= 0 ? __ldg(sc.lrank + e0 + xb + 32 * k) : 0u;
            }
#pragma unroll
            for (int k = 0; k < kListChunks; ++k) first[k] = key[k] >= 0 ? __ldg(sc.lcount + key[k]) : 0u;
#pragma unroll
            for (int k = 0; k < kListChunks; ++k) {
                const unsigned at = first[k] + rank[k];
                if (key[k] >= 0 && TP_CHECK(q.dbg, at < entries, 8)) sc.llist[at] = e0 + (unsigned)(xb + 32 * k);
            }
        }
    }
}

// Samples and items (parts with n samples give ceil(n / kListChunk) items)
// of every brick, and their sums before it within its block of kSumBlock
// bricks (the block's totals go to lblock).  Grid: (blocks of bricks,
// volumes).
constexpr int kSumBlock = 256;

__global__ void __launch_bounds__(kSumBlock) k_list_sums(int nbr, Scratch sc) {
    if (sc.lflag[1] == 0u) return;
    __shared__ int s_w[2][kSumBlock / 32];
    const int v = blockIdx.y, j = blockIdx.x * kSumBlock + threadIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x[2] = {0, 0};
    if (j < nbr) {
        const unsigned *cnt = sc.lcount + ((size_t)v * nbr + j) * kParts;
#pragma unroll
        for (int k = 0; k < kParts; k += 4) {
            const uint4 u = *reinterpret_cast<const uint4 *>(cnt + k);
            const unsigned c[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                x[0] += (int)c[i];
                x[1] += (int)((c[i] + kListChunk - 1) / kListChunk);
            }
        }
    }
    int incl[2] = {x[0], x[1]};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl[k], o);
            if (lane >= o) incl[k] += t;
        }
        if (lane == 31) s_w[k][warp] = incl[k];
    }
    __syncthreads();
    int before[2] = {0, 0};
#pragma unroll
    for (int k = 0; k < 2; ++k)
        for (int w = 0; w < warp; ++w) before[k] += s_w[k][w];
    if (j < nbr)
        sc.lbrick[(size_t)v * nbr + j] =
            make_int2(before[0] + incl[0] - x[0], before[1] + incl[1] - x[1]);
    if (threadIdx.x == kSumBlock - 1)
        sc.lblock[(size_t)v * gridDim.x + blockIdx.x] = make_int2(before[0] + incl[0], before[1] + incl[1]);
}

// Eight threads per brick, each taking two consecutive parts (an octant's):
// their list offsets (the counts become the fill cursors) and their items --
// a part with n samples gives ceil(n / kListChunk) items of consecutive
// entries, in brick and part order.
__global__ void __launch_bounds__(256) k_list_items(int nbr, Scratch sc, int nvol,
                                                    long long vol_entries) {
    const int id = (blockIdx.x * 256 + threadIdx.x) >> 3, o = threadIdx.x & 7;
    if (sc.lflag[1] == 0u || id >= nvol * nbr) return;
    const int v = id / nbr, j = id - v * nbr;
    // The brick's sums before it: within its block of bricks, plus the
    // totals of the volume's blocks before that one.
    int2 base = sc.lbrick[id];
    const int nblk = (nbr + kSumBlock - 1) / kSumBlock;
    for (int b = 0; b < j / kSumBlock; ++b) {
        const int2 t = sc.lblock[(size_t)v * nblk + b];
        base.x += t.x;
        base.y += t.y;
    }
    unsigned *cnt = sc.lcount + (size_t)id * kParts;
    unsigned c[kParts];
#pragma unroll
    for (int k = 0; k < kParts; k += 4) {
        const uint4 u = *reinterpret_cast<const uint4 *>(cnt + k);
        c[k] = u.x;
        c[k + 1] = u.y;
        c[k + 2] = u.z;
        c[k + 3] = u.w;
    }
    // Entries and items of the parts before this thread's two.
    unsigned first = (unsigned)((long long)v * vol_entries) + (unsigned)base.x;
    int it = base.y;
    unsigned c0 = 0u, c1 = 0u;   // this thread's two parts
#pragma unroll
    for (int k = 0; k < kParts / 2; ++k) {
        if (k < o) {
            first += c[2 * k] + c[2 * k + 1];
            it += (int)((c[2 * k] + kListChunk - 1) / kListChunk) +
                  (int)((c[2 * k + 1] + kListChunk - 1) / kListChunk);
        }
        if (k == o) {
            c0 = c[2 * k];
            c1 = c[2 * k + 1];
        }
    }
    __syncwarp(0xffu << (threadIdx.x & 24));   // the brick's 8 lanes have read its counts
    cnt[2 * o] = first;   // fill cursors
    cnt[2 * o + 1] = first + c0;
    int4 *items = sc.litems + (size_t)v * sc.itemcap;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int k = 2 * o + h;
        const int zq = ((k >> 3) << 1) | (k & 1), xy = (k >> 1) & 3;
        const unsigned n = h ? c1 : c0, f = h ? first + c0 : first;
        for (unsigned i = 0; i < n; i += kListChunk, ++it)
            if (it < sc.itemcap)   // never false: itemcap bounds the items
                items[it] = make_int4((int)(f + i), (int)min((unsigned)kListChunk, n - i), j, zq * 4 + xy);
    }
    if (j == nbr - 1 && o == kParts / 2 - 1)   // the volume's last items: their count
        sc.counters[4 * nvol + v] = (unsigned)min(it, sc.itemcap);
}

// Cubic: one lane spreads one sample, 32 samples of the item's list per
// round.  The tile's (x, y) layers are cut into 4 x 4 tiles of 16 complex
// words, so word (x, y, z) sits in bank pair (x mod 4) + 4 (y mod 4), and
// lane L visits its taps in its own order: at step (sx, sy, sz) it takes the
// tap whose tile coordinates are congruent to (sx + L, sy + L / 4, sz + L / 16)
// modulo 4.  The 32 lanes then touch taps of 32 distinct residue triples --
// 32 distinct words, wherever their samples lie -- and each half-warp's 16
// words fall into 16 distinct bank pairs, so every 64-bit read or write of
// the warp takes the minimum two wavefronts.  Steps sz and sz + 2 share one
// warp barrier: over the two, half-warp 0 touches the z residues sz and
// sz + 2 and half-warp 1 the residues sz + 1 and sz + 3, so the words of the
// pair are still distinct across lanes.
//
// The real weight tile (backprojection with the weight spectrum) pairs its
// z layers: word (x, y, z) sits in bank 16 (z mod 2) + 4 (y mod 4) + x mod 4,
// and since a step's two half-warps differ in the parity of z, a warp's
// 32-bit access covers the 32 banks once.
constexpr int kOct = kBS / 2;              // octant edge
constexpr int kOS = kOct + 3;              // octant + cubic halo (taps x0 - 1 .. x0 + 2)
constexpr int kCT = 12;                    // (x, y) extent of a tile layer: 3 x 3 tiles of 4 x 4
constexpr int kCLayer = kCT * kCT;         // complex words of one z layer
constexpr int kCWPair = 2 * kCLayer;       // weight words of a pair of z layers

// A work item covers one list part of a brick: half an octant in z
// (8 x 8 x 4 tap origins).  Its tile (12 x 12 x 7 complex words, 8.1 KB) lets
// 24 warps share an SM; with the weight spectrum the two tiles take 12.7 KB
// and 16 warps do.
template <bool WEIGHTS>
struct OctLayout {
    static constexpr int WARPS = 4;                  // warps per block (blocks only share an SM)
    static constexpr int OZ = kOct / 2;              // z extent of an item's box
    static constexpr int BLOCKS = WEIGHTS ? 4 : 6;   // resident blocks per SM
    static constexpr int SZ = OZ + 3;                // z layers of the tiles
    static constexpr int ELEMS = kCLayer * SZ;       // complex words of the tile
    static constexpr int WELEMS = WEIGHTS ? kCWPair * ((SZ + 1) / 2) : 0;   // words of the weight tile
    static constexpr size_t TILE = sizeof(float2) * ELEMS;
    static constexpr size_t WTILE = sizeof(float) * WELEMS;
    static constexpr size_t WARP_BYTES = TILE + WTILE;
    static_assert(TILE % 16 == 0 && WTILE % 16 == 0, "16-byte aligned tiles");
};

// Box of list part `w` of a brick: x and y halves from bits 0 and 1, the z
// quarter from the bits above.
__device__ __forceinline__ BrickBox part_box(const BrickBox &bx, int w) {
    constexpr int kQ = kOct / 2;   // z extent of a part
    BrickBox ob;
    const int off[3] = {kOct * (w & 1), kOct * ((w >> 1) & 1), kQ * (w >> 2)};
    const int ext[3] = {kOct, kOct, kQ};
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        ob.o[d] = bx.o[d] + off[d];
        ob.lo[d] = (float)ob.o[d] - kMargin;
        ob.hi[d] = (float)(ob.o[d] + ext[d]) + kMargin;
    }
    return ob;
}

__device__ __forceinline__ float2 lds_f2(unsigned a) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ void sts_f2(unsigned a, float2 v) {
    asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(v.x), "f"(v.y) : "memory");
}
// The same, made only when p is set (the partial rounds' lanes without a
// sample make no shared-memory access at all).
__device__ __forceinline__ float2 lds_f2_if(unsigned a, bool p) {
    float2 v = make_float2(0.f, 0.f);
    asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %3, 0;\n @q ld.shared.v2.f32 {%0, %1}, [%2];\n}"
                 : "+f"(v.x), "+f"(v.y)
                 : "r"(a), "r"((unsigned)p)
                 : "memory");
    return v;
}
__device__ __forceinline__ void sts_f2_if(unsigned a, float2 v, bool p) {
    asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %3, 0;\n @q st.shared.v2.f32 [%0], {%1, %2};\n}"
                 ::"r"(a), "f"(v.x), "f"(v.y), "r"((unsigned)p)
                 : "memory");
}
__device__ __forceinline__ float lds_f1_if(unsigned a, bool p) {
    float v = 0.f;
    asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %2, 0;\n @q ld.shared.f32 %0, [%1];\n}"
                 : "+f"(v)
                 : "r"(a), "r"((unsigned)p)
                 : "memory");
    return v;
}
__device__ __forceinline__ void sts_f1_if(unsigned a, float v, bool p) {
    asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %2, 0;\n @q st.shared.f32 [%0], %1;\n}"
                 ::"r"(a), "f"(v), "r"((unsigned)p)
                 : "memory");
}
__device__ __forceinline__ float lds_f1(unsigned a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ void sts_f1(unsigned a, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

// Every lane spreads its sample into the warp's tile (and weight tile):
// first tap (l0, l1, l2) in tile coordinates (each in [0, 8), l2 in
// [0, OZ)), fraction t of p, value c = conj(phase) * y, weight om.  A lane
// with !act adds zeros to in-range words, or, with PARTIAL, makes no access
// (the last round of an item; its predicated accesses cost an instruction
// each).  tile and wtile are shared-memory byte addresses.  Call with the
// whole warp.
template <bool WEIGHTS, bool PARTIAL>
__device__ __forceinline__ void spread_cubic(int l0, int l1, int l2, const float (&tf)[3], float2 c,
                                             float om, unsigned tile, unsigned wtile, bool act) {
    const int lane = threadIdx.x & 31;
    float t[3] = {tf[0], tf[1], tf[2]};
    if (!act) {
        l0 = l1 = l2 = 0;
        t[0] = t[1] = t[2] = 0.f;
        c = make_float2(0.f, 0.f);
        om = 0.f;
    }
    float w[3][4], r[3][4];
    Stencil<true>::weights(t[0], w[0]);
    Stencil<true>::weights(t[1], w[1]);
    Stencil<true>::weights(t[2], w[2]);
    const int cx = (lane - l0) & 3, cy = ((lane >> 2) - l1) & 3, cz = ((lane >> 4) - l2) & 3;
    rot4(w[0], cx, r[0]);
    rot4(w[1], cy, r[1]);
    rot4(w[2], cz, r[2]);
    // Byte offsets of the taps of step s on each axis.
    unsigned ox[4], oy[4], oz[4], wox[4], woy[4], woz[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int x = l0 + ((s + cx) & 3), y = l1 + ((s + cy) & 3), z = l2 + ((s + cz) & 3);
        ox[s] = 8u * ((x >> 2) * 16 + (x & 3));
        oy[s] = 8u * ((y >> 2) * (4 * kCT) + 4 * (y & 3));
        oz[s] = tile + 8u * (z * kCLayer);
        if (WEIGHTS) {
            wox[s] = 4u * ((x >> 2) * 32 + (x & 3));
            woy[s] = 4u * ((y >> 2) * (8 * kCT) + 4 * (y & 3));
            woz[s] = wtile + 4u * ((z >> 1) * kCWPair + 16 * (z & 1));
        }
    }
    float2 cz2[4];
    float czw[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        cz2[s] = make_float2(r[2][s] * c.x, r[2][s] * c.y);
        czw[s] = r[2][s] * om;
    }
#pragma unroll
    for (int sg = 0; sg < 2; ++sg) {
#pragma unroll
        for (int sy = 0; sy < 4; ++sy) {
            const float2 c0 = make_float2(r[1][sy] * cz2[sg].x, r[1][sy] * cz2[sg].y);
            const float2 c1 = make_float2(r[1][sy] * cz2[sg + 2].x, r[1][sy] * cz2[sg + 2].y);
            const unsigned a0 = oy[sy] + oz[sg], a1 = oy[sy] + oz[sg + 2];
            const float w0 = r[1][sy] * czw[sg], w1 = r[1][sy] * czw[sg + 2];
            const unsigned b0 = woy[sy] + woz[sg], b1 = woy[sy] + woz[sg + 2];
#pragma unroll
            for (int sx = 0; sx < 4; ++sx) {
                float2 v0, v1;
                if (PARTIAL) {
                    v0 = lds_f2_if(a0 + ox[sx], act);
                    v1 = lds_f2_if(a1 + ox[sx], act);
                } else {
                    v0 = lds_f2(a0 + ox[sx]);
                    v1 = lds_f2(a1 + ox[sx]);
                }
                cfma(r[0][sx], c0, v0);
                cfma(r[0][sx], c1, v1);
                if (PARTIAL) {
                    sts_f2_if(a0 + ox[sx], v0, act);
                    sts_f2_if(a1 + ox[sx], v1, act);
                } else {
                    sts_f2(a0 + ox[sx], v0);
                    sts_f2(a1 + ox[sx], v1);
                }
                if (WEIGHTS) {
                    if (PARTIAL) {
                        const float u0 = lds_f1_if(b0 + wox[sx], act), u1 = lds_f1_if(b1 + wox[sx], act);
                        sts_f1_if(b0 + wox[sx], fmaf(r[0][sx], w0, u0), act);
                        sts_f1_if(b1 + wox[sx], fmaf(r[0][sx], w1, u1), act);
                    } else {
                        const float u0 = lds_f1(b0 + wox[sx]), u1 = lds_f1(b1 + wox[sx]);
                        sts_f1(b0 + wox[sx], fmaf(r[0][sx], w0, u0));
                        sts_f1(b1 + wox[sx], fmaf(r[0][sx], w1, u1));
                    }
                }
                // The next steps' taps may be other lanes' words of these steps.
                __syncwarp();
            }
        }
    }
}

template <bool WEIGHTS>
__global__ void __launch_bounds__(32 * OctLayout<WEIGHTS>::WARPS, OctLayout<WEIGHTS>::BLOCKS)
    k_brick_scatter_cubic(Params q, int nb, Scratch sc, const float2 *__restrict__ img,
                          const float *__restrict__ omega, float2 *__restrict__ dst,
                          float *__restrict__ wdst) {
    using OL = OctLayout<WEIGHTS>;
    extern __shared__ float4 s_oct[];
    const int lane = threadIdx.x & 31;
    char *mine = reinterpret_cast<char *>(s_oct) + (threadIdx.x >> 5) * OL::WARP_BYTES;
    float2 *acc = reinterpret_cast<float2 *>(mine);
    float *wacc = reinterpret_cast<float *>(mine + OL::TILE);
    const unsigned tile = (unsigned)__cvta_generic_to_shared(acc);
    const unsigned wtile = (unsigned)__cvta_generic_to_shared(wacc);
    const int half = q.M >> 1;
    const int v = blockIdx.z, nvol = gridDim.z, nbr = nb * nb * nb;
    const int nitems = (int)__ldg(sc.counters + 4 * nvol + v);
    const int4 *items = sc.litems + (size_t)v * sc.itemcap;
    const unsigned entries = (unsigned)q.B * (unsigned)q.P * (unsigned)q.plane;
    float2 *Vd = dst + (size_t)v * q.src_stride;
    float *Wd = WEIGHTS && wdst ? wdst + (size_t)v * q.src_stride : nullptr;
    for (int e = lane; e < OL::ELEMS; e += 32) acc[e] = make_float2(0.f, 0.f);
    for (int e = lane; e < OL::WELEMS; e += 32) wacc[e] = 0.f;
    __syncwarp();
    for (;;) {
        int item = 0;
        if (lane == 0) item = (int)atomicAdd(sc.counters + 2 * nvol + v, 1u);
        item = __shfl_sync(0xffffffffu, item, 0);
        if (item >= nitems) break;
        const int4 it = __ldg(items + item);   // first entry, count, brick, part
        if (!TP_CHECK(q.dbg, it.z >= 0 && it.z < nbr && it.y > 0 && it.y <= kListChunk &&
                                 (unsigned)it.x + (unsigned)it.y <= entries, 8))
            continue;
        const BrickBox ob = part_box(brick_box(it.z, nb), it.w);
        for (int r = 0; r < it.y; r += 32) {
            bool act = r + lane < it.y;
            const unsigned e = act ? __ldg(sc.llist + it.x + r + lane) : 0u;
            act = act && TP_CHECK(q.dbg, e < entries, 8);
            float2 cv = make_float2(0.f, 0.f);
            float om = 1.0f;
            if (act) {
                cv = __ldg(img + e);
                if (WEIGHTS && omega) om = __ldg(omega + e);
            }
            int qx, qy;
            const unsigned bp = split_pixel(q, act ? e : 0u, qx, qy);
            const float4 A = __ldg(sc.pose8 + 2 * bp), Bv = __ldg(sc.pose8 + 2 * bp + 1);
            float p[3], t[3];
            pose8_position(A, Bv, qx, qy, p);
            const int l0 = split_coord(p[0], t[0]) - ob.o[0];
            const int l1 = split_coord(p[1], t[1]) - ob.o[1];
            const int l2 = split_coord(p[2], t[2]) - ob.o[2];
            // The list put the sample in this box (same position arithmetic);
            // the test keeps every tile access in range whatever happens.
            const bool inbox = (unsigned)l0 < (unsigned)kOct && (unsigned)l1 < (unsigned)kOct &&
                               (unsigned)l2 < (unsigned)OL::OZ;
            act = act && TP_CHECK(q.dbg, inbox, 4) && inbox;
            if (act && q.shift) cv = cmul_conj_a(shift_phase(qx, qy, Bv.z, Bv.w, q.fN, q.invN), cv);
            if (r + 32 <= it.y)
                spread_cubic<WEIGHTS, false>(l0, l1, l2, t, cv, om, tile, wtile, act);
            else   // the item's last, partly filled round
                spread_cubic<WEIGHTS, true>(l0, l1, l2, t, cv, om, tile, wtile, act);
        }
        __syncwarp();
        // Fold the tile into the stored half-spectrum and clear it.
        const int x0 = ob.o[0] - 1, y0 = ob.o[1] - 1, z0 = ob.o[2] - 1;
        if (x0 >= 0 || x0 + kOS - 1 < 0) {
            // Every word on one side of n_x = 0 (all but the parts at the
            // origin column): each lane takes four (x, y) columns of the tile,
            // whose layer offsets and stored (x, y) positions it forms once,
            // and walks them up the z layers.
            const int sg = x0 >= 0 ? 1 : -1;   // -1: Friedel side, conjugated at -n
            int toff[4], woff[4], gyx[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = lane + 32 * j;
                const int lx = c % kOS, ly = c / kOS;
                const int tl = (ly >> 2) * (kCT / 4) + (lx >> 2), in = 4 * (ly & 3) + (lx & 3);
                toff[j] = c < kOS * kOS ? tl * 16 + in : -1;
                woff[j] = tl * 32 + in;
                const int nx = sg * (x0 + lx), ny = sg * (y0 + ly);
                gyx[j] = nx <= half && row_ok(ny, half) ? wrap_row(ny, q.M) * q.Xs + nx : -1;
            }
            for (int lz = 0; lz < OL::SZ; ++lz) {
                const int nz = sg * (z0 + lz);
                const bool zok = row_ok(nz, half);
                const size_t zrow = (size_t)wrap_row(zok ? nz : 0, q.M) * q.M * q.Xs;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (toff[j] < 0) continue;
                    const int k = lz * kCLayer + toff[j];
                    const int kw = (lz >> 1) * kCWPair + woff[j] + 16 * (lz & 1);
                    const float2 cv = acc[k];
                    const float wv = WEIGHTS ? wacc[kw] : 0.f;
                    if (cv.x == 0.f && cv.y == 0.f && wv == 0.f) continue;
                    acc[k] = make_float2(0.f, 0.f);
                    if (WEIGHTS) wacc[kw] = 0.f;
                    if (!zok || gyx[j] < 0) continue;
                    const size_t idx = zrow + (size_t)gyx[j];
                    if (!TP_CHECK(q.dbg, idx < (size_t)q.M * q.M * q.Xs, 6)) continue;
                    if (cv.x != 0.f || cv.y != 0.f) atomicAdd(Vd + idx, make_float2(cv.x, sg * cv.y));
                    if (Wd && wv != 0.f) atomicAdd(Wd + idx, wv);
                }
            }
            __syncwarp();
            continue;
        }
        for (int e = lane; e < kOS * kOS * OL::SZ; e += 32) {
            const int lx = e % kOS, ly = (e / kOS) % kOS, lz = e / (kOS * kOS);
            const int tl = (ly >> 2) * (kCT / 4) + (lx >> 2), in = 4 * (ly & 3) + (lx & 3);
            const int k = lz * kCLayer + tl * 16 + in;
            const int kw = (lz >> 1) * kCWPair + tl * 32 + 16 * (lz & 1) + in;
            const float2 cv = acc[k];
            const float wv = WEIGHTS ? wacc[kw] : 0.f;
            if (cv.x == 0.f && cv.y == 0.f && wv == 0.f) continue;
            acc[k] = make_float2(0.f, 0.f);
            if (WEIGHTS) wacc[kw] = 0.f;
            int nx = x0 + lx, ny = y0 + ly, nz = z0 + lz;
            const bool cj = nx < 0;
            if (cj) {
                nx = -nx;
                ny = -ny;
                nz = -nz;
            }
            if (!stored(nx, ny, nz, half)) continue;
            const size_t idx = ((size_t)wrap_row(nz, q.M) * q.M + wrap_row(ny, q.M)) * q.Xs + nx;
            if (!TP_CHECK(q.dbg, idx < (size_t)q.M * q.M * q.Xs, 6)) continue;
            if (cv.x != 0.f || cv.y != 0.f) atomicAdd(Vd + idx, make_float2(cv.x, cj ? -cv.y : cv.y));
            if (Wd && wv != 0.f) atomicAdd(Wd + idx, wv);
        }
        __syncwarp();
    }
}

// Linear: warp-private tiles of one z-half part (8 x 8 x 4 tap origins) plus
// the one-voxel halo of the taps x0, x0 + 1, stored as 9 x 9 x 5 words with x
// and y pitches 10 (the 8 taps of one sample fall into 8 distinct bank
// pairs); the tiles and queue of a warp take 7.7 KB, so 32 warps share an SM.
// A round spreads four queued samples at once, the lanes of group g = lane / 8
// taking the 8 taps of sample r + R g (R = rounds of the queue).  Samples R
// slots apart rarely share a voxel; a round in which two of them do (their
// tile coordinates, exchanged by shuffles, differ by less than 2 on every
// axis) is spread one sample at a time, so the plain read-add-write never
// races.
constexpr int kLS = kOct + 1;               // part + linear halo in x and y
constexpr int kLZ = kOct / 2 + 1;           // the same in z
constexpr int kLPX = 10, kLPY = 10;         // x and y pitches of the tile
constexpr int kLElems = kLZ * kLPY * kLPX;  // complex words of the tile
constexpr int kLQW = 9;                     // floats per queued weight row (odd)

struct LinQueue {
    float w[32][kLQW];   // per sample: the 8 tap weights wx wy wz (x fastest), tile x | y << 8 | z << 16
    float4 rec[32];      // per sample: conj(phase) * y (re, im), omega, first tap
};

template <bool WEIGHTS>
struct LinLayout {
    static constexpr int WARPS = 4;
    static constexpr size_t TILE = sizeof(float2) * kLElems;
    static constexpr size_t WTILE = WEIGHTS ? sizeof(float) * kLElems : 0;
    static constexpr size_t WARP_BYTES = TILE + WTILE + sizeof(LinQueue);
    static_assert(TILE % 16 == 0 && WTILE % 16 == 0 && sizeof(LinQueue) % 16 == 0,
                  "16-byte aligned sections");
};

template <bool WEIGHTS>
__global__ void __launch_bounds__(32 * LinLayout<WEIGHTS>::WARPS, 8)
    k_brick_scatter_linear(Params q, int nb, Scratch sc, const float2 *__restrict__ img,
                           const float *__restrict__ omega, float2 *__restrict__ dst,
                           float *__restrict__ wdst) {
    using LL = LinLayout<WEIGHTS>;
    extern __shared__ float4 s_lin[];
    const int lane = threadIdx.x & 31;
    char *mine = reinterpret_cast<char *>(s_lin) + (threadIdx.x >> 5) * LL::WARP_BYTES;
    float2 *acc = reinterpret_cast<float2 *>(mine);
    float *wacc = reinterpret_cast<float *>(mine + LL::TILE);
    LinQueue &Q = *reinterpret_cast<LinQueue *>(mine + LL::TILE + LL::WTILE);
    const int grp = lane >> 3, jx = lane & 1, jy = (lane >> 1) & 1, jz = (lane >> 2) & 1;
    const int toff = jx + kLPX * (jy + kLPY * jz);
    const int half = q.M >> 1;
    const int v = blockIdx.z, nvol = gridDim.z, nbr = nb * nb * nb;
    const int nitems = (int)__ldg(sc.counters + 4 * nvol + v);
    const int4 *items = sc.litems + (size_t)v * sc.itemcap;
    const unsigned entries = (unsigned)q.B * (unsigned)q.P * (unsigned)q.plane;
    float2 *Vd = dst + (size_t)v * q.src_stride;
    float *Wd = WEIGHTS && wdst ? wdst + (size_t)v * q.src_stride : nullptr;
    for (int e = lane; e < kLElems; e += 32) {
        acc[e] = make_float2(0.f, 0.f);
        if (WEIGHTS) wacc[e] = 0.f;
    }
    __syncwarp();
    for (;;) {
        int item = 0;
        if (lane == 0) item = (int)atomicAdd(sc.counters + 2 * nvol + v, 1u);
        item = __shfl_sync(0xffffffffu, item, 0);
        if (item >= nitems) break;
        const int4 it = __ldg(items + item);   // first entry, count, brick, part
        if (!TP_CHECK(q.dbg, it.z >= 0 && it.z < nbr && it.y > 0 && it.y <= kListChunk &&
                                 (unsigned)it.x + (unsigned)it.y <= entries, 8))
            continue;
        const BrickBox ob = part_box(brick_box(it.z, nb), it.w);
        for (int r0 = 0; r0 < it.y; r0 += 32) {
            // Each lane sets up one sample of the list and queues it.
            bool own = r0 + lane < it.y;
            const unsigned e = own ? __ldg(sc.llist + it.x + r0 + lane) : 0u;
            own = own && TP_CHECK(q.dbg, e < entries, 8);
            int qx, qy;
            const unsigned bp = split_pixel(q, own ? e : 0u, qx, qy);
            float2 cv = own ? __ldg(img + e) : make_float2(0.f, 0.f);
            const float om = (WEIGHTS && omega && own) ? __ldg(omega + e) : 1.0f;
            const float4 A = __ldg(sc.pose8 + 2 * bp), Bv = __ldg(sc.pose8 + 2 * bp + 1);
            float p[3], w[3][2];
            int l[3];
            pose8_position(A, Bv, qx, qy, p);
#pragma unroll
            for (int a = 0; a < 3; ++a) {
                float t;
                l[a] = split_coord(p[a], t) - ob.o[a];
                Stencil<false>::weights(t, w[a]);
            }
            // The list put the sample in this part (same position arithmetic);
            // the test keeps every tile access in range whatever happens.
            const bool inbox = (unsigned)l[0] < (unsigned)kOct && (unsigned)l[1] < (unsigned)kOct &&
                               (unsigned)l[2] < (unsigned)(kOct / 2);
            own = own && TP_CHECK(q.dbg, inbox, 4) && inbox;
            const unsigned mask = __ballot_sync(0xffffffffu, own);
            if (own) {
                if (q.shift) cv = cmul_conj_a(shift_phase(qx, qy, Bv.z, Bv.w, q.fN, q.invN), cv);
                const int slot = __popc(mask & ((1u << lane) - 1u));
                float *wq = Q.w[slot];
#pragma unroll
                for (int t = 0; t < 8; ++t) wq[t] = w[0][t & 1] * w[1][(t >> 1) & 1] * w[2][t >> 2];
                wq[8] = __int_as_float(l[0] | (l[1] << 8) | (l[2] << 16));
                Q.rec[slot] = make_float4(cv.x, cv.y, om, __int_as_float((l[2] * kLPY + l[1]) * kLPX + l[0]));
            }
            __syncwarp();
            const int nq = __popc(mask);
            const int R = (nq + 3) >> 2;
            for (int r = 0; r < R; ++r) {
                const int sq = r + R * grp;
                const bool act = sq < nq;
                float wt = 0.f;
                float4 cur = make_float4(0.f, 0.f, 0.f, 0.f);
                int idx = 0, at = kFarAway;
                if (act) {
                    wt = Q.w[sq][lane & 7];
                    at = __float_as_int(Q.w[sq][8]);
                    cur = Q.rec[sq];
                    idx = __float_as_int(cur.w) + toff;
                }
                const bool clash = stencils_meet<4, 3>(at, 8, 2);
                for (int k = 0; k < 4; ++k) {
                    if (act && (!clash || grp == k) && TP_CHECK(q.dbg, idx >= 0 && idx < kLElems, 4)) {
                        float2 a = acc[idx];
                        cfma(wt, make_float2(cur.x, cur.y), a);
                        acc[idx] = a;
                        if (WEIGHTS) wacc[idx] = fmaf(wt, cur.z, wacc[idx]);
                    }
                    __syncwarp();
                    if (!clash) break;
                }
            }
            __syncwarp();
        }
        // Fold the tile into the stored half-spectrum and clear it.
        const int x0 = ob.o[0], y0 = ob.o[1], z0 = ob.o[2];
        if (x0 >= 0 || x0 + kLS - 1 < 0) {
            // Every word on one side of n_x = 0: by (x, y) columns, as in
            // the cubic scatter (three columns a lane).
            const int sg = x0 >= 0 ? 1 : -1;   // -1: Friedel side, conjugated at -n
            int toff[3], gyx[3];
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const int c = lane + 32 * j;
                const int lx = c % kLS, ly = c / kLS;
                toff[j] = c < kLS * kLS ? ly * kLPX + lx : -1;
                const int nx = sg * (x0 + lx), ny = sg * (y0 + ly);
                gyx[j] = nx <= half && row_ok(ny, half) ? wrap_row(ny, q.M) * q.Xs + nx : -1;
            }
            for (int lz = 0; lz < kLZ; ++lz) {
                const int nz = sg * (z0 + lz);
                const bool zok = row_ok(nz, half);
                const size_t zrow = (size_t)wrap_row(zok ? nz : 0, q.M) * q.M * q.Xs;
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    if (toff[j] < 0) continue;
                    const int k = lz * kLPY * kLPX + toff[j];
                    const float2 cv = acc[k];
                    const float wv = WEIGHTS ? wacc[k] : 0.f;
                    if (cv.x == 0.f && cv.y == 0.f && wv == 0.f) continue;
                    acc[k] = make_float2(0.f, 0.f);
                    if (WEIGHTS) wacc[k] = 0.f;
                    if (!zok || gyx[j] < 0) continue;
                    const size_t idx = zrow + (size_t)gyx[j];
                    if (!TP_CHECK(q.dbg, idx < (size_t)q.M * q.M * q.Xs, 6)) continue;
                    if (cv.x != 0.f || cv.y != 0.f) atomicAdd(Vd + idx, make_float2(cv.x, sg * cv.y));
                    if (Wd && wv != 0.f) atomicAdd(Wd + idx, wv);
                }
            }
            __syncwarp();
            continue;
        }
        for (int e = lane; e < kLS * kLS * kLZ; e += 32) {
            const int lx = e % kLS, ly = (e / kLS) % kLS, lz = e / (kLS * kLS);
            const int k = (lz * kLPY + ly) * kLPX + lx;
            const float2 cv = acc[k];
            const float wv = WEIGHTS ? wacc[k] : 0.f;
            if (cv.x == 0.f && cv.y == 0.f && wv == 0.f) continue;
            acc[k] = make_float2(0.f, 0.f);
            if (WEIGHTS) wacc[k] = 0.f;
            int nx = x0 + lx, ny = y0 + ly, nz = z0 + lz;
            const bool cj = nx < 0;
            if (cj) {
                nx = -nx;
                ny = -ny;
                nz = -nz;
            }
            if (!stored(nx, ny, nz, half)) continue;
            const size_t idx = ((size_t)wrap_row(nz, q.M) * q.M + wrap_row(ny, q.M)) * q.Xs + nx;
            if (!TP_CHECK(q.dbg, idx < (size_t)q.M * q.M * q.Xs, 6)) continue;
            if (cv.x != 0.f || cv.y != 0.f) atomicAdd(Vd + idx, make_float2(cv.x, cj ? -cv.y : cv.y));
            if (Wd && wv != 0.f) atomicAdd(Wd + idx, wv);
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// Launch geometry and scratch layout.
int bricks_per_axis(int M, bool cubic) {
    const int need = (M >> 1) + (cubic ? Stencil<true>::HI : Stencil<false>::HI);
    return 2 * ((need + kBS - 1) / kBS);
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct Layout {
    size_t counters, geo, pose8, reach, masks, hits, units, binning;   // the binning
    size_t lcount, lbrick, litems, llist, lrank, lblock, total;       // + the sample lists
    int nb, nchunks, itemcap;
    long long vol_entries;   // list entries per volume (its images' pixels)
};

// Workspace layout: the binning every 3D operator uses, then the sample lists
// of the scatters, sized for every output pixel.
Layout layout(const Params &q, bool cubic) {
    Layout L;
    L.nb = bricks_per_axis(q.M, cubic);
    const size_t nbr = (size_t)L.nb * L.nb * L.nb;
    const long long Pv = (q.Bsrc == 1) ? (long long)q.B * q.P : q.P;
    const size_t poses = (size_t)q.B * q.P;
    L.nchunks = (int)((Pv + 31) / 32);
    L.counters = 256;                                         // key and flags first
    L.geo = L.counters + align256(sizeof(unsigned) * 5 * (size_t)q.Bsrc);
    L.pose8 = L.geo + align256(sizeof(int4) * kGeoVec * poses);
    L.reach = L.pose8 + align256(2 * sizeof(float4) * poses);
    L.masks = L.reach + align256(sizeof(ReachGeo) * poses);
    L.hits = L.masks + align256(sizeof(unsigned) * (size_t)q.Bsrc * nbr * L.nchunks);
    L.units = L.hits + align256(sizeof(int) * (size_t)q.Bsrc * nbr);
    L.binning = L.units + align256(sizeof(int4) * (size_t)q.Bsrc * nbr * L.nchunks);
    L.vol_entries = Pv * (long long)q.N * (q.N / 2 + 1);
    L.itemcap = 0;
    L.lcount = L.lbrick = L.litems = L.llist = L.lrank = L.lblock = 0;
    L.total = L.binning;
    {
        L.itemcap = (int)(nbr * kParts + L.vol_entries / kListChunk + 1);
        L.lcount = L.binning;
        L.lbrick = L.lcount + align256(sizeof(unsigned) * (size_t)q.Bsrc * nbr * kParts);
        L.litems = L.lbrick + align256(sizeof(int2) * (size_t)q.Bsrc * nbr);
        L.llist = L.litems + align256(sizeof(int4) * (size_t)q.Bsrc * L.itemcap);
        L.lrank = L.llist + align256(sizeof(unsigned) * (size_t)(L.vol_entries * q.Bsrc));
        L.lblock = L.lrank + align256(sizeof(unsigned) * (size_t)(L.vol_entries * q.Bsrc));
        L.total = L.lblock + align256(sizeof(int2) * (size_t)q.Bsrc * ((nbr + kSumBlock - 1) / kSumBlock));
    }
    return L;
}

Scratch scratch_in(void *ws, const Layout &L) {
    Scratch sc;
    char *base = static_cast<char *>(ws);
    sc.key = reinterpret_cast<unsigned *>(base);
    sc.changed = sc.key + kKeyWords;
    sc.lflag = sc.changed + 1;
    sc.counters = reinterpret_cast<unsigned *>(base + L.counters);
    sc.geo = reinterpret_cast<int4 *>(base + L.geo);
    sc.pose8 = reinterpret_cast<float4 *>(base + L.pose8);
    sc.reach = reinterpret_cast<ReachGeo *>(base + L.reach);
    sc.masks = reinterpret_cast<unsigned *>(base + L.masks);
    sc.hits = reinterpret_cast<int *>(base + L.hits);
    sc.units = reinterpret_cast<int4 *>(base + L.units);
    sc.lcount = L.lcount ? reinterpret_cast<unsigned *>(base + L.lcount) : nullptr;
    sc.lbrick = L.lbrick ? reinterpret_cast<int2 *>(base + L.lbrick) : nullptr;
    sc.litems = L.litems ? reinterpret_cast<int4 *>(base + L.litems) : nullptr;
    sc.llist = L.llist ? reinterpret_cast<unsigned *>(base + L.llist) : nullptr;
    sc.lrank = L.lrank ? reinterpret_cast<unsigned *>(base + L.lrank) : nullptr;
    sc.lblock = L.lblock ? reinterpret_cast<int2 *>(base + L.lblock) : nullptr;
    sc.nchunks = L.nchunks;
    sc.itemcap = L.itemcap;
    return sc;
}

int resident_blocks(const void *kern, size_t smem) {
    int dev = 0, sms = 148, per_sm = 1;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    return sms * per_sm;
}

// Pose geometry, brick masks and work units for the poses of q (shared by
// the main kernels of one call).
BinKey bin_key(const Params &q, const Layout &L) {
    BinKey k{};
    k.w[0] = 0x6e696274u;   // tag: a binning of this library
    k.w[1] = (unsigned)q.M;
    k.w[2] = (unsigned)q.N;
    k.w[3] = (unsigned)q.B;
    k.w[4] = (unsigned)q.P;
    k.w[5] = (unsigned)q.Bsrc;
    k.w[6] = (unsigned)q.Bp;
    k.w[7] = (unsigned)q.Bs;
    k.w[8] = (unsigned)L.nb;
    k.w[9] = (unsigned)L.nchunks;
    k.w[10] = (unsigned)q.r2max;
    k.w[11] = q.shift ? 1u : 0u;
    return k;
}

cudaError_t bin(const Params &q, const Layout &L, const Scratch &sc, cudaStream_t st) {
    const int nbr = L.nb * L.nb * L.nb;
    const int pb = (int)((q.B * (long long)q.P + 255) / 256);
    cudaError_t e = cudaMemsetAsync(sc.changed, 0, sizeof(unsigned), st);
    if (e != cudaSuccess) return e;
    k_pose_geometry<<<pb, 256, 0, st>>>(q, nbr, sc, bin_key(q, L));
    const long long warps = (long long)q.Bsrc * L.nchunks * ((nbr + 31) / 32);
    long long blocks = (warps + 7) / 8;
    if (blocks > 65535LL * 32) blocks = 65535LL * 32;
    k_brick_masks<<<(unsigned)blocks, 256, 0, st>>>(q, L.nb, sc);
    k_plan_units<<<q.Bsrc, kPlanThreads, 0, st>>>(nbr, sc, q.dbg);
    return cudaGetLastError();
}

// Binning for a main kernel whose work counter is `slot` (0 forward, 1 pose
// gradient, 2 scatter).
cudaError_t prepare(const Params &q, const Layout &L, const Scratch &sc, int slot, BinMode mode,
                    cudaStream_t st) {
    (void)slot;
    return mode == kBinNew ? bin(q, L, sc, st) : cudaSuccess;
}

// Blocks of a main kernel: the resident ones, shared out over the volumes
// (each volume has its own unit list and counter, indexed by blockIdx.z).
dim3 main_grid(const Params &q, const void *kern, size_t smem) {
    const long long res = resident_blocks(kern, smem);
    long long per = (res + q.Bsrc - 1) / q.Bsrc;
    if (per < 1) per = 1;
    return dim3((unsigned)per, 1, (unsigned)q.Bsrc);
}

// Blocks of a kernel whose warps take work items on their own (the list-fed
// scatters): every resident block, shared out over the volumes.
dim3 warp_grid(const Params &q, const void *kern, int threads, size_t smem) {
    int dev = 0, sms = 148, per_sm = 1;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const long long per = ((long long)sms * per_sm + q.Bsrc - 1) / q.Bsrc;
    return dim3((unsigned)per, 1, (unsigned)q.Bsrc);
}

template <bool CUBIC, int MODE>
cudaError_t project_t(const Params &q, float2 *out, float2 *dout, const L2Args &l2, void *ws,
                      BinMode mode, cudaStream_t st) {
    const Layout L = layout(q, CUBIC);
    const Scratch sc = scratch_in(ws, L);
    const size_t smem = sizeof(float2) * Halo<CUBIC>::ELEMS;
    auto kern = k_brick_project<CUBIC, MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if ((e = prepare(q, L, sc, 0, mode, st)) != cudaSuccess) return e;
    kern<<<main_grid(q, (const void *)kern, smem), kThreads, smem, st>>>(q, L.nb, sc, out, dout, l2);
    return cudaGetLastError();
}

template <bool CUBIC>
cudaError_t pose_grad_t(const Params &q, const float2 *g, float *grot, float *gshift, void *ws,
                        BinMode mode, cudaStream_t st) {
    const Layout L = layout(q, CUBIC);
    const Scratch sc = scratch_in(ws, L);
    const size_t smem = sizeof(float2) * Halo<CUBIC>::ELEMS;
    auto kern = k_brick_pose_grad<CUBIC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if ((e = prepare(q, L, sc, 1, mode, st)) != cudaSuccess) return e;
    kern<<<main_grid(q, (const void *)kern, smem), kThreads, smem, st>>>(q, L.nb, sc, g, grot,
                                                                       gshift);
    return cudaGetLastError();
}

// The sample lists of the scatters, unless the workspace holds the ones
// of this binning (the kernels after k_list_begin then return at once).
cudaError_t build_lists(const Params &q, const Layout &L, const Scratch &sc, cudaStream_t st) {
    const int nbr = L.nb * L.nb * L.nb;
    cudaError_t e = cudaMemsetAsync(sc.lcount, 0, sizeof(unsigned) * (size_t)q.Bsrc * nbr * kParts, st);
    if (e != cudaSuccess) return e;
    k_list_begin<<<1, 32, 0, st>>>(sc);
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long rows = (long long)q.B * q.P * q.N;
    const unsigned blocks = (unsigned)std::min<long long>((rows + 7) / 8, 16LL * sms);
    const unsigned bricks = (unsigned)(((long long)q.Bsrc * nbr + 255) / 256);
    if (blocks == 0) return cudaGetLastError();
    const size_t tab = sizeof(int) * 3 * (16 * L.nb + 2);
    if ((e = cudaFuncSetAttribute(k_list_count, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tab)) !=
            cudaSuccess ||
        (e = cudaFuncSetAttribute(k_list_fill, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tab)) !=
            cudaSuccess)
        return e;
    k_list_count<<<blocks, 256, tab, st>>>(q, L.nb, sc);
    k_list_sums<<<dim3((unsigned)((nbr + kSumBlock - 1) / kSumBlock), (unsigned)q.Bsrc), kSumBlock, 0, st>>>(nbr, sc);
    k_list_items<<<8 * bricks, 256, 0, st>>>(nbr, sc, q.Bsrc, L.vol_entries);
    k_list_fill<<<blocks, 256, tab, st>>>(q, L.nb, sc);
    return cudaGetLastError();
}

template <bool WEIGHTS>
cudaError_t scatter_linear_t(const Params &q, const float2 *img, const float *omega, float2 *dst,
                             float *wdst, void *ws, BinMode mode, cudaStream_t st) {
    using LL = LinLayout<WEIGHTS>;
    const Layout L = layout(q, false);
    const Scratch sc = scratch_in(ws, L);
    const int threads = 32 * LL::WARPS;
    const size_t smem = LL::WARP_BYTES * LL::WARPS;
    auto kern = k_brick_scatter_linear<WEIGHTS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if ((e = prepare(q, L, sc, 2, mode, st)) != cudaSuccess) return e;
    if ((e = build_lists(q, L, sc, st)) != cudaSuccess) return e;
    kern<<<warp_grid(q, (const void *)kern, threads, smem), threads, smem, st>>>(q, L.nb, sc, img,
                                                                               omega, dst, wdst);
    return cudaGetLastError();
}

template <bool WEIGHTS>
cudaError_t scatter_cubic_t(const Params &q, const float2 *img, const float *omega, float2 *dst,
                            float *wdst, void *ws, BinMode mode, cudaStream_t st) {
    using OL = OctLayout<WEIGHTS>;
    const Layout L = layout(q, true);
    const Scratch sc = scratch_in(ws, L);
    const int threads = 32 * OL::WARPS;
    const size_t smem = OL::WARP_BYTES * OL::WARPS;
    auto kern = k_brick_scatter_cubic<WEIGHTS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if ((e = prepare(q, L, sc, 2, mode, st)) != cudaSuccess) return e;
    if ((e = build_lists(q, L, sc, st)) != cudaSuccess) return e;
    kern<<<warp_grid(q, (const void *)kern, threads, smem), threads, smem, st>>>(q, L.nb, sc, img,
                                                                               omega, dst, wdst);
    return cudaGetLastError();
}

}  // namespace

size_t brick_workspace_bytes(const Params &q, bool cubic) { return layout(q, cubic).total; }

size_t brick_binning_bytes(const Params &q, bool cubic) { return layout(q, cubic).binning; }

long long brick_parts(const Params &q, bool cubic) {
    const long long nb = bricks_per_axis(q.M, cubic);
    return nb * nb * nb * kParts;
}

cudaError_t launch_brick_project(bool cubic, const Params &q, float2 *out, float2 *dout, void *ws,
                                 BinMode mode, cudaStream_t st) {
    const L2Args none{};
    if (dout)
        return cubic ? project_t<true, kSave>(q, out, dout, none, ws, mode, st)
                     : project_t<false, kSave>(q, out, dout, none, ws, mode, st);
    return cubic ? project_t<true, kPlain>(q, out, nullptr, none, ws, mode, st)
                 : project_t<false, kPlain>(q, out, nullptr, none, ws, mode, st);
}

cudaError_t launch_brick_project_l2(bool cubic, const Params &q, const float2 *target, float2 *out,
                                    float2 *grad_out, float *grad_rot, float *grad_shift, void *ws,
                                    cudaStream_t st) {
    const L2Args l2{target, grad_out, grad_rot, grad_shift};
    return cubic ? project_t<true, kL2>(q, out, nullptr, l2, ws, kBinNew, st)
                 : project_t<false, kL2>(q, out, nullptr, l2, ws, kBinNew, st);
}

cudaError_t launch_brick_pose_grad(bool cubic, const Params &q, const float2 *g, float *grot,
                                   float *gshift, void *ws, BinMode mode, cudaStream_t st) {
    return cubic ? pose_grad_t<true>(q, g, grot, gshift, ws, mode, st)
                 : pose_grad_t<false>(q, g, grot, gshift, ws, mode, st);
}

cudaError_t launch_brick_scatter(bool cubic, const Params &q, const float2 *img, const float *omega,
                                 float2 *dst, float *wdst, void *ws, BinMode mode, cudaStream_t st) {
    if (wdst)
        return cubic ? scatter_cubic_t<true>(q, img, omega, dst, wdst, ws, mode, st)
                     : scatter_linear_t<true>(q, img, omega, dst, wdst, ws, mode, st);
    return cubic ? scatter_cubic_t<false>(q, img, omega, dst, nullptr, ws, mode, st)
                 : scatter_linear_t<false>(q, img, omega, dst, nullptr, ws, mode, st);
}

}  // namespace tp
