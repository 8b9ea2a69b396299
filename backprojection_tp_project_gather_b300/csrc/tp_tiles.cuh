// tp_tiles.cuh -- helpers of the 2D kernels that use 4 x 4-tiled shared-memory
// layouts (word (x, y) in bank pair (x mod 4) + 4 (y mod 4)) with a
// lane-rotated cubic tap order, and the per-pose tables of the separable
// shift phase.
#pragma once

#include "tp_device.cuh"

namespace tp {

// r[i] = v[(i + c) mod 4] with static register indexes (two selects per
// entry): the per-lane rotation of a cubic stencil's separable weights.
__device__ __forceinline__ void rot4(const float (&v)[4], int c, float (&r)[4]) {
    float t[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) t[i] = (c & 1) ? v[(i + 1) & 3] : v[i];
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = (c & 2) ? t[(i + 2) & 3] : t[i];
}

// Complex words of the phase tables of one pose (N/2 + 1 column and N row
// factors), rounded up to an even count so that what follows stays 16-byte
// aligned.
__host__ __device__ inline int table_words(int N) { return (N + N / 2 + 1 + 1) & ~1; }

// The two factors of the shift phase of one pose, exp(-2 pi i (kx sx + ky sy) / N)
// = exp(-2 pi i kx sx / N) exp(-2 pi i ky sy / N): phx[kx] for kx = 0 .. N/2 and
// phy[iy] = exp(-2 pi i ky(iy) sy / N) for iy = 0 .. N-1, each from the exactly
// period-reduced cycle count (frac_cycles).  Called by the whole block.
__device__ __forceinline__ void phase_tables(const Params &q, float sx, float sy, float2 *phx,
                                             float2 *phy) {
    for (int i = threadIdx.x; i < q.N + q.Xo; i += blockDim.x) {
        const bool col = i < q.Xo;
        const int k = col ? i : row_freq(i - q.Xo, q.N);
        float sn, cs;
        sincospif(-2.0f * frac_cycles(k, col ? sx : sy, q.fN, q.invN), &sn, &cs);
        (col ? phx[i] : phy[i - q.Xo]) = make_float2(cs, sn);
    }
}

}  // namespace tp
