// tp_tiles.cuh -- helpers of the 2D kernels that use 4 x 4-tiled shared-memory
// layouts (word (x, y) in bank pair (x mod 4) + 4 (y mod 4)) with a
// lane-rotated cubic tap order.
#pragma once

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

}  // namespace tp
