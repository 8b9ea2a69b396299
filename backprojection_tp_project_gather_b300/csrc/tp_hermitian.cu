// tp_hermitian.cu -- the symmetrised zero-frequency axis of accumulated
// half-spectra (TP_FLAG_HERMITIAN_X0, tp_hermitian_x0).
//
// "torch-projectors: A High-Performance Differentiable Projection Library
// for PyTorch" has its backward pass accumulate the contributions on the
// kx = 0 axis symmetrically, so that a Fourier coefficient of a real object
// and its conjugate partner are not counted twice with different values
// ([ar §2] Friedel symmetry, backward pass; [de §2 "Friedel-Symmetrie"]).
// With no formula on the pages, the reading taken is the Hermitian part of
// the stored kx = 0 plane (3D) or column (2D):
//   V(0, k) <- (V(0, k) + conj(V(0, -k))) / 2,   W(0, k) <- (W(0, k) + W(0, -k)) / 2,
// -k taken modulo the box in every stored axis (rfftn row order).  One
// thread per pair {k, -k}: the lower of the two plane indices does both.
// The plane holds M^2 (3D) or M (2D) of the spectrum's elements, so this is
// a small strided pass after the scatter.
#include <cuda_runtime.h>

#include "tp_launch.h"

namespace tp {

namespace {

__global__ void __launch_bounds__(256) k_hermitian_x0(float2 *__restrict__ V, float *__restrict__ W,
                                                      int B, int M, int X, int dim,
                                                      long long stride, unsigned *dbg) {
    const long long plane = dim == 3 ? (long long)M * M : M;
    const long long total = (long long)B * plane;
    for (long long t = (long long)blockIdx.x * 256 + threadIdx.x; t < total;
         t += (long long)gridDim.x * 256) {
        const int b = (int)(t / plane);
        const long long j = t - (long long)b * plane;
        long long jm;
        if (dim == 3) {
            const int z = (int)(j / M), y = (int)(j - (long long)z * M);
            jm = (long long)((M - z) % M) * M + (M - y) % M;
        } else {
            jm = (M - (int)j) % M;
        }
        if (jm < j) continue;   // the pair belongs to the lower index
        const long long e = (long long)b * stride + j * X, em = (long long)b * stride + jm * X;
        if (!TP_CHECK(dbg, j * X < stride && jm * X < stride, 6)) continue;
        if (V) {
            const float2 a = V[e], c = V[em];
            const float2 h = make_float2(0.5f * (a.x + c.x), 0.5f * (a.y - c.y));
            V[e] = h;
            V[em] = make_float2(h.x, -h.y);   // equals h when em == e (h.y is 0 there)
        }
        if (W) {
            const float h = 0.5f * (W[e] + W[em]);
            W[e] = h;
            W[em] = h;
        }
    }
}

}  // namespace

cudaError_t launch_hermitian_x0(float2 *V, float *W, int B, int M, int dim, cudaStream_t st,
                                unsigned *dbg) {
    if (B < 1 || (!V && !W)) return cudaSuccess;
    const int X = M / 2 + 1;
    const long long stride = (dim == 3 ? (long long)M * M : (long long)M) * X;
    const long long total = (long long)B * (dim == 3 ? (long long)M * M : M);
    long long blocks = (total + 255) / 256;
    if (blocks > 148LL * 16) blocks = 148LL * 16;
    k_hermitian_x0<<<(unsigned)blocks, 256, 0, st>>>(V, W, B, M, X, dim, stride, dbg);
    return cudaGetLastError();
}

}  // namespace tp
