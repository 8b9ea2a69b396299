// tp_noalloc.cu -- tp_project_3d_2d_noalloc: the 3D forward projection for
// callers that cannot allocate device memory.
//
// Why.  tp_project_3d_2d needs a few hundred kilobytes to a few megabytes of
// scratch (pose geometry and pose-to-brick bitmasks) that the caller passes
// as a workspace.  Some callers cannot provide one: code that must not call
// cudaMalloc (for example inside a CUDA-graph capture, or under an
// allocator that forbids it), or hosts that manage no device memory of
// their own.  This entry point takes the same inputs and outputs but keeps
// its scratch in a fixed array in the library's own device memory.
//
// Trade-offs a caller accepts:
//  - every GPU that loads the library reserves kMaxScratch bytes for that
//    array until the process exits;
//  - problems whose scratch would exceed kMaxScratch are rejected;
//  - all calls share the one array, so calls that overlap on the GPU (on
//    different streams, or from different threads) corrupt each other's
//    scratch and must be serialised by the caller;
//  - the first call on each device looks the array's address up (set-up
//    below), which can load the module; make that first call before any
//    stream capture;
//  - the address is kept for the life of the process, so after a
//    cudaDeviceReset() of a device this entry point must not be called on
//    that device again.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/tp.h"
#include "tp_launch.h"

namespace {

// Largest scratch this entry point can use: 16 MiB covers, for example,
// 4096 poses against a 256^3 volume (about 3.4 MB).
constexpr size_t kMaxScratch = 16u << 20;

// The scratch itself.  Host code must not use this name as an address:
// on the host it is a stand-in object, not device memory.  Device code in
// this file could name it directly; the kernels get its address instead.
static __device__ __align__(256) unsigned char g_scratch[kMaxScratch];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per
// device with that device current.
cudaError_t scratch_address(void **ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

tp_status tp_project_3d_2d_noalloc(const float *vol, int Bv, int Nv, const float *rot, int Bp,
                                   int P, const float *shift, int Bs, int N, tp_options opts,
                                   float *out, void *stream) {
    if (P == 0) return tp_project_3d_2d(vol, Bv, Nv, rot, Bp, P, shift, Bs, N, opts, out, nullptr,
                                        0, stream);
    int B = Bv > Bp ? Bv : Bp;
    if (shift && Bs > B) B = Bs;
    const size_t need = tp::workspace_bytes(Bv, B, P, Nv, N, opts, false);   // the forward's part
    if (need > kMaxScratch)
        return tp::fail(TP_ERR_SHAPE,
                        "tp_project_3d_2d_noalloc: this problem needs %zu bytes of scratch, the "
                        "fixed array holds %zu; use tp_project_3d_2d with a workspace",
                        need, kMaxScratch);
    void *scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess)
        return tp::fail(TP_ERR_CUDA, "tp_project_3d_2d_noalloc: scratch set-up failed: %s",
                        cudaGetErrorString(e));
    // Same validation, kernels and error reporting as tp_project_3d_2d.
    return tp_project_3d_2d(vol, Bv, Nv, rot, Bp, P, shift, Bs, N, opts, out, scratch,
                            kMaxScratch, stream);
}

}  // extern "C"
