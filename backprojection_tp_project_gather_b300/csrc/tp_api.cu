// tp_api.cu -- the exported C ABI (include/tp.h): argument validation,
// launch geometry and error reporting.  Every entry point validates first,
// then enqueues its kernels on the caller's stream and returns without
// synchronising.
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include "../../include/tp.h"
#include "tp_launch.h"

namespace {

thread_local char g_err[512] = "";

#ifdef TP_DEBUG_BOUNDS
// The bounds-check word of the debug build (see TP_CHECK), one per device.
__device__ unsigned g_dbg_word;

unsigned *dbg_word() {
    void *p = nullptr;
    return cudaGetSymbolAddress(&p, g_dbg_word) == cudaSuccess ? static_cast<unsigned *>(p)
                                                                : nullptr;
}

// A check that fails by construction and guards no access: it only sets
// bit `bit` of the word, so the reporting path can be tested on its own.
__global__ void k_check_selftest(unsigned *dbg, int bit) { (void)TP_CHECK(dbg, bit < 0, bit); }
#else
unsigned *dbg_word() { return nullptr; }
#endif

using tp::fail;

tp_status ok() {
    g_err[0] = '\0';
    return TP_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shared checks and parameter set-up for every operator.
struct Geometry {
    tp::Params q{};
    int dim = 3;
    bool cubic = false;
};

// allowed: the tp_options.flags bits the calling operator accepts.
tp_status setup(int dim, int Bsrc, int M, const float *rot, int Bp, int P, const float *shift,
                int Bs, int N, const tp_options &o, int Bout, Geometry &g, unsigned allowed = 0u) {
    if (o.flags & ~allowed)
        return fail(TP_ERR_UNSUPPORTED, "tp_options.flags 0x%x not supported by this operator%s",
                    o.flags & ~allowed,
                    (o.flags & TP_FLAG_HERMITIAN_X0)
                        ? " (TP_FLAG_HERMITIAN_X0 applies to accumulated spectra only)"
                        : "");
    if (o.interp != TP_LINEAR && o.interp != TP_CUBIC)
        return fail(TP_ERR_UNSUPPORTED, "interp must be TP_LINEAR or TP_CUBIC (got %d)", o.interp);
    if (!(o.oversampling > 0.0f) || !std::isfinite(o.oversampling))
        return fail(TP_ERR_UNSUPPORTED, "oversampling must be finite and > 0");
    if (!std::isfinite(o.radius)) return fail(TP_ERR_UNSUPPORTED, "radius must be finite");
    if (M < 2 || (M & 1) || N < 2 || (N & 1))
        return fail(TP_ERR_SHAPE, "box sizes must be even and >= 2 (source %d, output %d)", M, N);
    if (M > 4096 || N > 4096) return fail(TP_ERR_SHAPE, "box sizes above 4096 are not supported");
    if (P < 0 || Bsrc < 1 || Bp < 1 || Bs < 1 || Bout < 1)
        return fail(TP_ERR_SHAPE, "batch sizes must be >= 1 and P >= 0");
    if (dim == 3 && Bsrc > 65535)
        return fail(TP_ERR_SHAPE, "at most 65535 distinct volumes per call (got %d)", Bsrc);
    int B = Bout;
    if (Bsrc > B) B = Bsrc;
    if (Bp > B) B = Bp;
    if (shift && Bs > B) B = Bs;
    auto bc = [B](int b) { return b == 1 || b == B; };
    if (!bc(Bsrc) || !bc(Bp) || (shift && !bc(Bs)) || !bc(Bout))
        return fail(TP_ERR_SHAPE, "batch sizes do not broadcast (source %d, rot %d, shift %d, out %d)",
                    Bsrc, Bp, shift ? Bs : 1, Bout);
    if (!aligned(rot, 4) || (shift && !aligned(shift, 4)))
        return fail(TP_ERR_ALIGN, "rotation / shift pointers must be 4-byte aligned");
    const long long Xs = M / 2 + 1, Xo = N / 2 + 1;
    const long long src_elems = (dim == 3 ? (long long)M * M : (long long)M) * Xs;
    if (src_elems >= (1LL << 31)) return fail(TP_ERR_SHAPE, "source spectrum too large");
    const long long plane = (long long)N * Xo;
    const int threads = tp::kSampleBlock;
    const long long tiles = (plane + threads - 1) / threads;
    if ((long long)B * P * tiles >= (1LL << 31))
        return fail(TP_ERR_SHAPE, "too many samples for one launch (B*P*tiles = %lld)",
                    (long long)B * P * tiles);
    const double r = (o.radius < 0.0f) ? 0.5 * N : (double)o.radius;
    const double r2 = std::floor(r * r);
    tp::Params &q = g.q;
    q.src_stride = src_elems;
    q.Bsrc = Bsrc;
    q.M = M;
    q.Xs = (int)Xs;
    q.rot = rot;
    q.Bp = Bp;
    q.shift = shift;
    q.Bs = shift ? Bs : 1;
    q.P = P;
    q.B = B;
    q.N = N;
    q.Xo = (int)Xo;
    q.plane = (int)plane;
    q.tiles = (int)tiles;
    q.s = o.oversampling;
    q.fN = (float)N;
    q.invN = 1.0f / (float)N;
    q.r2max = r2 > 2e9 ? 2000000000 : (int)r2;
    q.mplane = (unsigned)((1ULL << 32) / (unsigned long long)plane);
    q.mxo = (unsigned)((1ULL << 32) / (unsigned long long)Xo);
    q.dbg = dbg_word();
    g.dim = dim;
    g.cubic = o.interp == TP_CUBIC;
    return TP_OK;
}

tp_status launched(cudaError_t e, const char *what) {
    if (e != cudaSuccess)
        return fail(TP_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
    return ok();
}

tp_status check_complex(const float *p, const char *name) {
    if (!aligned(p, 8)) return fail(TP_ERR_ALIGN, "%s must be 8-byte aligned (complex64)", name);
    return TP_OK;
}

// Workspace check for the 3D operators (the 2D ones need none).  lists: the
// call runs a scatter, whose sample lists follow the binning.
tp_status check_workspace(const Geometry &g, void *ws, size_t ws_bytes, bool lists) {
    if (g.dim != 3) return TP_OK;
    if (lists && (long long)g.q.B * g.q.P * g.q.plane >= (1LL << 31))
        return fail(TP_ERR_SHAPE, "too many output pixels for one scatter call (%lld); split the poses",
                    (long long)g.q.B * g.q.P * g.q.plane);
    if (lists && (long long)g.q.Bsrc * tp::brick_parts(g.q, g.cubic) >= (1LL << 31))
        return fail(TP_ERR_SHAPE, "too many volumes of this box for one scatter call; split the batch");
    const size_t need = lists ? tp::brick_workspace_bytes(g.q, g.cubic) : tp::brick_binning_bytes(g.q, g.cubic);
    if (!ws) return fail(TP_ERR_NULL, "workspace is required (%zu bytes, see tp_workspace_bytes)", need);
    if (!aligned(ws, 16)) return fail(TP_ERR_ALIGN, "workspace must be 16-byte aligned");
    if (ws_bytes < need)
        return fail(TP_ERR_SHAPE, "workspace too small: %zu bytes given, %zu needed", ws_bytes, need);
    return TP_OK;
}

// dout (3D only, may be NULL): also save D_a = phase * dS/dp_a per pixel.
tp_status forward(int dim, const float *src, int Bsrc, int M, const float *rot, int Bp, int P,
                  const float *shift, int Bs, int N, tp_options opts, float *out, float *dout,
                  void *ws, size_t ws_bytes, void *stream) {
    Geometry g;
    tp_status st = setup(dim, Bsrc, M, rot, Bp, P, shift, Bs, N, opts, 1, g);
    if (st != TP_OK) return st;
    if (P == 0) return ok();  // zero-size tensors may carry NULL pointers
    if (!src || !out || !rot) return fail(TP_ERR_NULL, "source, rotation and output pointers are required");
    if ((st = check_complex(src, "source")) != TP_OK || (st = check_complex(out, "out")) != TP_OK)
        return st;
    if (dout && (st = check_complex(dout, "dout")) != TP_OK) return st;
    if ((st = check_workspace(g, ws, ws_bytes, false)) != TP_OK) return st;
    g.q.src = reinterpret_cast<const float2 *>(src);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float2 *o = reinterpret_cast<float2 *>(out);
    return launched(dim == 3 ? tp::launch_brick_project(g.cubic, g.q, o, reinterpret_cast<float2 *>(dout),
                                                        ws, tp::kBinNew, s)
                             : tp::plane2d_fits(M, N) ? tp::launch_plane2d_project(g.cubic, g.q, o, s)
                                                   : tp::launch_project_2d(g.cubic, g.q, o, s),
                    "project");
}

tp_status backward(int dim, const float *grad_out, const float *src, int Bsrc, int M,
                   const float *rot, int Bp, int P, const float *shift, int Bs, int N,
                   tp_options opts, float *grad_src, float *grad_rot, float *grad_shift, void *ws,
                   size_t ws_bytes, void *stream) {
    Geometry g;
    tp_status st = setup(dim, Bsrc, M, rot, Bp, P, shift, Bs, N, opts, 1, g, TP_FLAG_HERMITIAN_X0);
    if (st != TP_OK) return st;
    if (P == 0) return ok();  // zero-size tensors may carry NULL pointers
    if (!grad_out || !rot) return fail(TP_ERR_NULL, "grad_out and rotation pointers are required");
    if ((grad_rot || grad_shift) && !src)
        return fail(TP_ERR_NULL, "the source spectrum is required for rotation / shift gradients");
    if (grad_shift && !shift) return fail(TP_ERR_NULL, "grad_shift requested without a shift tensor");
    if ((st = check_complex(grad_out, "grad_out")) != TP_OK) return st;
    if (src && (st = check_complex(src, "source")) != TP_OK) return st;
    if (grad_src && (st = check_complex(grad_src, "grad of the source")) != TP_OK) return st;
    if ((grad_rot && !aligned(grad_rot, 4)) || (grad_shift && !aligned(grad_shift, 4)))
        return fail(TP_ERR_ALIGN, "grad_rot / grad_shift must be 4-byte aligned");
    if ((st = check_workspace(g, ws, ws_bytes, grad_src != nullptr)) != TP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    tp::BinMode mode = tp::kBinNew;
    if (grad_rot || grad_shift) {
        g.q.src = reinterpret_cast<const float2 *>(src);
        const float2 *go = reinterpret_cast<const float2 *>(grad_out);
        cudaError_t e = dim == 3
                            ? tp::launch_brick_pose_grad(g.cubic, g.q, go, grad_rot, grad_shift, ws,
                                                         mode, s)
                            : tp::plane2d_fits(M, N)
                                ? tp::launch_plane2d_pose_grad(g.cubic, g.q, go, grad_rot, grad_shift, s)
                                : tp::launch_pose_grad_2d(g.cubic, g.q, go, grad_rot, grad_shift, s);
        if (e != cudaSuccess) return launched(e, "pose gradient");
        if (mode == tp::kBinNew) mode = tp::kBinSameCall;
    }
    if (grad_src) {
        g.q.src = nullptr;
        const float2 *go = reinterpret_cast<const float2 *>(grad_out);
        float2 *gs = reinterpret_cast<float2 *>(grad_src);
        cudaError_t e = dim == 3
                            ? tp::launch_brick_scatter(g.cubic, g.q, go, nullptr, gs, nullptr, ws,
                                                       mode, s)
                            : tp::launch_scatter_2d(g.cubic, g.q, go, gs, s);
        if (e != cudaSuccess) return launched(e, "spectrum gradient");
        if (opts.flags & TP_FLAG_HERMITIAN_X0) {
            e = tp::launch_hermitian_x0(gs, nullptr, Bsrc, M, dim, s, g.q.dbg);
            if (e != cudaSuccess) return launched(e, "zero-axis symmetrisation");
        }
    }
    return ok();
}

}  // namespace

namespace tp {

// Workspace bytes of the 3D operators; lists: with the scatters' sample
// lists (every operator), else the binning alone (the forward).
size_t workspace_bytes(int Bv, int B, int P, int Nv, int N, tp_options opts, bool lists) {
    if (Bv < 1 || B < 1 || P < 1 || Nv < 2 || (Nv & 1) || Nv > 4096 || N < 2 || (N & 1) || N > 4096 ||
        Bv > B)
        return 0;
    tp::Params q{};
    q.Bsrc = Bv;
    q.B = B;
    q.P = P;
    q.M = Nv;
    q.N = N;
    const bool cubic = opts.interp == TP_CUBIC;
    return lists ? tp::brick_workspace_bytes(q, cubic) : tp::brick_binning_bytes(q, cubic);
}

tp_status fail(tp_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

}  // namespace tp

extern "C" {

size_t tp_workspace_bytes(int Bv, int B, int P, int Nv, int N, tp_options opts) {
    return tp::workspace_bytes(Bv, B, P, Nv, N, opts, true);
}

tp_status tp_project_3d_2d(const float *vol, int Bv, int Nv, const float *rot, int Bp, int P,
                           const float *shift, int Bs, int N, tp_options opts, float *out,
                           void *workspace, size_t workspace_bytes, void *stream) {
    return forward(3, vol, Bv, Nv, rot, Bp, P, shift, Bs, N, opts, out, nullptr, workspace,
                   workspace_bytes, stream);
}

tp_status tp_project_3d_2d_save(const float *vol, int Bv, int Nv, const float *rot, int Bp, int P,
                                const float *shift, int Bs, int N, tp_options opts, float *out,
                                float *dout, void *workspace, size_t workspace_bytes,
                                void *stream) {
    if (!dout && P > 0) return fail(TP_ERR_NULL, "dout is required");
    return forward(3, vol, Bv, Nv, rot, Bp, P, shift, Bs, N, opts, out, dout, workspace,
                   workspace_bytes, stream);
}

tp_status tp_project_3d_2d_l2(const float *vol, int Bv, int Nv, const float *rot, int Bp, int P,
                              const float *shift, int Bs, int N, tp_options opts,
                              const float *target, float *out, float *grad_out, float *grad_rot,
                              float *grad_shift, void *workspace, size_t workspace_bytes,
                              void *stream) {
    Geometry g;
    tp_status st = setup(3, Bv, Nv, rot, Bp, P, shift, Bs, N, opts, 1, g);
    if (st != TP_OK) return st;
    if (P == 0) return ok();  // zero-size tensors may carry NULL pointers
    if (!vol || !rot || !target || !out || !grad_out)
        return fail(TP_ERR_NULL, "vol, rotation, target, out and grad_out pointers are required");
    if (grad_shift && !shift) return fail(TP_ERR_NULL, "grad_shift requested without a shift tensor");
    if ((st = check_complex(vol, "vol")) != TP_OK || (st = check_complex(target, "target")) != TP_OK ||
        (st = check_complex(out, "out")) != TP_OK || (st = check_complex(grad_out, "grad_out")) != TP_OK)
        return st;
    if ((grad_rot && !aligned(grad_rot, 4)) || (grad_shift && !aligned(grad_shift, 4)))
        return fail(TP_ERR_ALIGN, "grad_rot / grad_shift must be 4-byte aligned");
    if ((st = check_workspace(g, workspace, workspace_bytes, false)) != TP_OK) return st;
    g.q.src = reinterpret_cast<const float2 *>(vol);
    return launched(tp::launch_brick_project_l2(g.cubic, g.q, reinterpret_cast<const float2 *>(target),
                                                reinterpret_cast<float2 *>(out),
                                                reinterpret_cast<float2 *>(grad_out), grad_rot,
                                                grad_shift, workspace, static_cast<cudaStream_t>(stream)),
                    "project with L2 term");
}

tp_status tp_project_3d_2d_backward_saved(const float *grad_out, const float *out,
                                          const float *dout, int B, int P, int N, int Bp, int Bs,
                                          tp_options opts, float *grad_rot, float *grad_shift,
                                          void *stream) {
    if (opts.flags != 0) return fail(TP_ERR_UNSUPPORTED, "tp_options.flags must be 0 (got %u)", opts.flags);
    if (opts.interp != TP_LINEAR && opts.interp != TP_CUBIC)
        return fail(TP_ERR_UNSUPPORTED, "interp must be TP_LINEAR or TP_CUBIC (got %d)", opts.interp);
    if (!(opts.oversampling > 0.0f) || !std::isfinite(opts.oversampling))
        return fail(TP_ERR_UNSUPPORTED, "oversampling must be finite and > 0");
    if (!std::isfinite(opts.radius)) return fail(TP_ERR_UNSUPPORTED, "radius must be finite");
    if (N < 2 || (N & 1) || N > 4096) return fail(TP_ERR_SHAPE, "output box must be even, 2..4096 (got %d)", N);
    if (B < 1 || P < 0 || (Bp != 1 && Bp != B) || (Bs != 1 && Bs != B))
        return fail(TP_ERR_SHAPE, "batch sizes do not broadcast (B %d, rot %d, shift %d, P %d)", B, Bp,
                    Bs, P);
    const long long Xo = N / 2 + 1;
    if ((long long)B * P >= (1LL << 31) || (long long)B * P * N * Xo * 3 >= (1LL << 62))
        return fail(TP_ERR_SHAPE, "too many images (B*P = %lld)", (long long)B * P);
    if (P == 0 || (!grad_rot && !grad_shift)) return ok();
    if (!grad_out || !out || !dout)
        return fail(TP_ERR_NULL, "grad_out, out and dout pointers are required");
    tp_status st;
    if ((st = check_complex(grad_out, "grad_out")) != TP_OK || (st = check_complex(out, "out")) != TP_OK ||
        (st = check_complex(dout, "dout")) != TP_OK)
        return st;
    if ((grad_rot && !aligned(grad_rot, 4)) || (grad_shift && !aligned(grad_shift, 4)))
        return fail(TP_ERR_ALIGN, "grad_rot / grad_shift must be 4-byte aligned");
    tp::Params q{};
    q.B = B;
    q.P = P;
    q.Bp = Bp;
    q.Bs = Bs;
    q.N = N;
    q.Xo = (int)Xo;
    q.plane = (int)(N * Xo);
    q.s = opts.oversampling;
    q.fN = (float)N;
    q.invN = 1.0f / (float)N;
    const double r = (opts.radius < 0.0f) ? 0.5 * N : (double)opts.radius;
    const double r2 = std::floor(r * r);
    q.r2max = r2 > 2e9 ? 2000000000 : (int)r2;
    q.dbg = dbg_word();
    return launched(tp::launch_pose_grad_saved(q, reinterpret_cast<const float2 *>(grad_out),
                                               reinterpret_cast<const float2 *>(out),
                                               reinterpret_cast<const float2 *>(dout), grad_rot,
                                               grad_shift, static_cast<cudaStream_t>(stream)),
                    "pose gradient (saved)");
}

tp_status tp_project_2d_2d(const float *img, int Bi, int Ni, const float *rot, int Bp, int P,
                           const float *shift, int Bs, int N, tp_options opts, float *out,
                           void *stream) {
    return forward(2, img, Bi, Ni, rot, Bp, P, shift, Bs, N, opts, out, nullptr, nullptr, 0, stream);
}

tp_status tp_project_3d_2d_backward(const float *grad_out, const float *vol, int Bv, int Nv,
                                    const float *rot, int Bp, int P, const float *shift, int Bs,
                                    int N, tp_options opts, float *grad_vol, float *grad_rot,
                                    float *grad_shift, void *workspace, size_t workspace_bytes,
                                    void *stream) {
    return backward(3, grad_out, vol, Bv, Nv, rot, Bp, P, shift, Bs, N, opts, grad_vol, grad_rot,
                    grad_shift, workspace, workspace_bytes, stream);
}

tp_status tp_project_2d_2d_backward(const float *grad_out, const float *img, int Bi, int Ni,
                                    const float *rot, int Bp, int P, const float *shift, int Bs,
                                    int N, tp_options opts, float *grad_img, float *grad_rot,
                                    float *grad_shift, void *stream) {
    return backward(2, grad_out, img, Bi, Ni, rot, Bp, P, shift, Bs, N, opts, grad_img, grad_rot,
                    grad_shift, nullptr, 0, stream);
}

tp_status tp_backproject_2d_3d(const float *proj, const float *weights, int B, int P, int N,
                               const float *rot, int Bp, const float *shift, int Bs, int Bv,
                               int Nv, tp_options opts, float *data_vol, float *weight_vol,
                               void *workspace, size_t workspace_bytes, void *stream) {
    Geometry g;
    tp_status st = setup(3, Bv, Nv, rot, Bp, P, shift, Bs, N, opts, B, g, TP_FLAG_HERMITIAN_X0);
    if (st != TP_OK) return st;
    if (g.q.B != B)
        return fail(TP_ERR_SHAPE, "operand batches (%d) exceed the image batch B = %d", g.q.B, B);
    if (P == 0) return ok();  // zero-size tensors may carry NULL pointers
    if (!proj || !data_vol || !rot)
        return fail(TP_ERR_NULL, "proj, rotation and data_vol pointers are required");
    if ((st = check_complex(proj, "proj")) != TP_OK ||
        (st = check_complex(data_vol, "data_vol")) != TP_OK)
        return st;
    if ((weights && !aligned(weights, 4)) || (weight_vol && !aligned(weight_vol, 4)))
        return fail(TP_ERR_ALIGN, "weights / weight_vol must be 4-byte aligned");
    if ((st = check_workspace(g, workspace, workspace_bytes, true)) != TP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float2 *dv = reinterpret_cast<float2 *>(data_vol);
    cudaError_t e = tp::launch_brick_scatter(g.cubic, g.q, reinterpret_cast<const float2 *>(proj),
                                             weights, dv, weight_vol, workspace, tp::kBinNew, s);
    if (e == cudaSuccess && (opts.flags & TP_FLAG_HERMITIAN_X0))
        e = tp::launch_hermitian_x0(dv, weight_vol, Bv, Nv, 3, s, g.q.dbg);
    return launched(e, "backproject");
}

size_t tp_backproject_backward_scratch_bytes(int Bv, int B, int P, int N, int Nv,
                                             int with_weight_grad) {
    if (Bv < 1 || B < 1 || P < 1 || N < 2 || (N & 1) || Nv < 2 || (Nv & 1) || N > 4096 ||
        Nv > 4096 || Bv > B)
        return 0;
    auto a256 = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t img = (size_t)B * P * N * (N / 2 + 1);
    size_t bytes = a256(8 * img) + a256(24 * img);                        // y, D
    if (with_weight_grad)
        bytes += a256(8 * (size_t)Bv * Nv * Nv * (Nv / 2 + 1)) + a256(8 * img);   // GW + 0i, y_W
    return bytes;
}

tp_status tp_backproject_2d_3d_backward(const float *grad_data_vol, const float *grad_weight_vol,
                                        const float *proj, const float *weights, int B, int P,
                                        int N, const float *rot, int Bp, const float *shift, int Bs,
                                        int Bv, int Nv, tp_options opts, float *grad_proj,
                                        float *grad_weights, float *grad_rot, float *grad_shift,
                                        void *scratch, size_t scratch_bytes, void *workspace,
                                        size_t workspace_bytes, void *stream) {
    if (opts.flags & TP_FLAG_HERMITIAN_X0)
        return fail(TP_ERR_UNSUPPORTED,
                    "TP_FLAG_HERMITIAN_X0: the gradients of a symmetrised backprojection are those of "
                    "the plain one at symmetrised upstream gradients (apply tp_hermitian_x0 to them)");
    Geometry g;
    tp_status st = setup(3, Bv, Nv, rot, Bp, P, shift, Bs, N, opts, B, g);
    if (st != TP_OK) return st;
    if (g.q.B != B)
        return fail(TP_ERR_SHAPE, "operand batches (%d) exceed the image batch B = %d", g.q.B, B);
    if (P == 0) return ok();  // zero-size tensors may carry NULL pointers
    if (!rot) return fail(TP_ERR_NULL, "rotation pointer is required");
    const bool data_terms = grad_proj || grad_shift || (grad_rot && grad_data_vol);
    if (data_terms && !grad_data_vol)
        return fail(TP_ERR_NULL, "grad_proj / grad_shift need grad_data_vol");
    if (grad_weights && !grad_weight_vol)
        return fail(TP_ERR_NULL, "grad_weights needs grad_weight_vol");
    if ((grad_rot || grad_shift) && !proj)
        return fail(TP_ERR_NULL, "rotation / shift gradients need proj");
    if (grad_shift && !shift) return fail(TP_ERR_NULL, "grad_shift requested without a shift tensor");
    if ((grad_data_vol && (st = check_complex(grad_data_vol, "grad_data_vol")) != TP_OK) ||
        (proj && (st = check_complex(proj, "proj")) != TP_OK) ||
        (grad_proj && (st = check_complex(grad_proj, "grad_proj")) != TP_OK))
        return st;
    if ((grad_weight_vol && !aligned(grad_weight_vol, 4)) || (weights && !aligned(weights, 4)) ||
        (grad_weights && !aligned(grad_weights, 4)) || (grad_rot && !aligned(grad_rot, 4)) ||
        (grad_shift && !aligned(grad_shift, 4)))
        return fail(TP_ERR_ALIGN, "real arrays must be 4-byte aligned");
    const bool weight_terms = grad_weight_vol && (grad_weights || grad_rot);
    if (!data_terms && !weight_terms) return ok();
    if ((st = check_workspace(g, workspace, workspace_bytes, false)) != TP_OK) return st;
    const size_t need = tp_backproject_backward_scratch_bytes(Bv, B, P, N, Nv, weight_terms ? 1 : 0);
    if (!scratch) return fail(TP_ERR_NULL, "scratch is required (%zu bytes)", need);
    if (!aligned(scratch, 16)) return fail(TP_ERR_ALIGN, "scratch must be 16-byte aligned");
    if (scratch_bytes < need)
        return fail(TP_ERR_SHAPE, "scratch too small: %zu bytes given, %zu needed", scratch_bytes, need);
    auto a256 = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t img = (size_t)B * P * N * (N / 2 + 1);
    char *base = static_cast<char *>(scratch);
    float2 *sy = reinterpret_cast<float2 *>(base);
    float2 *sD = reinterpret_cast<float2 *>(base + a256(8 * img));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (data_terms) {
        // P(G) (the images' gradient) and its saved derivatives, then the
        // pose gradients with the images as the upstream gradient.
        g.q.src = reinterpret_cast<const float2 *>(grad_data_vol);
        float2 *y = grad_proj ? reinterpret_cast<float2 *>(grad_proj) : sy;
        e = tp::launch_brick_project(g.cubic, g.q, y, (grad_rot || grad_shift) ? sD : nullptr,
                                     workspace, tp::kBinNew, s);
        if (e != cudaSuccess) return launched(e, "backprojection gradient (data)");
        if (grad_rot || grad_shift) {
            e = tp::launch_pose_grad_saved(g.q, reinterpret_cast<const float2 *>(proj), y, sD,
                                           grad_rot, grad_shift, s);
            if (e != cudaSuccess) return launched(e, "backprojection pose gradient (data)");
        }
    }
    if (weight_terms) {
        float2 *gw = reinterpret_cast<float2 *>(base + a256(8 * img) + a256(24 * img));
        float2 *yw = reinterpret_cast<float2 *>(reinterpret_cast<char *>(gw) +
                                                a256(8 * (size_t)Bv * Nv * Nv * (Nv / 2 + 1)));
        e = tp::launch_real_to_complex(grad_weight_vol, gw, (long long)Bv * g.q.src_stride, s);
        if (e != cudaSuccess) return launched(e, "backprojection gradient (weights)");
        tp::Params qw = g.q;   // the weight spectrum has no phase
        qw.src = gw;
        qw.shift = nullptr;
        qw.Bs = 1;
        e = tp::launch_brick_project(g.cubic, qw, yw, grad_rot ? sD : nullptr, workspace,
                                     tp::kBinNew, s);
        if (e != cudaSuccess) return launched(e, "backprojection gradient (weights)");
        e = tp::launch_weight_grads(qw, weights, yw, sD, grad_weights, grad_rot, s);
        if (e != cudaSuccess) return launched(e, "backprojection gradient (weights)");
    }
    return ok();
}

tp_status tp_hermitian_x0(float *spec, float *weight, int B, int N, int dim, void *stream) {
    if (dim != 2 && dim != 3) return fail(TP_ERR_UNSUPPORTED, "dim must be 2 or 3 (got %d)", dim);
    if (B < 0 || N < 2 || (N & 1) || N > 4096)
        return fail(TP_ERR_SHAPE, "box must be even, 2..4096 and B >= 0 (got N %d, B %d)", N, B);
    if (B == 0) return ok();
    if (!spec && !weight) return fail(TP_ERR_NULL, "spec or weight is required");
    tp_status st;
    if (spec && (st = check_complex(spec, "spec")) != TP_OK) return st;
    if (weight && !aligned(weight, 4)) return fail(TP_ERR_ALIGN, "weight must be 4-byte aligned");
    return launched(tp::launch_hermitian_x0(reinterpret_cast<float2 *>(spec), weight, B, N, dim,
                                            static_cast<cudaStream_t>(stream), dbg_word()),
                    "zero-axis symmetrisation");
}

unsigned tp_debug_bounds_word(int reset) {
#ifdef TP_DEBUG_BOUNDS
    unsigned w = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return ~0u;
    if (cudaMemcpyFromSymbol(&w, g_dbg_word, sizeof w) != cudaSuccess) return ~0u;
    if (reset) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_dbg_word, &zero, sizeof zero) != cudaSuccess) return ~0u;
    }
    return w;
#else
    (void)reset;
    return 0u;
#endif
}

tp_status tp_debug_bounds_selftest(int bit, void *stream) {
#ifdef TP_DEBUG_BOUNDS
    if (bit < 0 || bit > 31) return fail(TP_ERR_SHAPE, "bit must be in [0, 31] (got %d)", bit);
    unsigned *w = dbg_word();
    if (!w) return fail(TP_ERR_CUDA, "no bounds-check word on this device");
    k_check_selftest<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(w, bit);
    return launched(cudaGetLastError(), "bounds-check self-test");
#else
    (void)bit;
    (void)stream;
    return fail(TP_ERR_UNSUPPORTED, "not a bounds-checking build (TP_DEBUG_BOUNDS)");
#endif
}

const char *tp_last_error(void) { return g_err; }

const char *tp_version(void) { return "0.1.0"; }

}  // extern "C"
