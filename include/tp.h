/*
 * tp.h -- C ABI of the B300 Fourier-space projection library (libtp_b300.so).
 *
 * The operators are the ones named on the summary pages of "torch-projectors:
 * A High-Performance Differentiable Projection Library for PyTorch"
 * (D. Tegunov, 2026), cited by language and by the section of each page's
 * technical summary ([de §2] = German page, section 2, and so on).
 *
 * ---------------------------------------------------------------------------
 * Conventions shared by every entry point
 * ---------------------------------------------------------------------------
 * Memory.  Every array argument is a DEVICE pointer to C-contiguous memory
 * owned by the caller.  The library allocates nothing, keeps no state between
 * calls except a per-thread error message, and never synchronises: each call
 * enqueues its kernels on `stream` (a cudaStream_t; NULL = the legacy default
 * stream) and returns.  Results are ready when the stream reaches that point.
 *
 * Complex arrays are interleaved (re, im) float pairs (PyTorch complex64) and
 * must be 8-byte aligned; real arrays are float32 and 4-byte aligned.
 *
 * Half-spectrum layout [it §2 "Spazio di Fourier e Formati"; ar §2]:
 *   3D spectrum of box M: (M, M, M/2+1) indexed [z][y][x];
 *   2D spectrum / image of box N: (N, N/2+1) indexed [y][x];
 * exactly the output of torch.fft.rfftn / rfft2 (no fftshift).  Row i of a
 * box-M axis holds frequency i for i < M/2, else i - M.  Box sizes are even.
 *
 * Geometry.  Output pixel (iy, ix) has frequency k = (ix, ky(iy)).  It is
 * sampled at p = s * R^T k (p_j = s * sum_i R[i][j] k_i, k_z = 0 in 3D): the
 * coordinates go through the inverse rotation [ko §2 "Forward Projection"].
 * R is row-major (3x3 or 2x2) and need not be orthogonal.  s is
 * tp_options.oversampling.  Pixels with kx^2 + ky^2 > radius^2 are zero and
 * scatter nothing.
 *
 * Interpolation [it §2 "Interpolazione"; ko §2 "보간법"]: per axis, linear
 * (taps floor(p), floor(p)+1, w = 1-|t|) or Catmull-Rom cubic (Keys kernel,
 * a = -1/2, taps floor(p)-1 .. floor(p)+2), t = p - tap, weight = product
 * over axes.  Friedel reads [ar §2 "التمرير الأمامي"]: a tap n with n_x < 0
 * reads conj(V[-n]).  Taps outside the stored range (0 <= n_x <= M/2,
 * -M/2 <= n_y, n_z <= M/2-1) read zero.
 *
 * Shift [de §2 "Interpolation"; ar §2]: the sample is multiplied by
 * exp(-2 pi i (kx sx + ky sy) / N), a real-space shift by (sx, sy) pixels.
 *
 * Batches [de §3 item 3].  B = max of the operand batch sizes; each operand
 * batch (Bv / Bi, Bp, Bs) is 1 (shared by all) or B.  P poses per batch
 * element.  Rotations are (Bp, P, d, d), shifts (Bs, P, 2) or NULL (= 0).
 *
 * Outputs.  Forward outputs are overwritten.  Backprojection and gradient
 * outputs are ACCUMULATED (+=) into caller-initialised memory, so that
 * several calls can add into one volume.  A NULL gradient pointer means
 * "not requested".  Gradients of a broadcast operand sum over the batch.
 * Gradients are with respect to the matrix entries and shift components
 * [de §3 item 4]; angle or quaternion chain rules belong to the caller.
 * Complex gradients follow PyTorch's convention: for a real loss L,
 * grad = dL/dRe + i dL/dIm, and each backward entry point applies the real
 * adjoint of the forward map's Jacobian.
 *
 * Workspace.  The 3D entry points bin poses against bricks of the volume in
 * a scratch area the caller provides: `workspace` must point to at least
 * tp_workspace_bytes(...) bytes of device memory, 16-byte aligned, owned by
 * the caller.  A call that finds in it the binning of identical poses and
 * sizes (its key and the pose records compared on the device, bit for bit:
 * for example the backward call after the forward call of one step) keeps
 * the brick masks and work units stored there instead of recomputing them;
 * any difference recomputes them.  The scatters (backprojection, spectrum
 * gradient) also sort the in-radius output pixels by brick part into lists
 * kept there under the same rule; the forward
 * entry points and the pose-gradient-only backward need only the binning,
 * the first part of the workspace (they accept any size that holds it).  So
 * the first 256 bytes of a workspace that is new to the library, or whose
 * memory served anything else since its last call, must be zero (the rest
 * needs no initialisation): memory recycled by an allocator can hold the
 * key and poses of an old workspace but other data in its masks.  It must
 * not be used by two calls that can run at the same time (one workspace
 * per stream).  A scatter call handles fewer than 2^31 output pixels
 * (B * P * N * (N/2+1)); larger ones fail with TP_ERR_SHAPE.
 *
 * Errors.  Each call returns a tp_status.  Argument errors are detected
 * before anything is enqueued; TP_ERR_CUDA reports a launch failure.  No
 * C++ exception crosses this interface.  tp_last_error() returns a message
 * for the calling thread's most recent failure.  Empty problems (P == 0)
 * succeed without launching anything.
 */
#ifndef TP_B300_H
#define TP_B300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TP_OK = 0,
    TP_ERR_NULL = 1,        /* a required pointer is NULL */
    TP_ERR_SHAPE = 2,       /* bad size, odd box, batch that does not broadcast */
    TP_ERR_ALIGN = 3,       /* pointer not aligned to its element type */
    TP_ERR_UNSUPPORTED = 4, /* option value not supported */
    TP_ERR_CUDA = 5,        /* a kernel launch failed (message has the CUDA error) */
    TP_ERR_INTERNAL = 6
} tp_status;

enum { TP_LINEAR = 0, TP_CUBIC = 1 };

/*
 * Option flags (tp_options.flags).
 *
 * TP_FLAG_HERMITIAN_X0: symmetrise the zero-frequency axis of an accumulated
 * spectrum.  The pages' backward pass accumulates the contributions on the
 * kx = 0 axis symmetrically, so that a Fourier coefficient of a real object
 * and its conjugate partner are not counted twice with different values
 * ([ar §2] Friedel symmetry, backward pass; [de §2 "Friedel-Symmetrie"]).
 * They give no formula; this library takes the Hermitian part of the stored
 * kx = 0 plane (3D) or column (2D) after the accumulation:
 *   V(0, k) <- (V(0, k) + conj(V(0, -k))) / 2,  W(0, k) <- (W(0, k) + W(0, -k)) / 2
 * with -k taken modulo the box in every stored axis (self-conjugate points
 * keep their real part); every other coefficient is unchanged.  The whole
 * plane is symmetrised, including what the output held before the call.
 * Accepted by tp_backproject_2d_3d (data and weight spectra),
 * tp_project_3d_2d_backward (grad_vol) and tp_project_2d_2d_backward
 * (grad_img); other outputs of those calls are unaffected.  Without it
 * (the default) the backward operators are the exact real adjoint of the
 * forward on any input; with it they are the adjoint of the forward
 * restricted to spectra of real objects (Hermitian on kx = 0), which the
 * symmetrisation leaves unchanged.  The forward operators and
 * tp_project_3d_2d_backward_saved reject it (TP_ERR_UNSUPPORTED), as does
 * tp_backproject_2d_3d_backward: the gradients of a symmetrised
 * backprojection are the plain ones at symmetrised upstream gradients
 * (tp_hermitian_x0 applied to them; the symmetrisation is self-adjoint).
 */
#define TP_FLAG_HERMITIAN_X0 1u

typedef struct {
    int interp;         /* TP_LINEAR or TP_CUBIC */
    float oversampling; /* s > 0: sample position p = s * R^T k */
    float radius;       /* cutoff in output-pixel frequency units; < 0 means N/2 */
    unsigned flags;     /* TP_FLAG_* bits where the operator accepts them, else 0 */
} tp_options;

/*
 * 3D -> 2D forward projection: central slices of a 3D half-spectrum
 * [it §2 "Operazioni Supportate"; de §2 "Unterstützte Operationen" item 3;
 * ja §2 "演算の種類"].
 *   vol    (Bv, Nv, Nv, Nv/2+1) complex        in
 *   rot    (Bp, P, 3, 3) float                  in
 *   shift  (Bs, P, 2) float, or NULL            in
 *   out    (B, P, N, N/2+1) complex             out, overwritten
 */
tp_status tp_project_3d_2d(const float *vol, int Bv, int Nv,
                           const float *rot, int Bp, int P,
                           const float *shift, int Bs,
                           int N, tp_options opts, float *out,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * Gradients through tp_project_3d_2d for an upstream gradient grad_out
 * (B, P, N, N/2+1) complex [de §2 "Differentiable Backpropagation"; ko §2
 * "그라디언트 계산"; ar §2 "الإزاحات والدورات"].
 *   grad_vol    (Bv, Nv, Nv, Nv/2+1) complex, += adjoint applied to grad_out
 *   grad_rot    (Bp, P, 3, 3) float, += dL/dR (row 3 is always 0: k_z = 0)
 *   grad_shift  (Bs, P, 2) float, += dL/dshift; requires shift != NULL
 * Any of the three may be NULL.  opts.flags may hold TP_FLAG_HERMITIAN_X0
 * (applied to grad_vol after the accumulation).
 */
tp_status tp_project_3d_2d_backward(const float *grad_out, const float *vol, int Bv, int Nv,
                                    const float *rot, int Bp, int P,
                                    const float *shift, int Bs, int N, tp_options opts,
                                    float *grad_vol, float *grad_rot, float *grad_shift,
                                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * tp_project_3d_2d that also saves what the rotation and shift gradients
 * need, so that tp_project_3d_2d_backward_saved gets them without touching
 * the volume again (a save-for-backward split of the gradients of [de §2
 * "Differentiable Backpropagation"; ar §2 "الإزاحات والدورات"]; the pages
 * recompute instead).  Arguments, out and errors as tp_project_3d_2d, plus
 *   dout   (B, P, N, N/2+1, 3) complex          out, overwritten
 * with dout[b][p][y][x][a] = phase * dS/dp_a, the derivative of out[b][p][y][x]
 * with respect to component a of the pixel's sample position p = s R^T k
 * (zero where out is zero by the radius).  dout must be 8-byte aligned.
 */
tp_status tp_project_3d_2d_save(const float *vol, int Bv, int Nv,
                                const float *rot, int Bp, int P,
                                const float *shift, int Bs,
                                int N, tp_options opts, float *out, float *dout,
                                void *workspace, size_t workspace_bytes, void *stream);

/*
 * Rotation and shift gradients of a tp_project_3d_2d_save forward for an
 * upstream gradient grad_out, from its out and dout alone (no volume and no
 * workspace): per pixel dL/dp_a = Re(conj(grad_out) dout_a), then
 *   grad_rot    (Bp, P, 3, 3) float, += s k_i dL/dp_a at [i][a] (row 3 is 0)
 *   grad_shift  (Bs, P, 2) float, += (2 pi k_a / N) Im(conj(grad_out) out)
 * the same values as tp_project_3d_2d_backward.  grad_out, out (B, P, N,
 * N/2+1) and dout are complex; B is the output batch, Bp and Bs (each 1 or
 * B) the rotation and shift batches of the forward (Bs = 1 when it had no
 * shift; grad_shift is then the gradient at zero shift).  opts must be the
 * forward's (oversampling and radius are used).  Either gradient may be
 * NULL; with both NULL the call does nothing.
 */
tp_status tp_project_3d_2d_backward_saved(const float *grad_out, const float *out,
                                          const float *dout, int B, int P, int N,
                                          int Bp, int Bs, tp_options opts,
                                          float *grad_rot, float *grad_shift, void *stream);

/*
 * tp_project_3d_2d fused with an L2 data term L = sum over all stored pixels
 * of |out - target|^2: one pass that gives the forward output, the residual
 * gradient and the rotation and shift gradients of L.  The pages train the
 * projection through losses the caller writes ([de §2 "Differentiable
 * Backpropagation"]); this entry point fuses the most common one so that
 * the rotation and shift gradients come from the forward's own gather of the
 * stencil derivatives, with nothing saved for a later pass.  Arguments and
 * errors as tp_project_3d_2d, plus
 *   target      (B, P, N, N/2+1) complex                      in
 *   out         (B, P, N, N/2+1) complex, overwritten: the projection
 *   grad_out    (B, P, N, N/2+1) complex, overwritten: dL/dout = 2 (out - target)
 *               (PyTorch's complex convention), also where out is 0 by the radius
 *   grad_rot    (Bp, P, 3, 3) float, += dL/dR (row 3 is 0), or NULL
 *   grad_shift  (Bs, P, 2) float, += dL/dshift, or NULL; requires shift != NULL
 * The rotation and shift gradients equal those of tp_project_3d_2d_backward
 * for upstream gradient grad_out; the volume gradient is
 * tp_project_3d_2d_backward of grad_out (the binning in the workspace is kept
 * for it).  target, out and grad_out must be 8-byte aligned.
 */
tp_status tp_project_3d_2d_l2(const float *vol, int Bv, int Nv,
                              const float *rot, int Bp, int P,
                              const float *shift, int Bs,
                              int N, tp_options opts, const float *target,
                              float *out, float *grad_out, float *grad_rot, float *grad_shift,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * 2D -> 3D backprojection: the adjoint of tp_project_3d_2d scattered into a
 * data spectrum, plus an optional real weight spectrum [it §2 "accumulo di
 * pesi"; de §2 "Dual-Volumen-Ansatz"; ko §2 "Backward Projection"].
 *   proj        (B, P, N, N/2+1) complex                      in
 *   weights     (B, P, N, N/2+1) float, or NULL (= 1)         in
 *   rot         (Bp, P, 3, 3);  shift (Bs, P, 2) or NULL      in
 *   data_vol    (Bv, Nv, Nv, Nv/2+1) complex, +=              out
 *   weight_vol  (Bv, Nv, Nv, Nv/2+1) float, +=, or NULL       out
 * A direct tap adds w * conj(phase) * proj to data_vol[n]; a Friedel tap adds
 * the conjugate of that to data_vol[-n]; weight_vol gets w * weight at the
 * same location.  Bv is 1 (all batch elements add into one volume) or B.
 * opts.flags may hold TP_FLAG_HERMITIAN_X0 (applied to both spectra after
 * the accumulation).
 */
tp_status tp_backproject_2d_3d(const float *proj, const float *weights, int B, int P, int N,
                               const float *rot, int Bp, const float *shift, int Bs,
                               int Bv, int Nv, tp_options opts,
                               float *data_vol, float *weight_vol,
                               void *workspace, size_t workspace_bytes, void *stream);

/*
 * Gradients of tp_backproject_2d_3d for upstream gradients of its data and
 * weight spectra (the gradient of the backprojection "with respect to all
 * inputs" [de §2 "Differentiable Backpropagation"] and through the weight
 * spectrum [ar §2]).  The backprojection is the real adjoint of
 * tp_project_3d_2d, so with G = grad_data_vol and GW = grad_weight_vol:
 *   grad_proj     (B, P, N, N/2+1) complex = the projection of G (with the
 *                 shift phase), WRITTEN, not accumulated;
 *   grad_weights  (B, P, N, N/2+1) float = Re of the unshifted projection of
 *                 GW, WRITTEN; needs grad_weight_vol;
 *   grad_rot      (Bp, P, 3, 3) float, += the rotation gradient of the
 *                 projection of G for upstream proj, plus (with GW) that of
 *                 the unshifted projection of GW for upstream weights (1 when
 *                 weights is NULL);
 *   grad_shift    (Bs, P, 2) float, += the shift gradient of the projection
 *                 of G for upstream proj; requires shift != NULL.
 * Any output may be NULL.  grad_data_vol (Bv, Nv, Nv, Nv/2+1) complex is
 * required for grad_proj and grad_shift, proj for grad_rot / grad_shift;
 * grad_weight_vol (same shape, float) may be NULL (no weight terms).  The
 * other arguments are those of tp_backproject_2d_3d.  scratch: at least
 * tp_backproject_backward_scratch_bytes(Bv, B, P, N, Nv, weight terms?) bytes
 * of device memory, 16-byte aligned, owned by the caller; workspace as for
 * the other 3D calls.  opts.flags must be 0 (see TP_FLAG_HERMITIAN_X0).
 */
tp_status tp_backproject_2d_3d_backward(const float *grad_data_vol, const float *grad_weight_vol,
                                        const float *proj, const float *weights, int B, int P,
                                        int N, const float *rot, int Bp, const float *shift, int Bs,
                                        int Bv, int Nv, tp_options opts, float *grad_proj,
                                        float *grad_weights, float *grad_rot, float *grad_shift,
                                        void *scratch, size_t scratch_bytes, void *workspace,
                                        size_t workspace_bytes, void *stream);

/*
 * Scratch bytes tp_backproject_2d_3d_backward needs (with_weight_grad != 0
 * when grad_weight_vol is given and grad_weights or grad_rot is requested);
 * 0 for invalid sizes.
 */
size_t tp_backproject_backward_scratch_bytes(int Bv, int B, int P, int N, int Nv,
                                             int with_weight_grad);

/*
 * 2D -> 2D forward: rotated and shifted 2D half-spectra
 * [it §2 "Operazioni Supportate"; de §2 item 1; ja §2].
 *   img    (Bi, Ni, Ni/2+1) complex;  rot (Bp, P, 2, 2);  shift (Bs, P, 2) or NULL
 *   out    (B, P, N, N/2+1) complex, overwritten
 */
tp_status tp_project_2d_2d(const float *img, int Bi, int Ni,
                           const float *rot, int Bp, int P,
                           const float *shift, int Bs,
                           int N, tp_options opts, float *out, void *stream);

/*
 * Gradients through tp_project_2d_2d [de §2 item 4 "2D -> 2D Backward"].
 *   grad_img    (Bi, Ni, Ni/2+1) complex, +=
 *   grad_rot    (Bp, P, 2, 2) float, +=
 *   grad_shift  (Bs, P, 2) float, +=; requires shift != NULL
 * opts.flags may hold TP_FLAG_HERMITIAN_X0 (applied to grad_img after the
 * accumulation).
 */
tp_status tp_project_2d_2d_backward(const float *grad_out, const float *img, int Bi, int Ni,
                                    const float *rot, int Bp, int P,
                                    const float *shift, int Bs, int N, tp_options opts,
                                    float *grad_img, float *grad_rot, float *grad_shift,
                                    void *stream);

/*
 * The symmetrisation of TP_FLAG_HERMITIAN_X0 on its own, in place, enqueued
 * on `stream`: the kx = 0 plane (dim 3: spec (B, N, N, N/2+1)) or column
 * (dim 2: spec (B, N, N/2+1)) of a complex spectrum and / or of a real
 * weight spectrum of the same shape.  Either pointer may be NULL, not both;
 * spec must be 8-byte aligned.  B == 0 does nothing.  Errors:
 * TP_ERR_UNSUPPORTED for dim other than 2 or 3, TP_ERR_SHAPE for an odd box
 * or one outside 2..4096, TP_ERR_NULL, TP_ERR_ALIGN.
 */
tp_status tp_hermitian_x0(float *spec, float *weight, int B, int N, int dim, void *stream);

/*
 * Bytes of workspace the 3D entry points need for a volume batch Bv, batch
 * B (Bv is 1 or B), P poses per batch element, volume box Nv, image box N
 * and the interpolation of opts: enough for every 3D entry point on these
 * sizes (the backward uses it for both of its passes).  This includes
 * 8 bytes per output pixel (B * P * N * (N/2+1)) for the scatters' sample
 * lists.  Returns 0 for invalid sizes.
 */
size_t tp_workspace_bytes(int Bv, int B, int P, int Nv, int N, tp_options opts);

/*
 * tp_project_3d_2d without a workspace, for callers that cannot allocate
 * device memory (no cudaMalloc allowed where they run, e.g. during a graph
 * capture or under a foreign allocator).  The paper has no counterpart: it
 * is an interface convenience of this library.  Arguments and results are
 * those of tp_project_3d_2d.  The scratch lives in a fixed 16 MiB array in
 * the library's device memory, reserved on every GPU that loads the
 * library until the process exits; problems whose binning (the forward's
 * part of tp_workspace_bytes) needs more than that fail with TP_ERR_SHAPE
 * (tp_last_error says why).
 * All calls share the array: calls that can overlap on the GPU race and
 * must be serialised by the caller.  The first call on each device looks
 * the array up (and may load the module); make it before any stream
 * capture.  The address found then is kept for the life of the process:
 * after cudaDeviceReset() of a device, do not call this entry point on that
 * device again.  No memory is allocated.
 */
tp_status tp_project_3d_2d_noalloc(const float *vol, int Bv, int Nv,
                                   const float *rot, int Bp, int P,
                                   const float *shift, int Bs,
                                   int N, tp_options opts, float *out, void *stream);

/*
 * Bounds checks of a debug build of this library (compiled with
 * -DTP_DEBUG_BOUNDS, libtp_b300_debug.so): waits for the current device and
 * returns the bits of the index checks that have failed since the last reset
 * (0 = none; a failed check skips its access).  reset != 0 clears the word.
 * The normal build checks nothing and returns 0; ~0u reports a CUDA error.
 * Bits: 0 source spectrum read, 1 staged-brick write, 2 staged tap read,
 * 3 output image row, 4 scatter accumulator tile, 5 weight accumulator
 * tile, 6 spectrum fold / scatter target, 7 image read, 8 workspace lists
 * (work units, pose masks, pose records), 9 rotation / shift gradient row,
 * 10 saved-derivative or weight-gradient row.
 */
unsigned tp_debug_bounds_word(int reset);

/*
 * Debug build only: enqueue on `stream` one check that fails by
 * construction and guards no memory access, so that bit `bit` (0..31) of
 * the word above is set.  Tests the reporting path itself.  Returns
 * TP_ERR_SHAPE for a bit outside 0..31 and TP_ERR_UNSUPPORTED in the
 * normal build (nothing is launched).
 */
tp_status tp_debug_bounds_selftest(int bit, void *stream);

/* Message for the calling thread's most recent failure ("" if none). */
const char *tp_last_error(void);

/* Library version as "major.minor.patch". */
const char *tp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TP_B300_H */
