/*
 * tp_oracle.c -- float64 CPU oracle for Fourier-space projection and
 * backprojection on RFFT half-spectra.
 *
 * TEST INFRASTRUCTURE ONLY.  This file exists to check the CUDA library
 * against a plain, slow, obviously correct restatement of the method.  It
 * shares no source, header, table or helper with the CUDA path, and the
 * product path never calls it.  Only the test-suite, the smoke check and the
 * CPU-baseline leg of the benchmark load it.
 *
 * Method source: the summary pages of "torch-projectors: A High-Performance
 * Differentiable Projection Library for PyTorch" (D. Tegunov, 2026).  They
 * are cited by language and by the section of their technical summary:
 *   [it §2]  Italian page, "Sommario tecnico", 2. Metodologia e Architettura
 *   [de §2]  German page, "Technische Zusammenfassung", 2. Methodik und Architektur
 *   [ja §2]  Japanese page, "技術概要", 2. 手法とアーキテクチャ
 *   [ko §2]  Korean page, "기술 요약", 2. 방법론
 *   [ar §2]  Arabic page, technical summary, 2. المنهجية
 * The pages state the method in words only; where they leave a step open the
 * plainest reading is taken and marked READING below.
 *
 * Conventions (shared by every function here):
 *  - Half-spectrum layout [it §2 "Spazio di Fourier e Formati"; ar §2]:
 *    a 3D spectrum of box M is stored as (M, M, M/2+1) indexed [z][y][x], a
 *    2D spectrum as (M, M/2+1) indexed [y][x], exactly as rfftn returns it.
 *    Row index i of a box-M axis holds frequency i for i < M/2, else i - M.
 *  - Complex values are interleaved (re, im) doubles.
 *  - Output pixel (iy, ix) of a box-N image has frequency k = (ix, f(iy)).
 *  - READING: pixels with kx^2 + ky^2 > r^2 are zero and scatter nothing.
 *  - Rotation by the inverse matrix [ko §2 "Forward Projection"; ar §2
 *    "الإزاحات والدورات"]: the sample position is p = s * R^T k, i.e.
 *    p_j = s * sum_i R[i][j] k_i, with k_z = 0 for the 3D->2D case.
 *  - Interpolation [it §2 "Interpolazione"; ko §2 "보간법"]: per axis, linear
 *    taps floor(p), floor(p)+1 with w(t) = 1 - |t|, or Catmull-Rom (Keys cubic
 *    convolution, a = -1/2) taps floor(p)-1 .. floor(p)+2; t = p - tap; the
 *    weight of a tap is the product over axes.
 *  - Friedel reads [ar §2 "التمرير الأمامي"; ko §2 "Friedel 대칭성 처리"]:
 *    a tap n with n_x < 0 reads conj(V[-n]).  READING: the reflection is
 *    applied per tap.  After it, a tap outside the stored range
 *    (0 <= n_x <= M/2, -M/2 <= n_y, n_z <= M/2 - 1) reads zero.
 *  - Shift as a phase ramp [de §2 "Interpolation"; ar §2]:
 *    out = exp(-2 pi i (kx sx + ky sy) / N) * (interpolated value).
 *  - Adjoint [ko §2 "Backward Projection"]: the exact real adjoint of the
 *    forward map, i.e. a direct tap adds w * conj(phase) * y to V[n] and a
 *    Friedel tap adds conj of that to V[-n].  The weight spectrum [it §2
 *    "accumulo di pesi"; de §2 "Dual-Volumen-Ansatz"] adds w * omega to the
 *    same location.
 *  - Gradients w.r.t. rotation matrices and shifts [de §3 item 4; ko §2
 *    "그라디언트 계산"; ar §2]: chain rule through the analytic derivative
 *    of the interpolation kernel.
 *  - Batch broadcast [de §3 item 3]: B = max(Bv, Bp, Bs) and each of them
 *    is 1 or B.  Gradients of a broadcast operand sum over the batch.
 *
 * Every accumulating output (+=) must be zeroed by the caller.
 */
#include <math.h>
#include <stddef.h>
#include <string.h>

#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif

typedef struct {
    double re, im;
} cplx;

/* ---- interpolation kernels ------------------------------------------- */

/* Keys (1981) cubic convolution kernel with a = -1/2 (Catmull-Rom). */
static double keys_w(double t)
{
    const double a = -0.5;
    double u = fabs(t);
    if (u <= 1.0)
        return (a + 2.0) * u * u * u - (a + 3.0) * u * u + 1.0;
    if (u < 2.0)
        return a * u * u * u - 5.0 * a * u * u + 8.0 * a * u - 4.0 * a;
    return 0.0;
}

/* d/dt of keys_w. */
static double keys_dw(double t)
{
    const double a = -0.5;
    double u = fabs(t);
    double sg = (t < 0.0) ? -1.0 : 1.0;
    if (u <= 1.0)
        return sg * (3.0 * (a + 2.0) * u * u - 2.0 * (a + 3.0) * u);
    if (u < 2.0)
        return sg * (3.0 * a * u * u - 10.0 * a * u + 8.0 * a);
    return 0.0;
}

/*
 * One axis of the stencil at position p: tap indices, weights and their
 * derivatives with respect to p.  Returns the number of taps (2 or 4).
 * READING: the linear derivative is the one of the branch on [x0, x0+1),
 * i.e. -1 for tap x0 and +1 for tap x0+1, also when p is an integer.
 */
static int stencil_axis(double p, int cubic, int *tap, double *w, double *dw)
{
    int x0 = (int)floor(p);
    if (cubic) {
        for (int j = 0; j < 4; ++j) {
            tap[j] = x0 - 1 + j;
            w[j] = keys_w(p - (double)tap[j]);
            dw[j] = keys_dw(p - (double)tap[j]);
        }
        return 4;
    }
    tap[0] = x0;
    tap[1] = x0 + 1;
    w[0] = 1.0 - (p - (double)x0);
    w[1] = 1.0 - ((double)x0 + 1.0 - p);
    dw[0] = -1.0;
    dw[1] = 1.0;
    return 2;
}

/* ---- spectrum access -------------------------------------------------- */

typedef struct {
    int dim;   /* 2 or 3 */
    int M;     /* box size */
} spec_shape;

static size_t spec_elems(spec_shape s)
{
    size_t X = (size_t)s.M / 2 + 1;
    return (s.dim == 3) ? (size_t)s.M * s.M * X : (size_t)s.M * X;
}

/* Frequency (y or z) -> stored row, or -1 when outside -M/2 .. M/2-1. */
static int row_of(int f, int M)
{
    if (f < -M / 2 || f > M / 2 - 1)
        return -1;
    return (f < 0) ? f + M : f;
}

/*
 * Resolve a tap n (n[0]=x, n[1]=y, n[2]=z) to a stored element.  Sets
 * *conj to 1 when the tap was Friedel-reflected.  Returns the flat element
 * index, or -1 when the tap lies outside the stored range.
 */
static long resolve_tap(spec_shape s, const int *n, int *conj)
{
    int m[3] = {n[0], n[1], s.dim == 3 ? n[2] : 0};
    *conj = 0;
    if (m[0] < 0) {
        m[0] = -m[0];
        m[1] = -m[1];
        m[2] = -m[2];
        *conj = 1;
    }
    int X = s.M / 2 + 1;
    if (m[0] > s.M / 2)
        return -1;
    int ry = row_of(m[1], s.M);
    if (ry < 0)
        return -1;
    if (s.dim == 2)
        return (long)ry * X + m[0];
    int rz = row_of(m[2], s.M);
    if (rz < 0)
        return -1;
    return ((long)rz * s.M + ry) * X + m[0];
}

/* ---- per-sample geometry ---------------------------------------------- */

static int freq_of_row(int iy, int N)
{
    return (iy < N / 2) ? iy : iy - N;
}

/* p_j = s * sum_i R[i][j] k_i, R row-major dim x dim, k = (kx, ky[, 0]). */
static void sample_position(const double *R, int dim, double s, double kx,
                            double ky, double *p)
{
    for (int j = 0; j < dim; ++j)
        p[j] = s * (R[0 * dim + j] * kx + R[1 * dim + j] * ky);
}

/* exp(-2 pi i (kx sx + ky sy) / N); identity when shift is NULL. */
static cplx phase_of(const double *t, double kx, double ky, int N)
{
    cplx ph = {1.0, 0.0};
    if (t) {
        double ang = -2.0 * M_PI * (kx * t[0] + ky * t[1]) / (double)N;
        ph.re = cos(ang);
        ph.im = sin(ang);
    }
    return ph;
}

static cplx cmul(cplx a, cplx b)
{
    cplx r = {a.re * b.re - a.im * b.im, a.re * b.im + a.im * b.re};
    return r;
}

static cplx cconj(cplx a)
{
    cplx r = {a.re, -a.im};
    return r;
}

/*
 * Interpolated value S = sum_n w_n v_n at p, and (when dS != NULL) its
 * derivatives dS[a] = sum_n (d w_n / d p_a) v_n.  Friedel-reflected taps
 * take the conjugate value; their derivative still comes from w only.
 */
static cplx interpolate(const double *V, spec_shape s, const double *p,
                        int cubic, cplx *dS)
{
    int tap[3][4];
    double w[3][4], dw[3][4];
    int cnt = 0;
    for (int a = 0; a < s.dim; ++a)
        cnt = stencil_axis(p[a], cubic, tap[a], w[a], dw[a]);
    int cz = (s.dim == 3) ? cnt : 1;
    cplx S = {0.0, 0.0};
    if (dS)
        for (int a = 0; a < s.dim; ++a)
            dS[a].re = dS[a].im = 0.0;
    for (int jz = 0; jz < cz; ++jz)
        for (int jy = 0; jy < cnt; ++jy)
            for (int jx = 0; jx < cnt; ++jx) {
                int n[3] = {tap[0][jx], tap[1][jy], s.dim == 3 ? tap[2][jz] : 0};
                int cj;
                long e = resolve_tap(s, n, &cj);
                if (e < 0)
                    continue;
                cplx v = {V[2 * e], V[2 * e + 1]};
                if (cj)
                    v = cconj(v);
                double wz = (s.dim == 3) ? w[2][jz] : 1.0;
                double wt = w[0][jx] * w[1][jy] * wz;
                S.re += wt * v.re;
                S.im += wt * v.im;
                if (dS) {
                    double g[3];
                    g[0] = dw[0][jx] * w[1][jy] * wz;
                    g[1] = w[0][jx] * dw[1][jy] * wz;
                    g[2] = (s.dim == 3) ? w[0][jx] * w[1][jy] * dw[2][jz] : 0.0;
                    for (int a = 0; a < s.dim; ++a) {
                        dS[a].re += g[a] * v.re;
                        dS[a].im += g[a] * v.im;
                    }
                }
            }
    return S;
}

/*
 * Adjoint of interpolate(): spread c over the stencil at p.  A direct tap
 * adds w*c to V[n], a Friedel tap adds w*conj(c) to V[-n].  When W is not
 * NULL it also adds w*omega to the same (unconjugated, real) location.
 */
static void spread(double *V, double *W, spec_shape s, const double *p,
                   int cubic, cplx c, double omega)
{
    int tap[3][4];
    double w[3][4], dw[3][4];
    int cnt = 0;
    for (int a = 0; a < s.dim; ++a)
        cnt = stencil_axis(p[a], cubic, tap[a], w[a], dw[a]);
    int cz = (s.dim == 3) ? cnt : 1;
    for (int jz = 0; jz < cz; ++jz)
        for (int jy = 0; jy < cnt; ++jy)
            for (int jx = 0; jx < cnt; ++jx) {
                int n[3] = {tap[0][jx], tap[1][jy], s.dim == 3 ? tap[2][jz] : 0};
                int cj;
                long e = resolve_tap(s, n, &cj);
                if (e < 0)
                    continue;
                double wz = (s.dim == 3) ? w[2][jz] : 1.0;
                double wt = w[0][jx] * w[1][jy] * wz;
                double re = wt * c.re;
                double im = wt * (cj ? -c.im : c.im);
                if (V) {
#pragma omp atomic
                    V[2 * e] += re;
#pragma omp atomic
                    V[2 * e + 1] += im;
                }
                if (W) {
#pragma omp atomic
                    W[e] += wt * omega;
                }
            }
}

static int bcast_ok(int b, int B)
{
    return b == 1 || b == B;
}

static int imax3(int a, int b, int c)
{
    int m = a > b ? a : b;
    return m > c ? m : c;
}

/* ---- the operators ---------------------------------------------------- */

/*
 * Forward projection (3D->2D central slice when dim == 3, 2D->2D rotation
 * and shift when dim == 2) [it §2 "Operazioni Supportate"; de §2
 * "Unterstützte Operationen"; ja §2 "演算の種類"].
 *   src   (Bsrc, M, M[, M], M/2+1) complex
 *   rot   (Bp, P, dim, dim);  shift (Bs, P, 2) or NULL
 *   out   (B, P, N, N/2+1) complex, overwritten
 * Returns 0, or -1 on a bad shape.
 */
int oracle_project(int dim, const double *src, int Bsrc, int M,
                   const double *rot, int Bp, int P, const double *shift,
                   int Bs, int N, int cubic, double s, double radius,
                   double *out)
{
    int B = imax3(Bsrc, Bp, shift ? Bs : 1);
    if ((dim != 2 && dim != 3) || !bcast_ok(Bsrc, B) || !bcast_ok(Bp, B) ||
        (shift && !bcast_ok(Bs, B)) || N < 2 || (N & 1) || M < 2 || (M & 1))
        return -1;
    spec_shape sh = {dim, M};
    size_t selems = spec_elems(sh);
    int X = N / 2 + 1;
    double r = (radius < 0.0) ? 0.5 * N : radius;
#pragma omp parallel for collapse(2) schedule(static)
    for (int bp = 0; bp < B * P; ++bp)
        for (int iy = 0; iy < N; ++iy) {
            int b = bp / P, pi = bp % P;
            const double *V = src + 2 * selems * (size_t)(Bsrc == 1 ? 0 : b);
            const double *R = rot + (size_t)((Bp == 1 ? 0 : b) * P + pi) * dim * dim;
            const double *t = shift ? shift + (size_t)((Bs == 1 ? 0 : b) * P + pi) * 2 : NULL;
            double *o = out + 2 * ((size_t)bp * N + iy) * X;
            double ky = freq_of_row(iy, N);
            for (int ix = 0; ix < X; ++ix) {
                double kx = ix;
                o[2 * ix] = o[2 * ix + 1] = 0.0;
                if (kx * kx + ky * ky > r * r)
                    continue;
                double p[3];
                sample_position(R, dim, s, kx, ky, p);
                cplx S = interpolate(V, sh, p, cubic, NULL);
                cplx y = cmul(phase_of(t, kx, ky, N), S);
                o[2 * ix] = y.re;
                o[2 * ix + 1] = y.im;
            }
        }
    return 0;
}

/*
 * Backprojection: the adjoint of oracle_project() applied to img, plus the
 * weight spectrum [de §2 "Dual-Volumen-Ansatz"; ar §3 "وزن الحجم المزدوج"].
 *   img     (B, P, N, N/2+1) complex;  omega (B, P, N, N/2+1) real or NULL (= 1)
 *   dst     (Bdst, M, M[, M], M/2+1) complex, accumulated (+=), Bdst in {1, B}
 *   wdst    same shape, real, accumulated, or NULL
 */
int oracle_backproject(int dim, const double *img, const double *omega, int B,
                       int P, int N, const double *rot, int Bp,
                       const double *shift, int Bs, int Bdst, int M, int cubic,
                       double s, double radius, double *dst, double *wdst)
{
    if ((dim != 2 && dim != 3) || !bcast_ok(Bdst, B) || !bcast_ok(Bp, B) ||
        (shift && !bcast_ok(Bs, B)) || N < 2 || (N & 1) || M < 2 || (M & 1))
        return -1;
    spec_shape sh = {dim, M};
    size_t selems = spec_elems(sh);
    int X = N / 2 + 1;
    double r = (radius < 0.0) ? 0.5 * N : radius;
#pragma omp parallel for collapse(2) schedule(dynamic, 4)
    for (int bp = 0; bp < B * P; ++bp)
        for (int iy = 0; iy < N; ++iy) {
            int b = bp / P, pi = bp % P;
            size_t boff = selems * (size_t)(Bdst == 1 ? 0 : b);
            double *V = dst ? dst + 2 * boff : NULL;
            double *W = wdst ? wdst + boff : NULL;
            const double *R = rot + (size_t)((Bp == 1 ? 0 : b) * P + pi) * dim * dim;
            const double *t = shift ? shift + (size_t)((Bs == 1 ? 0 : b) * P + pi) * 2 : NULL;
            const double *y = img + 2 * ((size_t)bp * N + iy) * X;
            const double *om = omega ? omega + ((size_t)bp * N + iy) * X : NULL;
            double ky = freq_of_row(iy, N);
            for (int ix = 0; ix < X; ++ix) {
                double kx = ix;
                if (kx * kx + ky * ky > r * r)
                    continue;
                double p[3];
                sample_position(R, dim, s, kx, ky, p);
                cplx yk = {y[2 * ix], y[2 * ix + 1]};
                cplx c = cmul(cconj(phase_of(t, kx, ky, N)), yk);
                spread(V, W, sh, p, cubic, c, om ? om[ix] : 1.0);
            }
        }
    return 0;
}

/*
 * Gradients of a real loss L through oracle_project(), given
 * g = dL/dRe(out) + i dL/dIm(out) (PyTorch's convention for complex
 * tensors).  Any output may be NULL; all are accumulated (+=).
 *   gsrc   (Bsrc, ...) complex: the adjoint applied to g
 *   grot   (Bp, P, dim, dim): dL/dR[i][j] = sum s k_i dL/dp_j
 *   gshift (Bs, P, 2):       dL/dt_a = sum Re(conj(g) (-2 pi i k_a / N) out)
 * with dL/dp_a = Re(conj(g) phase sum_n (d w_n / d p_a) v_n).
 */
int oracle_project_backward(int dim, const double *grad_out, const double *src,
                            int Bsrc, int M, const double *rot, int Bp, int P,
                            const double *shift, int Bs, int N, int cubic,
                            double s, double radius, double *gsrc,
                            double *grot, double *gshift)
{
    int B = imax3(Bsrc, Bp, shift ? Bs : 1);
    if ((dim != 2 && dim != 3) || !bcast_ok(Bsrc, B) || !bcast_ok(Bp, B) ||
        (shift && !bcast_ok(Bs, B)) || N < 2 || (N & 1) || M < 2 || (M & 1))
        return -1;
    if (gsrc) {
        int rc = oracle_backproject(dim, grad_out, NULL, B, P, N, rot, Bp,
                                    shift, Bs, Bsrc, M, cubic, s, radius, gsrc,
                                    NULL);
        if (rc)
            return rc;
    }
    if (!grot && !gshift)
        return 0;
    spec_shape sh = {dim, M};
    size_t selems = spec_elems(sh);
    int X = N / 2 + 1;
    double r = (radius < 0.0) ? 0.5 * N : radius;
#pragma omp parallel for schedule(dynamic, 1)
    for (int bp = 0; bp < B * P; ++bp) {
        int b = bp / P, pi = bp % P;
        const double *V = src + 2 * selems * (size_t)(Bsrc == 1 ? 0 : b);
        size_t ridx = (size_t)((Bp == 1 ? 0 : b) * P + pi);
        size_t sidx = (size_t)((Bs == 1 ? 0 : b) * P + pi);
        const double *R = rot + ridx * dim * dim;
        const double *t = shift ? shift + sidx * 2 : NULL;
        double gR[9] = {0}, gt[2] = {0, 0};
        for (int iy = 0; iy < N; ++iy) {
            double ky = freq_of_row(iy, N);
            const double *g = grad_out + 2 * ((size_t)bp * N + iy) * X;
            for (int ix = 0; ix < X; ++ix) {
                double kx = ix;
                if (kx * kx + ky * ky > r * r)
                    continue;
                double p[3], k[2] = {kx, ky};
                sample_position(R, dim, s, kx, ky, p);
                cplx dS[3];
                cplx S = interpolate(V, sh, p, cubic, dS);
                cplx ph = phase_of(t, kx, ky, N);
                cplx gk = {g[2 * ix], g[2 * ix + 1]};
                for (int j = 0; j < dim; ++j) {
                    cplx d = cmul(cconj(gk), cmul(ph, dS[j]));
                    for (int i = 0; i < 2; ++i)
                        gR[i * dim + j] += s * k[i] * d.re;
                }
                cplx y = cmul(ph, S);
                for (int a = 0; a < 2; ++a) {
                    cplx dy = {0.0, -2.0 * M_PI * k[a] / (double)N};
                    cplx d = cmul(cconj(gk), cmul(dy, y));
                    gt[a] += d.re;
                }
            }
        }
        if (grot)
            for (int e = 0; e < dim * dim; ++e) {
#pragma omp atomic
                grot[ridx * dim * dim + e] += gR[e];
            }
        if (gshift && shift)
            for (int a = 0; a < 2; ++a) {
#pragma omp atomic
                gshift[sidx * 2 + a] += gt[a];
            }
    }
    return 0;
}

/* Threads the oracle runs on (for the CPU-baseline record). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the oracle's later calls (n >= 1; the single-thread CPU figure). */
void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    if (n >= 1)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
