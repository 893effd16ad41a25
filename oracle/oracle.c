/*
 * CPU oracle for Conv2d backward-data (dgrad).  TEST INFRASTRUCTURE ONLY.
 *
 * This file is the plain, slow, obviously correct statement of what the GPU
 * library computes.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark load it; the library itself never links, loads or calls
 * it, and it shares no code, header, table or helper with the CUDA sources.
 *
 * What it computes (the definition, written out):
 *
 *   dX[n,h,w,c] = sum over k, r, s and every (p, q) with
 *                 h = p*stride - pad + r*dil  and  w = q*stride - pad + s*dil,
 *                 0 <= p < P, 0 <= q < Q, of dY[n,p,q,k] * W[k,r,s,c]
 *
 * i.e. the gradient of a cross-correlation Conv2d with respect to its input,
 * the operation named "Conv2d dgrad" on apache/tvm PR #10110 ("[CUTLASS]
 * Conv2d dgrad", opening description).  For a fixed output pixel h and filter
 * row r there is at most one p solving h = p*stride - pad + r*dil, so the sum
 * over (p, q) is taken by solving for them; nothing is reordered beyond that.
 *
 * P and Q are the forward convolution's output extents,
 *     P = floor((H + 2*pad - dil*(R-1) - 1) / stride) + 1,
 * the usual floor convention; H and W are the sizes of dX.
 *
 * Optional ReLU-backward epilogue (the "activation fusion" for dgrad that the
 * same page says is not enabled yet, last comments): the saved activation x
 * gates each output, out = (x > 0) ? dX : +0.0.  x <= 0, -0.0 and NaN give +0.0.
 * Other activations (GELU, SiLU) multiply dX by the activation's derivative at
 * the saved input x instead (oracle_act_grad).
 *
 * Precision: every product and sum is taken in IEEE double.  fp16 and bf16
 * inputs are decoded from their bit patterns (IEEE-754 binary16; bfloat16 =
 * the upper half of a binary32) by the decoders below.
 *
 * Tensor layouts: dY is NHWC [N][P][Q][K], W is KRSC [K][R][S][C], dX and x
 * are NHWC [N][H][W][C].  All contiguous.
 *
 * Pins: the tests check this file against a materialised forward-convolution
 * matrix (brute force), the adjoint identity with the forward convolution
 * below, closed forms (1x1 GEMM, impulse response, identity filter), a
 * hand-worked case, integer-exact results and an independent library routine.
 *
 * The file also states the weight gradient (wgrad) of the same convolution,
 * the page's announced follow-up, pinned the same ways (oracle_wgrad below),
 * and the per-channel sums of the output that a fused epilogue produces
 * (oracle_channel_sums below).
 */
#define _USE_MATH_DEFINES
#include <math.h>
#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1, ORACLE_F32 = 2, ORACLE_F64 = 3 };

/* IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 * 2^-10 */
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(frac | 0x400), expo - 25); /* (1 + frac/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round a double once, to nearest with ties to even, to a 16-bit binary
 * format with `frac` fraction bits and `expo` exponent bits (IEEE-754
 * binary16: 10 and 5; bfloat16: 7 and 8): subnormals kept, values beyond the
 * largest finite one become infinities, NaN stays NaN (a quiet one).  The
 * significand is scaled to an integer at the format's spacing for the value's
 * binade (the smallest normal binade's spacing below it) and rounded with
 * nearbyint in the default rounding mode, which rounds ties to even.
 */
static uint16_t encode_16(double x, int frac, int expo)
{
    const int bias = (1 << (expo - 1)) - 1, emin = 1 - bias, emax = bias;
    const uint16_t sign = signbit(x) ? (uint16_t)0x8000u : (uint16_t)0;
    const uint16_t inf = (uint16_t)(((1u << expo) - 1u) << frac);
    if (isnan(x)) return (uint16_t)(sign | inf | (1u << (frac - 1)));
    const double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | inf);
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);           /* a = m * 2^e2, 0.5 <= m < 1 */
    int E = e2 - 1;          /* a = (1.f...) * 2^E */
    if (E < emin) E = emin;  /* subnormals share the smallest normal binade's spacing */
    double r = nearbyint(ldexp(a, frac - E));
    if (r >= ldexp(1.0, frac + 1)) { /* rounded up into the next binade */
        r = ldexp(r, -1);
        E += 1;
    }
    if (E > emax) return (uint16_t)(sign | inf);
    const unsigned sig = (unsigned)r;
    if (sig < (1u << frac)) return (uint16_t)(sign | sig); /* subnormal (E == emin) */
    return (uint16_t)(sign | ((unsigned)(E + bias) << frac) | (sig - (1u << frac)));
}

uint16_t oracle_double_to_half(double x) { return encode_16(x, 10, 5); }
uint16_t oracle_double_to_bf16(double x) { return encode_16(x, 7, 8); }

/* Forward output extent along one axis; -1 when the geometry is empty. */
int oracle_out_extent(int in, int filt, int stride, int pad, int dil)
{
    if (in <= 0 || filt <= 0 || stride <= 0 || dil <= 0 || pad < 0) return -1;
    int span = in + 2 * pad - dil * (filt - 1) - 1;
    if (span < 0) return -1;
    return span / stride + 1;
}

/* Decode a whole buffer of the given element type into doubles. */
static double *decode_all(const void *src, size_t n, int dtype)
{
    double *out = (double *)malloc(n ? n * sizeof(double) : sizeof(double));
    if (!out) return NULL;
    if (dtype == ORACLE_F64) {
        memcpy(out, src, n * sizeof(double));
    } else if (dtype == ORACLE_F32) {
        const float *s = (const float *)src;
        for (size_t i = 0; i < n; ++i) out[i] = s[i];
    } else if (dtype == ORACLE_BF16) {
        const uint16_t *s = (const uint16_t *)src;
        for (size_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_double(s[i]);
    } else {
        const uint16_t *s = (const uint16_t *)src;
        for (size_t i = 0; i < n; ++i) out[i] = oracle_half_to_double(s[i]);
    }
    return out;
}

/* One element of a buffer of the given type, as a double. */
static double load_one(const void *src, size_t i, int dtype)
{
    switch (dtype) {
    case ORACLE_F64: return ((const double *)src)[i];
    case ORACLE_F32: return (double)((const float *)src)[i];
    case ORACLE_BF16: return oracle_bf16_to_double(((const uint16_t *)src)[i]);
    default: return oracle_half_to_double(((const uint16_t *)src)[i]);
    }
}

static int floor_mod(int a, int m)
{
    int r = a % m;
    return r < 0 ? r + m : r;
}

/*
 * The sum for one dX pixel (n, h, w), all C channels, into acc[0..C).
 * Wd is W decoded to double.  For each filter tap (r, s) the unique (p, q)
 * with h = p*stride - pad + r*dil (and likewise for w) is found; taps with no
 * integer or in-range solution contribute nothing.
 */
static void pixel_sum(const void *dY, int dtype, const double *Wd, double *acc,
                      int n, int h, int w, int C, int K, int R, int S,
                      int stride, int pad, int dil, int P, int Q)
{
    for (int c = 0; c < C; ++c) acc[c] = 0.0;
    for (int r = 0; r < R; ++r) {
        int th = h + pad - r * dil; /* = p * stride */
        if (floor_mod(th, stride) != 0) continue;
        int p = th / stride; /* exact */
        if (p < 0 || p >= P) continue;
        for (int s = 0; s < S; ++s) {
            int tw = w + pad - s * dil; /* = q * stride */
            if (floor_mod(tw, stride) != 0) continue;
            int q = tw / stride;
            if (q < 0 || q >= Q) continue;
            size_t dy_base = (((size_t)n * P + p) * Q + q) * (size_t)K;
            for (int k = 0; k < K; ++k) {
                double dy = load_one(dY, dy_base + k, dtype);
                const double *wrow = Wd + (((size_t)k * R + r) * S + s) * (size_t)C;
                for (int c = 0; c < C; ++c) acc[c] += dy * wrow[c];
            }
        }
    }
}

/*
 * Derivative of an activation function at x, for the activation-backward
 * epilogues (the activation fusion of the tvm page's last comments, with
 * activations other than ReLU):
 *   act 1, GELU in its erf form:  f(x) = x * Phi(x),  Phi(x) = (1 + erf(x / sqrt 2)) / 2,
 *                                 f'(x) = Phi(x) + x * phi(x),  phi(x) = exp(-x^2 / 2) / sqrt(2 pi)
 *   act 2, SiLU:                  f(x) = x * s(x),  s(x) = 1 / (1 + exp(-x)),
 *                                 f'(x) = s(x) * (1 + x * (1 - s(x)))
 * (act 0, ReLU, is the select in apply_gate, not a product.)
 */
double oracle_act_grad(double x, int act)
{
    if (act == 1) {
        const double Phi = 0.5 * (1.0 + erf(x / sqrt(2.0)));
        const double phi = exp(-0.5 * x * x) / sqrt(2.0 * M_PI);
        return Phi + x * phi;
    }
    const double sg = 1.0 / (1.0 + exp(-x));
    return sg * (1.0 + x * (1.0 - sg));
}

/* Backward of the activation whose input was x: act 0 (ReLU) keeps the value
 * where x > 0 (NaN, -0.0 and negatives give +0.0: a select); act 1 and 2
 * multiply it by f'(x) (oracle_act_grad). */
static void apply_gate(double *acc, const void *x, int dtype, size_t base, int C, int act)
{
    for (int c = 0; c < C; ++c) {
        double xv = load_one(x, base + c, dtype);
        if (act == 0) {
            if (!(xv > 0.0)) acc[c] = 0.0;
        } else {
            acc[c] *= oracle_act_grad(xv, act);
        }
    }
}

static int check_geometry(int N, int H, int W, int C, int K, int R, int S,
                          int stride, int pad, int dil, int *P, int *Q)
{
    if (N <= 0 || C <= 0 || K <= 0) return -1;
    *P = oracle_out_extent(H, R, stride, pad, dil);
    *Q = oracle_out_extent(W, S, stride, pad, dil);
    if (*P <= 0 || *Q <= 0) return -1;
    return 0;
}

/*
 * Full dgrad.  dY, W and x (x may be NULL: no gate) are of element type
 * `dtype`; dX is written as doubles, NHWC.  Returns 0, or -1 on bad geometry
 * or allocation failure.  OpenMP-parallel over (n, h).
 */
int oracle_dgrad_act(const void *dY, const void *Wt, const void *x, int act, int dtype, double *dX,
                     int N, int H, int W, int C, int K, int R, int S,
                     int stride, int pad, int dil)
{
    int P, Q;
    if (check_geometry(N, H, W, C, K, R, S, stride, pad, dil, &P, &Q)) return -1;
    double *Wd = decode_all(Wt, (size_t)K * R * S * C, dtype);
    if (!Wd) return -1;
    int failed = 0;
#pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)C * sizeof(double));
        if (!acc) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for collapse(2) schedule(dynamic, 1)
            for (int n = 0; n < N; ++n)
                for (int h = 0; h < H; ++h)
                    for (int w = 0; w < W; ++w) {
                        pixel_sum(dY, dtype, Wd, acc, n, h, w, C, K, R, S, stride, pad, dil, P, Q);
                        size_t base = (((size_t)n * H + h) * W + w) * (size_t)C;
                        if (x) apply_gate(acc, x, dtype, base, C, act);
                        memcpy(dX + base, acc, (size_t)C * sizeof(double));
                    }
            free(acc);
        }
    }
    free(Wd);
    return failed ? -1 : 0;
}

/*
 * dgrad at selected pixels only: pix holds npix triples (n, h, w); out gets
 * npix rows of C doubles.  Same arithmetic as oracle_dgrad, for checking
 * sampled outputs of problems too large to evaluate in full.
 */
int oracle_dgrad_pixels_act(const void *dY, const void *Wt, const void *x, int act, int dtype,
                            const int32_t *pix, int64_t npix, double *out,
                            int N, int H, int W, int C, int K, int R, int S,
                            int stride, int pad, int dil)
{
    int P, Q;
    if (check_geometry(N, H, W, C, K, R, S, stride, pad, dil, &P, &Q)) return -1;
    for (int64_t i = 0; i < npix; ++i) {
        const int32_t *t = pix + 3 * i;
        if (t[0] < 0 || t[0] >= N || t[1] < 0 || t[1] >= H || t[2] < 0 || t[2] >= W) return -1;
    }
    double *Wd = decode_all(Wt, (size_t)K * R * S * C, dtype);
    if (!Wd) return -1;
    int failed = 0;
#pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)C * sizeof(double));
        if (!acc) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t i = 0; i < npix; ++i) {
                int n = pix[3 * i], h = pix[3 * i + 1], w = pix[3 * i + 2];
                pixel_sum(dY, dtype, Wd, acc, n, h, w, C, K, R, S, stride, pad, dil, P, Q);
                if (x) apply_gate(acc, x, dtype, (((size_t)n * H + h) * W + w) * (size_t)C, C, act);
                memcpy(out + (size_t)i * C, acc, (size_t)C * sizeof(double));
            }
            free(acc);
        }
    }
    free(Wd);
    return failed ? -1 : 0;
}

/* The ReLU-backward forms (x may be NULL: no gate). */
int oracle_dgrad(const void *dY, const void *Wt, const void *x, int dtype, double *dX,
                 int N, int H, int W, int C, int K, int R, int S,
                 int stride, int pad, int dil)
{
    return oracle_dgrad_act(dY, Wt, x, 0, dtype, dX, N, H, W, C, K, R, S, stride, pad, dil);
}

int oracle_dgrad_pixels(const void *dY, const void *Wt, const void *x, int dtype,
                        const int32_t *pix, int64_t npix, double *out,
                        int N, int H, int W, int C, int K, int R, int S,
                        int stride, int pad, int dil)
{
    return oracle_dgrad_pixels_act(dY, Wt, x, 0, dtype, pix, npix, out, N, H, W, C, K, R, S, stride, pad, dil);
}

/*
 * Forward cross-correlation, the operation whose input gradient dgrad is:
 *   y[n,p,q,k] = sum_{r,s,c} x[n, p*stride - pad + r*dil, q*stride - pad + s*dil, c] * W[k,r,s,c]
 * with out-of-range input positions reading zero.  x is NHWC of `dtype`,
 * y is written as doubles, NHWC [N][P][Q][K].  Used by the adjoint-identity pin.
 */
int oracle_conv_fwd(const void *x, const void *Wt, int dtype, double *y,
                    int N, int H, int W, int C, int K, int R, int S,
                    int stride, int pad, int dil)
{
    int P, Q;
    if (check_geometry(N, H, W, C, K, R, S, stride, pad, dil, &P, &Q)) return -1;
    double *Wd = decode_all(Wt, (size_t)K * R * S * C, dtype);
    if (!Wd) return -1;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int n = 0; n < N; ++n)
        for (int p = 0; p < P; ++p)
            for (int q = 0; q < Q; ++q)
                for (int k = 0; k < K; ++k) {
                    double acc = 0.0;
                    for (int r = 0; r < R; ++r) {
                        int h = p * stride - pad + r * dil;
                        if (h < 0 || h >= H) continue;
                        for (int s = 0; s < S; ++s) {
                            int w = q * stride - pad + s * dil;
                            if (w < 0 || w >= W) continue;
                            size_t xb = (((size_t)n * H + h) * W + w) * (size_t)C;
                            const double *wrow = Wd + (((size_t)k * R + r) * S + s) * (size_t)C;
                            for (int c = 0; c < C; ++c) acc += load_one(x, xb + c, dtype) * wrow[c];
                        }
                    }
                    y[(((size_t)n * P + p) * Q + q) * (size_t)K + k] = acc;
                }
    free(Wd);
    return 0;
}

/*
 * Weight gradient (wgrad) of the same cross-correlation: the gradient of y
 * above with respect to the filter, which the apache/tvm PR #10110 page
 * ("[CUTLASS] Conv2d dgrad") names as the follow-up to dgrad (opening
 * description; merge comment: "wgrad + parallel split-k").  The page gives
 * no formula; this is the definition written out:
 *   dW[k,r,s,c] = sum over n, p, q of
 *                 dY[n,p,q,k] * x[n, p*stride - pad + r*dil, q*stride - pad + s*dil, c]
 * with out-of-range input positions contributing zero (the padding the
 * forward pass read as zero).  dY is NHWC [N][P][Q][K], x NHWC [N][H][W][C],
 * both of `dtype`; dW is written as doubles, KRSC [K][R][S][C].  Each filter
 * element's sum runs over (n, p, q) in that order; nothing else is reordered.
 */
int oracle_wgrad(const void *dY, const void *x, int dtype, double *dW,
                 int N, int H, int W, int C, int K, int R, int S,
                 int stride, int pad, int dil)
{
    int P, Q;
    if (check_geometry(N, H, W, C, K, R, S, stride, pad, dil, &P, &Q)) return -1;
    double *g = decode_all(dY, (size_t)N * P * Q * K, dtype);
    double *xd = decode_all(x, (size_t)N * H * W * C, dtype);
    if (!g || !xd) {
        free(g);
        free(xd);
        return -1;
    }
#pragma omp parallel for collapse(3) schedule(dynamic, 1)
    for (int k = 0; k < K; ++k)
        for (int r = 0; r < R; ++r)
            for (int s = 0; s < S; ++s) {
                double *out = dW + (((size_t)k * R + r) * S + s) * (size_t)C;
                for (int c = 0; c < C; ++c) out[c] = 0.0;
                for (int n = 0; n < N; ++n)
                    for (int p = 0; p < P; ++p) {
                        int h = p * stride - pad + r * dil;
                        if (h < 0 || h >= H) continue;
                        for (int q = 0; q < Q; ++q) {
                            int w = q * stride - pad + s * dil;
                            if (w < 0 || w >= W) continue;
                            const double gv = g[(((size_t)n * P + p) * Q + q) * (size_t)K + k];
                            const double *xrow = xd + (((size_t)n * H + h) * W + w) * (size_t)C;
                            for (int c = 0; c < C; ++c) out[c] += gv * xrow[c];
                        }
                    }
            }
    free(g);
    free(xd);
    return 0;
}

/*
 * Selected elements of the same weight gradient: idx holds nidx rows of
 * (k, r, s, c); out[i] = dW[k,r,s,c] by the definition above, each summed over
 * (n, p, q) in that order.  For spot checks of full-size problems: nothing is
 * decoded ahead, every operand is read where the sum needs it.
 */
int oracle_wgrad_elements(const void *dY, const void *x, int dtype, const int32_t *idx, int64_t nidx,
                          double *out, int N, int H, int W, int C, int K, int R, int S,
                          int stride, int pad, int dil)
{
    int P, Q;
    if (check_geometry(N, H, W, C, K, R, S, stride, pad, dil, &P, &Q)) return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nidx; ++i) {
        const int k = idx[4 * i], r = idx[4 * i + 1], s = idx[4 * i + 2], c = idx[4 * i + 3];
        double acc = 0.0;
        if (k >= 0 && k < K && r >= 0 && r < R && s >= 0 && s < S && c >= 0 && c < C) {
            for (int n = 0; n < N; ++n)
                for (int p = 0; p < P; ++p) {
                    const int h = p * stride - pad + r * dil;
                    if (h < 0 || h >= H) continue;
                    for (int q = 0; q < Q; ++q) {
                        const int w = q * stride - pad + s * dil;
                        if (w < 0 || w >= W) continue;
                        acc += load_one(dY, (((size_t)n * P + p) * Q + q) * (size_t)K + k, dtype) *
                               load_one(x, (((size_t)n * H + h) * W + w) * (size_t)C + c, dtype);
                    }
                }
        }
        out[i] = acc;
    }
    return 0;
}

/*
 * Per-channel sums of the dgrad output, the reductions a fused epilogue hands
 * to the layer below (the epilogue fusion of the Bolt reading notes: work
 * that would otherwise re-read the output is done where the output is made):
 *
 *   s1[c] = sum over n, h, w of out[n,h,w,c]
 *   s2[c] = sum over n, h, w with x[n,h,w,c] > 0 of out[n,h,w,c] * x[n,h,w,c]
 *
 * out is the (gated) dX as this oracle computes it, in double, NHWC with
 * `pixels` = N*H*W rows of C channels; x is the saved activation the gate
 * reads (element type `dtype`; NULL: s2 is not computed).  s1 is the bias
 * gradient of a bias added before the ReLU and BatchNorm's beta gradient;
 * with x the BatchNorm output y (or relu(y)), s2 = sum out*y, from which
 * BatchNorm's gamma gradient is (s2 - beta*s1)/gamma.  Positions the gate
 * masks contribute nothing to s2, whatever x holds there (NaN included).
 * a1[c] and a2[c] receive the sums of the absolute values of the same terms
 * (the scale against which rounding errors of a reordered sum are bounded).
 * Each channel's sums run over the pixels in order.
 */
int oracle_channel_sums(const double *out, const void *x, int dtype, int64_t pixels, int C,
                        double *s1, double *s2, double *a1, double *a2)
{
    if (pixels < 0 || C <= 0) return -1;
    for (int c = 0; c < C; ++c) {
        s1[c] = 0.0;
        a1[c] = 0.0;
        if (x) {
            s2[c] = 0.0;
            a2[c] = 0.0;
        }
    }
    for (int64_t i = 0; i < pixels; ++i) {
        const double *row = out + (size_t)i * (size_t)C;
        for (int c = 0; c < C; ++c) {
            s1[c] += row[c];
            a1[c] += fabs(row[c]);
            if (x) {
                double xv = load_one(x, (size_t)i * (size_t)C + c, dtype);
                if (xv > 0.0) {
                    s2[c] += row[c] * xv;
                    a2[c] += fabs(row[c] * xv);
                }
            }
        }
    }
    return 0;
}

/* Threads an OpenMP region of this library would use. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
