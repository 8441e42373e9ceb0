/*
 * CPU oracle numerics: plain fp64 definitions of the three operations the stream-K path serves.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this library. It shares no code, header or table with the CUDA path.
 *
 * Stream-K only re-orders the fp32 summation of a GEMM, so what the path computes has a plain
 * definition, written out here with one fp64 accumulator per output element and the reduction
 * taken in its natural order (rocm-libraries PR #13151, PR body: "Stream-K balances MAC
 * iterations instead of tiles"; the same holds for the CK Tile stream-K GEMM bridge page):
 *
 *   GEMM, rcr layout (CK Tile stream-K GEMM TE to dispatcher bridge, Summary: "fp16/rcr"):
 *       C[m][n] = sum_k A[m*lda + k] * B[n*ldb + k]
 *   Convolution backward-weight as an implicit GEMM, NHWC activations, KRSC filter per group
 *   (PR #13151, PR body "Wgrad kernel"; commit "Port CK Tile's stream-K to the backward-weight
 *   convolution": the reduction runs over N*Ho*Wo and conv groups fold into GEMM-M):
 *       dW[g*Kg+k][r][s][c] = sum_{n,ho,wo} dy[n][ho][wo][g*Kg+k]
 *                                          * x[n][ho*sh-ph+r][wo*sw-pw+s][g*Cg+c]
 *       with x outside the image taken as 0 and Ho = (H+2ph-R)/sh + 1 (likewise Wo).
 *   RowColQuant fp8 GEMM (rocm-libraries PR #9979, Scope: per-row scale of A, per-column scale
 *   of B, fp32 accumulator narrowed only at the end):
 *       C[m][n] = (sum_k deq(A8[m][k]) * deq(B8[n][k])) * sa[m] * sb[n]
 *   Block-scaled fp8 GEMM (PR #10439, Summary: "aquant" scales A in blocks along K, "bquant" scales
 *   B in blocks along N and K, "abquant" both), with a missing scale read as 1:
 *       C[m][n] = sum_k sa[m][k/gka] * sb[n/gnb][k/gkb] * deq(A8[m][k]) * deq(B8[n][k])
 *   Forward convolution and data gradient (PR #13151 lists the forward convolution as future work
 *   on the same machinery; both are the plain definitions, NHWC activations, KRSC filters):
 *       y[n][ho][wo][g*Kg+k]  = sum_{r,s,c} x[n][ho*sh-ph+r][wo*sw-pw+s][g*Cg+c] * w[g*Kg+k][r][s][c]
 *       dx[n][h][w][g*Cg+c]   = sum_{r,s,k} dy[n][ho][wo][g*Kg+k] * w[g*Kg+k][r][s][c]
 *                               over the (ho, wo) with ho*sh-ph+r = h and wo*sw-pw+s = w
 *
 * Inputs are the raw 16-bit or 8-bit patterns; they are decoded here from the format
 * definitions (binary16, bfloat16, OCP E4M3). Outputs are fp64 and are rounded to the output
 * type by the Python side of the oracle.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { FMT_F16 = 0, FMT_BF16 = 1, FMT_E4M3 = 3 };

/* binary16: sign | 5-bit exponent (bias 15) | 10-bit fraction */
static double dec_f16(uint32_t b) {
    double sign = (b >> 15) & 1 ? -1.0 : 1.0;
    int e = (int)((b >> 10) & 0x1F);
    int f = (int)(b & 0x3FF);
    if (e == 0) return sign * ldexp((double)f, -24);        /* f/2^10 * 2^-14 */
    if (e == 31) return f ? NAN : sign * INFINITY;
    return sign * ldexp(1024.0 + f, e - 25);                  /* (1 + f/2^10) * 2^(e-15) */
}

/* bfloat16: sign | 8-bit exponent (bias 127) | 7-bit fraction */
static double dec_bf16(uint32_t b) {
    double sign = (b >> 15) & 1 ? -1.0 : 1.0;
    int e = (int)((b >> 7) & 0xFF);
    int f = (int)(b & 0x7F);
    if (e == 0) return sign * ldexp((double)f, -133);       /* f/2^7 * 2^-126 */
    if (e == 255) return f ? NAN : sign * INFINITY;
    return sign * ldexp(128.0 + f, e - 134);                  /* (1 + f/2^7) * 2^(e-127) */
}

/* OCP E4M3 ("fn"): sign | 4-bit exponent (bias 7) | 3-bit fraction; no inf; S.1111.111 is NaN */
static double dec_e4m3(uint32_t b) {
    double sign = (b >> 7) & 1 ? -1.0 : 1.0;
    int e = (int)((b >> 3) & 0xF);
    int f = (int)(b & 0x7);
    if (e == 15 && f == 7) return NAN;
    if (e == 0) return sign * ldexp((double)f, -9);          /* f/2^3 * 2^-6 */
    return sign * ldexp(8.0 + f, e - 10);                     /* (1 + f/2^3) * 2^(e-7) */
}

static double *make_table(int fmt) {
    int n = fmt == FMT_E4M3 ? 256 : 65536;
    double *t = (double *)malloc(sizeof(double) * (size_t)n);
    for (int i = 0; i < n; ++i)
        t[i] = fmt == FMT_F16 ? dec_f16((uint32_t)i) : fmt == FMT_BF16 ? dec_bf16((uint32_t)i)
                                                                      : dec_e4m3((uint32_t)i);
    return t;
}

static int set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Decode n patterns of format fmt to fp64 (exposed so the decoders can be pinned). */
void oracle_decode(int fmt, const void *bits, int64_t n, double *out) {
    for (int64_t i = 0; i < n; ++i) {
        uint32_t b = fmt == FMT_E4M3 ? ((const uint8_t *)bits)[i] : ((const uint16_t *)bits)[i];
        out[i] = fmt == FMT_F16 ? dec_f16(b) : fmt == FMT_BF16 ? dec_bf16(b) : dec_e4m3(b);
    }
}

int oracle_threads(int nthreads) { return set_threads(nthreads); }

/* C[m][n] = sum_k A[m][k] * B[n][k]  (rcr), for the (m, n) pairs listed. */
void oracle_gemm_rcr_points(int fmt, int64_t K, const uint16_t *A, int64_t lda, const uint16_t *B,
                            int64_t ldb, const int64_t *ms, const int64_t *ns, int64_t npts,
                            double *out, int nthreads) {
    double *tab = make_table(fmt);
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t p = 0; p < npts; ++p) {
        const uint16_t *a = A + ms[p] * lda;
        const uint16_t *b = B + ns[p] * ldb;
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += tab[a[k]] * tab[b[k]];
        out[p] = acc;
    }
    free(tab);
}

/* Full rows [m0, m1) of C (dense, row stride N). */
void oracle_gemm_rcr_rows(int fmt, int64_t m0, int64_t m1, int64_t N, int64_t K, const uint16_t *A,
                          int64_t lda, const uint16_t *B, int64_t ldb, double *out, int nthreads) {
    double *tab = make_table(fmt);
    set_threads(nthreads);
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = m0; m < m1; ++m)
        for (int64_t n = 0; n < N; ++n) {
            const uint16_t *a = A + m * lda;
            const uint16_t *b = B + n * ldb;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += tab[a[k]] * tab[b[k]];
            out[(m - m0) * N + n] = acc;
        }
    free(tab);
}

/* C[m][n] = (sum_k deq(A8[m][k]) * deq(B8[n][k])) * sa[m] * sb[n], for the listed (m, n). */
void oracle_fp8_rowcol_points(int64_t K, const uint8_t *A8, int64_t lda, const uint8_t *B8,
                              int64_t ldb, const float *sa, const float *sb, const int64_t *ms,
                              const int64_t *ns, int64_t npts, double *out, int nthreads) {
    double *tab = make_table(FMT_E4M3);
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t p = 0; p < npts; ++p) {
        const uint8_t *a = A8 + ms[p] * lda;
        const uint8_t *b = B8 + ns[p] * ldb;
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) acc += tab[a[k]] * tab[b[k]];
        out[p] = acc * (double)sa[ms[p]] * (double)sb[ns[p]];
    }
    free(tab);
}

void oracle_fp8_rowcol_rows(int64_t m0, int64_t m1, int64_t N, int64_t K, const uint8_t *A8,
                            int64_t lda, const uint8_t *B8, int64_t ldb, const float *sa,
                            const float *sb, double *out, int nthreads) {
    double *tab = make_table(FMT_E4M3);
    set_threads(nthreads);
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = m0; m < m1; ++m)
        for (int64_t n = 0; n < N; ++n) {
            const uint8_t *a = A8 + m * lda;
            const uint8_t *b = B8 + n * ldb;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += tab[a[k]] * tab[b[k]];
            out[(m - m0) * N + n] = acc * (double)sa[m] * (double)sb[n];
        }
    free(tab);
}

/*
 * Backward-weight convolution, direct loops. x: [N][H][W][C], dy: [N][Ho][Wo][K] (NHWC),
 * dw: [K][R][S][Cg] dense (Cg = C/groups), computed for filters k in [k0, k1).
 */
void oracle_wgrad_nhwc(int fmt, int64_t N, int64_t H, int64_t W, int64_t C, int64_t K, int64_t R,
                       int64_t S, int sh, int sw, int ph, int pw, int groups, const uint16_t *x,
                       const uint16_t *dy, int64_t k0, int64_t k1, double *dw, int nthreads) {
    double *tab = make_table(fmt);
    set_threads(nthreads);
    const int64_t Ho = (H + 2 * ph - R) / sh + 1;
    const int64_t Wo = (W + 2 * pw - S) / sw + 1;
    const int64_t Kg = K / groups, Cg = C / groups;
#pragma omp parallel for collapse(3) schedule(dynamic, 1)
    for (int64_t k = k0; k < k1; ++k)
        for (int64_t r = 0; r < R; ++r)
            for (int64_t s = 0; s < S; ++s) {
                const int64_t g = k / Kg;
                for (int64_t c = 0; c < Cg; ++c) {
                    double acc = 0.0;
                    for (int64_t n = 0; n < N; ++n)
                        for (int64_t ho = 0; ho < Ho; ++ho) {
                            const int64_t h = ho * sh - ph + r;
                            if (h < 0 || h >= H) continue;
                            for (int64_t wo = 0; wo < Wo; ++wo) {
                                const int64_t w = wo * sw - pw + s;
                                if (w < 0 || w >= W) continue;
                                acc += tab[dy[((n * Ho + ho) * Wo + wo) * K + k]] *
                                       tab[x[((n * H + h) * W + w) * C + g * Cg + c]];
                            }
                        }
                    dw[(((k - k0) * R + r) * S + s) * Cg + c] = acc;
                }
            }
    free(tab);
}

/*
 * Forward convolution, direct loops. x: [N][H][W][C], w: [K][R][S][Cg] (Cg = C/groups),
 * y: [N*Ho*Wo][K] for the output pixels p in [p0, p1), p = (n*Ho + ho)*Wo + wo.
 */
void oracle_fprop_nhwc(int fmt, int64_t N, int64_t H, int64_t W, int64_t C, int64_t K, int64_t R,
                       int64_t S, int sh, int sw, int ph, int pw, int groups, const uint16_t *x,
                       const uint16_t *w, int64_t p0, int64_t p1, double *y, int nthreads) {
    double *tab = make_table(fmt);
    set_threads(nthreads);
    const int64_t Ho = (H + 2 * ph - R) / sh + 1;
    const int64_t Wo = (W + 2 * pw - S) / sw + 1;
    const int64_t Kg = K / groups, Cg = C / groups;
    (void)N;
#pragma omp parallel for collapse(2) schedule(dynamic, 16)
    for (int64_t p = p0; p < p1; ++p)
        for (int64_t k = 0; k < K; ++k) {
            const int64_t n = p / (Ho * Wo), ho = (p / Wo) % Ho, wo = p % Wo;
            const int64_t g = k / Kg;
            double acc = 0.0;
            for (int64_t r = 0; r < R; ++r) {
                const int64_t h = ho * sh - ph + r;
                if (h < 0 || h >= H) continue;
                for (int64_t s = 0; s < S; ++s) {
                    const int64_t ww = wo * sw - pw + s;
                    if (ww < 0 || ww >= W) continue;
                    for (int64_t c = 0; c < Cg; ++c)
                        acc += tab[x[((n * H + h) * W + ww) * C + g * Cg + c]] *
                               tab[w[((k * R + r) * S + s) * Cg + c]];
                }
            }
            y[(p - p0) * K + k] = acc;
        }
    free(tab);
}

/*
 * Data gradient of the convolution, direct loops. dy: [N][Ho][Wo][K], w: [K][R][S][Cg],
 * dx: [N*H*W][C] for the input pixels p in [p0, p1), p = (n*H + h)*W + w. Every stride.
 */
void oracle_dgrad_nhwc(int fmt, int64_t N, int64_t H, int64_t W, int64_t C, int64_t K, int64_t R,
                       int64_t S, int sh, int sw, int ph, int pw, int groups, const uint16_t *dy,
                       const uint16_t *w, int64_t p0, int64_t p1, double *dx, int nthreads) {
    double *tab = make_table(fmt);
    set_threads(nthreads);
    const int64_t Ho = (H + 2 * ph - R) / sh + 1;
    const int64_t Wo = (W + 2 * pw - S) / sw + 1;
    const int64_t Kg = K / groups, Cg = C / groups;
    (void)N;
#pragma omp parallel for collapse(2) schedule(dynamic, 16)
    for (int64_t p = p0; p < p1; ++p)
        for (int64_t ci = 0; ci < C; ++ci) {
            const int64_t n = p / (H * W), h = (p / W) % H, ww = p % W;
            const int64_t g = ci / Cg, c = ci % Cg;
            double acc = 0.0;
            for (int64_t r = 0; r < R; ++r) {
                const int64_t th = h + ph - r;   /* = ho * sh */
                if (th < 0 || th % sh) continue;
                const int64_t ho = th / sh;
                if (ho >= Ho) continue;
                for (int64_t s = 0; s < S; ++s) {
                    const int64_t tw = ww + pw - s;
                    if (tw < 0 || tw % sw) continue;
                    const int64_t wo = tw / sw;
                    if (wo >= Wo) continue;
                    for (int64_t k = 0; k < Kg; ++k)
                        acc += tab[dy[((n * Ho + ho) * Wo + wo) * K + g * Kg + k]] *
                               tab[w[(((g * Kg + k) * R + r) * S + s) * Cg + c]];
                }
            }
            dx[(p - p0) * C + ci] = acc;
        }
    free(tab);
}

/*
 * Block-scaled fp8 GEMM for the listed (m, n): sa [M][ceil(K/gka)] or NULL, sb [ceil(N/gnb)]
 * [ceil(K/gkb)] or NULL; A8 [M][K], B8 [N][K] row-major E4M3.
 */
void oracle_fp8_blockscale_points(int64_t M, int64_t N, int64_t K, const uint8_t *A8,
                                  const uint8_t *B8, const float *sa, int64_t gka, const float *sb,
                                  int64_t gnb, int64_t gkb, const int64_t *ms, const int64_t *ns,
                                  int64_t npts, double *out, int nthreads) {
    double *tab = make_table(3);
    set_threads(nthreads);
    const int64_t nka = sa ? (K + gka - 1) / gka : 0;
    const int64_t nkb = sb ? (K + gkb - 1) / gkb : 0;
    (void)M;
    (void)N;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < npts; ++i) {
        const int64_t m = ms[i], n = ns[i];
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double s = (sa ? (double)sa[m * nka + k / gka] : 1.0) *
                             (sb ? (double)sb[(n / gnb) * nkb + k / gkb] : 1.0);
            acc += s * tab[A8[m * K + k]] * tab[B8[n * K + k]];
        }
        out[i] = acc;
    }
    free(tab);
}
