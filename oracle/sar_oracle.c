/*
 * sar_oracle.c -- plain, slow, fp64 CPU oracle for SAR range compression and
 * time-domain backprojection.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg load this file's library.  It shares no code, header,
 * table or constant generator with the CUDA library, and the CUDA library
 * never calls it.
 *
 * Sources (pages are cited by title and section):
 *   - "GPU-accelerated backprojection SAR imaging" (blog write-up):
 *       section 1.1 (per-pixel sum over pulses of the range-compressed echo at
 *       the pixel's range, phase-compensated), section 2.2 (linear
 *       interpolation of the compressed line; phase compensation), section 3.1
 *       (range compression = FFT, multiply by the matched filter spectrum,
 *       IFFT, per pulse), section 3.3 (the bp_kernel listing: pixel on z = 0,
 *       distance, index (d - r0) / dr, floor, linear interpolation, phase
 *       4 pi d / lambda, accumulate).
 *   - "Fused FFT -> filter -> IFFT for SAR on Apple Silicon": section 3.1
 *       (range compression per line), section 3.2 (IFFT(x) = conj(FFT(conj x))/N
 *       -- used only by the tests as an identity to pin the FFT here), sections
 *       2.1 and 5.1 (range-Doppler image formation: azimuth DFT, migration
 *       correction by sinc interpolation, azimuth matched filter, IDFT).
 *   - "Ultra-high-resolution airborne SAR on CUDA": section 5.1 (chirp-z /
 *       Bluestein transform for lengths that are not powers of two).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - chirp: baseband up-chirp exp(j pi K tau^2), K = B / Tp, on the integer
 *     samples n with -Tp fs / 2 <= n < Tp fs / 2 (Tp fs snapped to an integer
 *     when it is one), stored circularly centred on index 0 of an N-point line;
 *   - matched filter H = conj(DFT_N(h)), no amplitude normalisation;
 *   - range upsampling by U: the N-point spectrum Y is zero-padded to U N
 *     points, bins k with 2k >= N going to the negative-frequency end, and
 *     rc = U * IDFT_{UN}(Y') (IDFT including 1/(UN)), so rc_U[U m] = rc_1[m];
 *   - backprojection samples outside [0, U N) contribute zero (the listing in
 *     section 3.3 clamps instead; the benchmark scenes never reach the edges);
 *   - floor is the mathematical floor; the sum over pulses runs in pulse order.
 *
 * Layouts: complex numbers are interleaved (re, im).  raw is [lines][N]
 * complex64; rc is [lines][U N] complex128; positions are [pulses][3] float64;
 * images are [ny][nx] complex128, x fastest.
 */
#include <complex.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_C0 299792458.0

typedef double complex cplx;

typedef struct {
    double fc, bandwidth, pulse_width, fs, range_start;
    int32_t n_pulses, n_range, upsample;
} or_radar;

typedef struct {
    double x0, y0, z0, dx, dy;
    int32_t nx, ny;
} or_grid;

/* ---------------------------------------------------------------- FFT ---- */

static int is_pow2(int64_t n) { return n > 0 && (n & (n - 1)) == 0; }

/* In-place iterative radix-2 DFT of length n (a power of two):
 * X[k] = sum_j x[j] exp(sign * 2 pi i j k / n), no scaling.
 * Twiddles come straight from cos/sin of each index (no recurrences). */
static void fft_pow2(cplx *x, int64_t n, int sign)
{
    if (n <= 1) return;
    for (int64_t i = 1, j = 0; i < n; i++) {        /* bit-reversal permutation */
        int64_t bit = n >> 1;
        for (; j & bit; bit >>= 1) j ^= bit;
        j ^= bit;
        if (i < j) { cplx t = x[i]; x[i] = x[j]; x[j] = t; }
    }
    cplx *w = malloc(sizeof(cplx) * (size_t)(n / 2));
    for (int64_t t = 0; t < n / 2; t++) {
        double a = sign * 2.0 * M_PI * (double)t / (double)n;
        w[t] = cos(a) + I * sin(a);
    }
    for (int64_t len = 2; len <= n; len <<= 1) {
        int64_t half = len / 2, step = n / len;
        for (int64_t s = 0; s < n; s += len)
            for (int64_t k = 0; k < half; k++) {
                cplx u = x[s + k];
                cplx v = x[s + k + half] * w[k * step];
                x[s + k] = u + v;
                x[s + k + half] = u - v;
            }
    }
    free(w);
}

/* DFT of any length n via Bluestein's chirp-z identity
 * j k = (j^2 + k^2 - (k - j)^2) / 2, which turns the DFT into a linear
 * convolution evaluated with power-of-two FFTs of length m >= 2n - 1.
 * Same sign convention and no scaling, like fft_pow2. */
static void dft_bluestein(cplx *x, int64_t n, int sign)
{
    int64_t m = 1;
    while (m < 2 * n - 1) m <<= 1;
    cplx *w = malloc(sizeof(cplx) * (size_t)n);    /* w_t = exp(sign i pi t^2 / n) */
    for (int64_t t = 0; t < n; t++) {
        int64_t t2 = (t * t) % (2 * n);             /* the phase is periodic in t^2 with period 2n */
        double a = sign * M_PI * (double)t2 / (double)n;
        w[t] = cos(a) + I * sin(a);
    }
    cplx *A = calloc((size_t)m, sizeof(cplx));
    cplx *B = calloc((size_t)m, sizeof(cplx));
    for (int64_t j = 0; j < n; j++) A[j] = x[j] * w[j];
    B[0] = conj(w[0]);
    for (int64_t t = 1; t < n; t++) { B[t] = conj(w[t]); B[m - t] = conj(w[t]); }
    fft_pow2(A, m, -1);
    fft_pow2(B, m, -1);
    for (int64_t k = 0; k < m; k++) A[k] *= B[k];
    fft_pow2(A, m, +1);
    for (int64_t k = 0; k < n; k++) x[k] = w[k] * A[k] / (double)m;
    free(w); free(A); free(B);
}

/* X[k] = sum_j x[j] exp(sign 2 pi i j k / n), in place, no scaling. */
void or_dft(double *xy, int64_t n, int sign)
{
    cplx *x = (cplx *)xy;
    if (is_pow2(n)) fft_pow2(x, n, sign);
    else dft_bluestein(x, n, sign);
}

/* ----------------------------------------------------- matched filter ---- */

/* Number of samples the transmitted pulse spans: Tp fs, snapped to an integer
 * when it is one within 1e-6. */
int32_t or_chirp_count(const or_radar *r)
{
    double x = r->pulse_width * r->fs;
    double k = nearbyint(x);
    return (int32_t)(fabs(x - k) < 1e-6 ? k : floor(x));
}

/* Range weighting of the reference chirp ("GPU-accelerated backprojection
 * SAR imaging", section 3.1: an unweighted matched filter leaves range
 * sidelobes of about -13 dB; Hamming or Taylor weighting lowers them and widens
 * the main lobe).  Reading: the weight multiplies the nc samples of the
 * reference chirp in time, sample i = s - s_first in [0, nc).
 *   kind 0: none, w = 1;
 *   kind 1: Hamming, w = 0.54 - 0.46 cos(2 pi i / (nc - 1));
 *   kind 2: Taylor with nbar terms and peak sidelobes sll_db below the peak
 *     (Taylor's line-source distribution sampled at the chirp samples):
 *     A = acosh(10^(sll_db / 20)) / pi,  sigma^2 = nbar^2 / (A^2 + (nbar - 1/2)^2),
 *     F_m = (-1)^(m+1) / 2 * prod_{n=1}^{nbar-1} (1 - m^2 / (sigma^2 (A^2 + (n - 1/2)^2)))
 *                          / prod_{n=1, n != m}^{nbar-1} (1 - m^2 / n^2),   m = 1 .. nbar - 1,
 *     w = 1 + 2 sum_m F_m cos(2 pi m x),  x = (i - (nc - 1) / 2) / nc.
 * Writes nc weights. */
void or_window(int32_t kind, int32_t nc, int32_t nbar, double sll_db, double *w)
{
    for (int32_t i = 0; i < nc; i++) w[i] = 1.0;
    if (kind == 1) {
        for (int32_t i = 0; i < nc; i++) w[i] = 0.54 - 0.46 * cos(2.0 * M_PI * i / (double)(nc - 1));
    } else if (kind == 2) {
        const double A = acosh(pow(10.0, sll_db / 20.0)) / M_PI;
        const double sig2 = (double)nbar * nbar / (A * A + (nbar - 0.5) * (nbar - 0.5));
        double *F = calloc((size_t)(nbar > 1 ? nbar : 1), sizeof(double));
        for (int32_t m = 1; m < nbar; m++) {
            double num = 1.0, den = 1.0;
            for (int32_t k = 1; k < nbar; k++) {
                num *= 1.0 - (double)m * m / (sig2 * (A * A + (k - 0.5) * (k - 0.5)));
                if (k != m) den *= 1.0 - (double)m * m / ((double)k * k);
            }
            F[m] = ((m % 2) ? 0.5 : -0.5) * num / den;
        }
        for (int32_t i = 0; i < nc; i++) {
            const double x = (i - 0.5 * (nc - 1)) / nc;
            double v = 1.0;
            for (int32_t m = 1; m < nbar; m++) v += 2.0 * F[m] * cos(2.0 * M_PI * m * x);
            w[i] = v;
        }
        free(F);
    }
}

/* The reference chirp h on an N-point circular line (centred on index 0),
 * weighted by or_window(kind, ...), then H = conj(DFT_N h).  Writes N complex
 * values. */
void or_matched_filter_w(const or_radar *r, int32_t n, int32_t kind, int32_t nbar, double sll_db, double *H_out)
{
    cplx *h = calloc((size_t)n, sizeof(cplx));
    double K = r->bandwidth / r->pulse_width;
    int32_t nc = or_chirp_count(r);
    double *w = malloc(sizeof(double) * (size_t)nc);
    or_window(kind, nc, nbar, sll_db, w);
    /* integer sample offsets s with -nc/2 <= s < nc/2; the first is s_first = -floor(nc / 2) */
    const int64_t s_first = -(int64_t)(nc / 2);
    for (int64_t s = -(int64_t)n; s <= (int64_t)n; s++) {
        if (2 * s < -nc || 2 * s >= nc) continue;
        double tau = (double)s / r->fs;
        int64_t idx = ((s % n) + n) % n;
        h[idx] = w[s - s_first] * cexp(I * M_PI * K * tau * tau);
    }
    or_dft((double *)h, n, -1);
    cplx *H = (cplx *)H_out;
    for (int32_t k = 0; k < n; k++) H[k] = conj(h[k]);
    free(w);
    free(h);
}

/* The unweighted matched filter. */
void or_matched_filter(const or_radar *r, int32_t n, double *H_out)
{
    or_matched_filter_w(r, n, 0, 0, 0.0, H_out);
}

/* ------------------------------------------------- range compression ---- */

/* Range-compress n_lines lines of raw [n_lines][N] complex64 into
 * rc [n_lines][U N] complex128 with the matched filter weighted by
 * or_window(kind, ...):
 *   X = DFT_N(s); Y = X H; Y' = zero-pad of Y to U N points (bins with
 *   2k >= N at the top end); rc = U * IDFT_{UN}(Y') with IDFT's 1/(U N).  */
void or_range_compress_w(const or_radar *r, const float *raw, int64_t n_lines, int32_t kind, int32_t nbar,
                         double sll_db, double *rc_out, int threads)
{
    const int32_t n = r->n_range, U = r->upsample;
    const int64_t un = (int64_t)U * n;
    cplx *H = malloc(sizeof(cplx) * (size_t)n);
    or_matched_filter_w(r, n, kind, nbar, sll_db, (double *)H);
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t line = 0; line < n_lines; line++) {
        cplx *X = malloc(sizeof(cplx) * (size_t)n);
        const float *s = raw + 2 * (size_t)line * (size_t)n;
        for (int32_t k = 0; k < n; k++) X[k] = (double)s[2 * k] + I * (double)s[2 * k + 1];
        or_dft((double *)X, n, -1);
        cplx *Yp = calloc((size_t)un, sizeof(cplx));
        for (int32_t k = 0; k < n; k++) {
            cplx y = X[k] * H[k];
            if (2 * (int64_t)k < n) Yp[k] = y;            /* non-negative frequencies */
            else Yp[un - n + k] = y;                       /* negative frequencies (incl. Nyquist) */
        }
        or_dft((double *)Yp, un, +1);
        cplx *out = (cplx *)rc_out + (size_t)line * (size_t)un;
        for (int64_t j = 0; j < un; j++) out[j] = Yp[j] * (double)U / (double)un;
        free(X); free(Yp);
    }
    free(H);
}

/* Unweighted range compression. */
void or_range_compress(const or_radar *r, const float *raw, int64_t n_lines, double *rc_out, int threads)
{
    or_range_compress_w(r, raw, n_lines, 0, 0, 0.0, rc_out, threads);
}

/* ------------------------------------------------------- backprojection ---- */

/* Kernel of the 8-tap sinc interpolation ("GPU-accelerated backprojection SAR
 * imaging", section 2.2 names sinc interpolation as the accurate choice; the
 * truncation length and taper are this oracle's reading):
 *   h(d) = sinc(d) (1 + cos(pi d / 4)) / 2 for |d| < 4, 0 otherwise,
 *   sinc(d) = sin(pi d) / (pi d), sinc(0) = 1. */
double or_sinc8_kernel(double d)
{
    if (fabs(d) >= 4.0) return 0.0;
    const double s = d == 0.0 ? 1.0 : sin(M_PI * d) / (M_PI * d);
    return s * 0.5 * (1.0 + cos(M_PI * d / 4.0));
}

/* Sample of line[0 .. un) at fractional index q: interp 0 is the linear
 * L(q) = (1 - f) line[i] + f line[i + 1]; interp 1 the 8-tap sinc
 * sum_k h(f - k) line[i + k] / sum_k h(f - k), k = -3 .. 4; with i = floor(q),
 * f = q - i, and samples outside [0, un) taken as zero. */
static cplx or_interp(const cplx *line, int64_t un, double q, int interp)
{
    const double fi = floor(q);
    const double f = q - fi;
    const int64_t i = (int64_t)fi;
    if (interp == 0) {
        cplx v0 = (i >= 0 && i < un) ? line[i] : 0.0;
        cplx v1 = (i + 1 >= 0 && i + 1 < un) ? line[i + 1] : 0.0;
        return (1.0 - f) * v0 + f * v1;
    }
    cplx num = 0.0;
    double den = 0.0;
    for (int k = -3; k <= 4; k++) {
        const double w = or_sinc8_kernel(f - (double)k);
        den += w;
        if (i + k >= 0 && i + k < un) num += w * line[i + k];
    }
    return num / den;
}

/* Backproject pulses [pulse_begin, pulse_begin + pulse_count) of rc [pulses][U N]
 * complex128 into pixels.  pixels == NULL means every pixel of the grid in
 * row-major order; otherwise pixels holds n_pix flat indices iy * nx + ix.
 * out[p] = (accumulate ? out[p] : 0) + sum_n L_n(q) exp(+j 4 pi fc R / c0),
 * R = |pixel - a_n|, q = (R - R_start) / dr_U, dr_U = c0 / (2 fs U), and L_n
 * the interpolation of line n (or_interp; interp 0 linear, 1 sinc). */
void or_backproject_interp(const or_radar *r, const or_grid *g, const double *rc, const double *pos,
                           int32_t pulse_begin, int32_t pulse_count, const int64_t *pixels, int64_t n_pix,
                           double *out, int accumulate, int interp, int threads)
{
    const int64_t un = (int64_t)r->upsample * r->n_range;
    const double dr = OR_C0 / (2.0 * r->fs * (double)r->upsample);
    const double k4 = 4.0 * M_PI * r->fc / OR_C0;
    const int64_t total = pixels ? n_pix : (int64_t)g->nx * g->ny;
    const cplx *rcz = (const cplx *)rc;
    cplx *o = (cplx *)out;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 16)
#endif
    for (int64_t p = 0; p < total; p++) {
        int64_t flat = pixels ? pixels[p] : p;
        int64_t ix = flat % g->nx, iy = flat / g->nx;
        double x = g->x0 + (double)ix * g->dx;
        double y = g->y0 + (double)iy * g->dy;
        double z = g->z0;
        cplx acc = 0.0;
        for (int32_t n = pulse_begin; n < pulse_begin + pulse_count; n++) {
            const double *a = pos + 3 * (size_t)n;
            double ddx = x - a[0], ddy = y - a[1], ddz = z - a[2];
            double R = sqrt(ddx * ddx + ddy * ddy + ddz * ddz);
            double q = (R - r->range_start) / dr;
            cplx val = or_interp(rcz + (size_t)n * (size_t)un, un, q, interp);
            acc += val * cexp(I * k4 * R);
        }
        o[p] = accumulate ? o[p] + acc : acc;
    }
}

/* Linear interpolation (or_backproject_interp with interp 0). */
void or_backproject(const or_radar *r, const or_grid *g, const double *rc, const double *pos,
                    int32_t pulse_begin, int32_t pulse_count, const int64_t *pixels, int64_t n_pix,
                    double *out, int accumulate, int threads)
{
    or_backproject_interp(r, g, rc, pos, pulse_begin, pulse_count, pixels, n_pix, out, accumulate, 0, threads);
}

/* Interpolate line[0 .. un) at the n_q fractional indices q (for the tests). */
void or_interp_line(const double *line, int64_t un, const double *q, int64_t n_q, int interp, double *out)
{
    for (int64_t j = 0; j < n_q; j++) ((cplx *)out)[j] = or_interp((const cplx *)line, un, q[j], interp);
}

/* ---------------------------------------------------- range-Doppler ---- */

/* Range-Doppler image formation of a straight, uniformly sampled track
 * ("Fused FFT -> filter -> IFFT for SAR on Apple Silicon", sections 2.1 and
 * 5.1: range compression, azimuth DFT, range cell migration correction by sinc
 * interpolation, azimuth matched filter, azimuth IDFT; "Ultra-high-resolution
 * airborne SAR on CUDA", section 2 names the same three steps).
 *
 * rc [Na][Nr] complex128: range-compressed lines at the native spacing
 * dr = c0 / (2 fs) (upsample 1); du: along-track distance between pulses (m).
 * img [Nr][Na] complex128: row i is slant range R0 = R_start + i dr, column n
 * the along-track position of pulse n.
 *   S(m, i)  = sum_n rc[n][i] exp(-2 pi i m n / Na);
 *   k_m      = m_s / (Na du) cycles per metre, m_s the signed bin (Nyquist negative);
 *   D_m      = sqrt(1 - (lambda k_m / 2)^2);
 *   S'(m, i) = S(m, .) interpolated by the 8-tap sinc at i + R0 (1/D_m - 1) / dr
 *              (rcmc != 0; otherwise S(m, i) itself);
 *   S''      = S' exp(+j 4 pi R0 D_m / lambda);
 *   img[i][n] = (1/Na) sum_m S''(m, i) exp(+2 pi i m n / Na).
 * Returns 0, or -1 when lambda / (4 du) >= 1 (D_m would not be real). */
int or_range_doppler(const or_radar *r, double du, const double *rc, double *img, int rcmc, int threads)
{
    const int64_t na = r->n_pulses, nr = r->n_range;
    const double dr = OR_C0 / (2.0 * r->fs);
    const double lambda = OR_C0 / r->fc;
    if (!(du > 0.0) || lambda / (4.0 * du) >= 1.0) return -1;
    const cplx *in = (const cplx *)rc;
    cplx *out = (cplx *)img;
    cplx *S = malloc(sizeof(cplx) * (size_t)(na * nr));          /* [Na][Nr]: Doppler bin, range bin */
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 8)
#endif
    for (int64_t i = 0; i < nr; i++) {
        cplx *col = malloc(sizeof(cplx) * (size_t)na);
        for (int64_t n = 0; n < na; n++) col[n] = in[n * nr + i];
        or_dft((double *)col, na, -1);
        for (int64_t m = 0; m < na; m++) S[m * nr + i] = col[m];
        free(col);
    }
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 8)
#endif
    for (int64_t m = 0; m < na; m++) {
        const int64_t ms = (2 * m < na) ? m : m - na;
        const double kx = (double)ms / ((double)na * du);
        const double D = sqrt(1.0 - (lambda * kx / 2.0) * (lambda * kx / 2.0));
        cplx *row = malloc(sizeof(cplx) * (size_t)nr);
        memcpy(row, S + m * nr, sizeof(cplx) * (size_t)nr);
        for (int64_t i = 0; i < nr; i++) {
            const double R0 = r->range_start + (double)i * dr;
            const cplx v = rcmc ? or_interp(row, nr, (double)i + R0 * (1.0 / D - 1.0) / dr, 1) : row[i];
            S[m * nr + i] = v * cexp(I * 4.0 * M_PI * R0 * D / lambda);
        }
        free(row);
    }
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 8)
#endif
    for (int64_t i = 0; i < nr; i++) {
        cplx *col = malloc(sizeof(cplx) * (size_t)na);
        for (int64_t m = 0; m < na; m++) col[m] = S[m * nr + i];
        or_dft((double *)col, na, +1);
        for (int64_t n = 0; n < na; n++) out[i * na + n] = col[n] / (double)na;
        free(col);
    }
    free(S);
    return 0;
}

int or_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
