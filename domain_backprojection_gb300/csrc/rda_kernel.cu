// rda_kernel.cu -- range-Doppler image formation of a straight, uniformly
// sampled track ("Fused FFT -> filter -> IFFT for SAR on Apple Silicon",
// sections 2.1 and 5.1): after range compression, a transpose, one azimuth DFT
// per range bin, and one fused kernel per output range bin that corrects the
// range cell migration by 8-tap sinc interpolation across range bins, applies
// the phase-only azimuth matched filter and runs the azimuth IDFT.
//
// With m the Doppler bin (signed m_s, Nyquist negative), k_m = m_s / (Na du)
// cycles per metre and D_m = sqrt(1 - (lambda k_m / 2)^2), output range bin i
// (slant range R0 = R_start + i dr) takes
//     S'(m, i) = sum_k h(f - k) S(m, r + k) / sum_k h(f - k),  q = i + R0 (1/D_m - 1) / dr,
//                r = floor(q), f = q - r, k = -3 .. 4 (samples outside the range axis zero),
//     img[i][n] = (1/Na) sum_m S'(m, i) exp(+j 4 pi R0 D_m / lambda) exp(+j 2 pi m n / Na),
// h the Hann-tapered sinc of the backprojection's sinc option.  The matched
// filter's phase is 2 pi [(2/lambda) R0 - (2/lambda)(1 - D_m) R0]: the first
// term is one float64 value per range bin, the second a double-float product
// (about 48 bits) per element, so the phase stays exact to ~1e-6 rad at
// ~4e5 turns.
#include "fft_reg.cuh"

namespace sar {
namespace {

constexpr int kTrTile = 32;

// in [rows][cols] -> out [cols][rows], 32 x 32 tiles through padded shared memory (both sides
// coalesced)
__global__ void __launch_bounds__(256) rd_transpose_kernel(const float2 *__restrict__ in, float2 *__restrict__ out,
                                                           int rows, int cols)
{
    __shared__ float2 tile[kTrTile][kTrTile + 1];
    const int c0 = blockIdx.x * kTrTile, r0 = blockIdx.y * kTrTile;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
    for (int k = 0; k < kTrTile; k += 8) {
        const int r = r0 + ty + k, c = c0 + tx;
        if (r < rows && c < cols) tile[ty + k][tx] = in[(int64_t)r * cols + c];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kTrTile; k += 8) {
        const int c = c0 + ty + k, r = r0 + tx;
        if (r < rows && c < cols) out[(int64_t)c * rows + r] = tile[tx][ty + k];
    }
}

// Resident CTAs per SM each kernel is built for (its register budget): 16 warps per SM for short
// transforms, one CTA at 8192 points; at 4096 points the transform alone fits 64 registers (4 CTAs)
// and the fused migration kernel 80 (3 CTAs), measured on GB300 at 0.332 -> 0.309 ms per 4096^2
// image against 2 CTAs each.
template <int N>
constexpr int rd_min_ctas() { return N >= 8192 ? 1 : N == 4096 ? 2 : (16 * 32) / (N / 16); }
template <int N>
constexpr int rd_fft_min_ctas() { return N == 4096 ? 4 : rd_min_ctas<N>(); }
template <int N>
constexpr int rd_compress_min_ctas() { return N == 4096 ? 3 : rd_min_ctas<N>(); }

// Azimuth DFT of every range bin, in place: row i of s [nr][N] (the range bin's N pulses) becomes
// its N-point spectrum in natural bin order.
template <int N>
__global__ void __launch_bounds__(N / 16, rd_fft_min_ctas<N>()) rd_azfft_kernel(float2 *__restrict__ s, int nr, RdaArgs args)
{
    extern __shared__ float4 smem4[];
    constexpr int T = N / 16;
    float2 *a = reinterpret_cast<float2 *>(smem4), *b = a;
    const int t = threadIdx.x;
    for (int i = blockIdx.x; i < nr; i += gridDim.x) {
        float2 *row = s + (int64_t)i * N;
        float2 x[16];
#pragma unroll
        for (int p = 0; p < 16; p++) x[p] = row[t + T * p];      // plain loads: the row is rewritten below
        reg_dft<N, false>(x, a, b, args.tw);
#pragma unroll
        for (int p = 0; p < 16; p++) row[t + T * p] = x[p];
    }
}

// Normalised 8-tap sinc weights for two fractions f.x, f.y in [0, 1] at once (float2 lanes: paired
// FFMA2 / FMUL2 / FADD2): w[k] for samples r - 3 + k.  The unnormalised weights
// (-1)^k W(f - k) prod_{j != k} (f - j) are those of the backprojection's sinc option (the common
// factors sin(pi f) / pi and prod_j (f - j) cancel in the normalisation).
__device__ __forceinline__ void sinc8_weights2(float2 f, float2 (&w)[8])
{
    constexpr float r2 = 0.35355339059327376220f;             // sqrt(2) / 4
    constexpr float kC[8] = {r2, 0.0f, -r2, 0.5f, -r2, 0.0f, r2, -0.5f};
    constexpr float kS[8] = {r2, -0.5f, r2, 0.0f, -r2, 0.5f, -r2, 0.0f};
    constexpr float kH[8] = {-0.5f, 0.5f, -0.5f, 0.5f, -0.5f, 0.5f, -0.5f, 0.5f};
    float2 sq, cq;
    __sincosf(0.78539816339744830962f * f.x, &sq.x, &cq.x);
    __sincosf(0.78539816339744830962f * f.y, &sq.y, &cq.y);
    float2 d[8], pre[8];
#pragma unroll
    for (int k = 0; k < 8; k++) d[k] = __fadd2_rn(f, make_float2((float)(3 - k), (float)(3 - k)));
    pre[0] = make_float2(1.0f, 1.0f);
#pragma unroll
    for (int k = 1; k < 8; k++) pre[k] = __fmul2_rn(pre[k - 1], d[k - 1]);
    float2 suf = make_float2(1.0f, 1.0f), sum = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int k = 7; k >= 0; k--) {
        const float2 wk = __ffma2_rn(cq, make_float2(kC[k], kC[k]),
                                     __ffma2_rn(sq, make_float2(kS[k], kS[k]), make_float2(kH[k], kH[k])));
        w[k] = __fmul2_rn(wk, __fmul2_rn(pre[k], suf));
        suf = __fmul2_rn(suf, d[k]);
        sum = __fadd2_rn(sum, w[k]);
    }
    const float2 inv = make_float2(__fdividef(1.0f, sum.x), __fdividef(1.0f, sum.y));
#pragma unroll
    for (int k = 0; k < 8; k++) w[k] = __fmul2_rn(w[k], inv);
}

// One element's matched filter, conjugated for the inverse transform: v exp(+j 2 pi turns) with
// turns = frac((2/lambda) R0) - (2/lambda)(1 - D_m) R0, the product in double-float (c = per-bin
// coefficient (hi, lo), R0 = r_hi + r_lo).
__device__ __forceinline__ float2 rd_filter(float2 v, float2 c, float ph0, float r_hi, float r_lo)
{
    const float pr = c.x * r_hi;
    const float e = fmaf(c.x, r_lo, fmaf(c.y, r_hi, fmaf(c.x, r_hi, -pr)));
    const float tq = (pr - rintf(pr)) + e;
    float turns = ph0 - tq;
    turns -= rintf(turns);
    float sn, cs;
    __sincosf(6.28318530717958648f * turns, &sn, &cs);
    // conjugate of the filtered value: the inverse DFT runs as conj(DFT(conj(.)))
    return make_float2(v.x * cs - v.y * sn, -(v.x * sn + v.y * cs));
}

// Migration correction, azimuth matched filter and azimuth IDFT of output range bin i: s [nr][N]
// holds the range-Doppler spectrum (row = range bin, natural Doppler order), img [nr][N] the image.
template <int N>
__global__ void __launch_bounds__(N / 16, rd_compress_min_ctas<N>()) rd_compress_kernel(const float2 *__restrict__ s,
                                                                              float2 *__restrict__ img, int nr,
                                                                              RdaArgs args)
{
    extern __shared__ float4 smem4[];
    constexpr int T = N / 16;
    float2 *a = reinterpret_cast<float2 *>(smem4), *b = a;
    const int t = threadIdx.x;
    for (int i = blockIdx.x; i < nr; i += gridDim.x) {
        const double R0 = args.range_start + (double)i * args.dr;
        const double turns0 = args.two_over_lambda * R0;
        const float ph0 = (float)(turns0 - floor(turns0));          // frac((2/lambda) R0)
        const float r_hi = (float)R0, r_lo = (float)(R0 - (double)r_hi);
        const float r_bins = (float)(R0 / args.dr);                  // R0 / dr
        float2 x[16];
        // elements in pairs (p, p + 8): the sinc weights of both come from paired float2 arithmetic
#pragma unroll
        for (int p = 0; p < 8; p++) {
            const int m0 = t + T * p, m1 = t + T * (p + 8);
            // migration: sample the range axis at q = i + (R0 / dr)(1/D_m - 1)
            const float q0 = (float)i + r_bins * __ldg(args.rcm + m0);
            const float q1 = (float)i + r_bins * __ldg(args.rcm + m1);
            const float fl0 = floorf(q0), fl1 = floorf(q1);
            const int r00 = (int)fl0 - 3, r01 = (int)fl1 - 3;
            // the taps first (rows clamped into the axis, so every load is in bounds and none waits on
            // a branch), the weights while they are in flight; taps outside the axis weigh zero
            float2 s0[8], s1[8];
#pragma unroll
            for (int k = 0; k < 8; k++) {
                s0[k] = __ldg(s + (int64_t)min(max(r00 + k, 0), nr - 1) * N + m0);
                s1[k] = __ldg(s + (int64_t)min(max(r01 + k, 0), nr - 1) * N + m1);
            }
            float2 w[8];
            sinc8_weights2(make_float2(q0 - fl0, q1 - fl1), w);
            float2 v0 = make_float2(0.0f, 0.0f), v1 = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int k = 0; k < 8; k++) {
                const float w0 = (r00 + k >= 0 && r00 + k < nr) ? w[k].x : 0.0f;
                const float w1 = (r01 + k >= 0 && r01 + k < nr) ? w[k].y : 0.0f;
                v0 = __ffma2_rn(make_float2(w0, w0), s0[k], v0);
                v1 = __ffma2_rn(make_float2(w1, w1), s1[k], v1);
            }
            x[p] = rd_filter(v0, __ldg(args.phc + m0), ph0, r_hi, r_lo);
            x[p + 8] = rd_filter(v1, __ldg(args.phc + m1), ph0, r_hi, r_lo);
        }
        reg_dft<N, false>(x, a, b, args.tw);
        float2 *out = img + (int64_t)i * N;
#pragma unroll
        for (int p = 0; p < 16; p++) out[t + T * p] = make_float2(x[p].x * args.inv_na, -x[p].y * args.inv_na);
    }
}

template <int N>
size_t rd_smem() { return (size_t)(N + N / 16) * sizeof(float2); }

template <int N>
cudaError_t rd_configure_n()
{
    cudaError_t e = cudaFuncSetAttribute(rd_azfft_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rd_smem<N>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rd_compress_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rd_smem<N>());
    return e;
}

template <int N>
void launch_rd_n(const RdaArgs &a, float2 *s, float2 *img, cudaStream_t st)
{
    const unsigned grid = (unsigned)(a.nr < (1 << 20) ? a.nr : (1 << 20));
    rd_azfft_kernel<N><<<grid, N / 16, rd_smem<N>(), st>>>(s, a.nr, a);
    rd_compress_kernel<N><<<grid, N / 16, rd_smem<N>(), st>>>(s, img, a.nr, a);
}

}  // namespace

bool rd_supported_pulses(int na) { return na == 512 || na == 1024 || na == 2048 || na == 4096 || na == 8192; }

cudaError_t rd_configure()
{
    cudaError_t e = rd_configure_n<512>();
    if (e == cudaSuccess) e = rd_configure_n<1024>();
    if (e == cudaSuccess) e = rd_configure_n<2048>();
    if (e == cudaSuccess) e = rd_configure_n<4096>();
    if (e == cudaSuccess) e = rd_configure_n<8192>();
    return e;
}

cudaError_t launch_rd(const RdaArgs &a, const float2 *rc, float2 *work, float2 *img, cudaStream_t st)
{
    const dim3 tgrid((a.nr + kTrTile - 1) / kTrTile, (a.na + kTrTile - 1) / kTrTile);
    rd_transpose_kernel<<<tgrid, 256, 0, st>>>(rc, work, a.na, a.nr);
    switch (a.na) {
    case 512: launch_rd_n<512>(a, work, img, st); break;
    case 1024: launch_rd_n<1024>(a, work, img, st); break;
    case 2048: launch_rd_n<2048>(a, work, img, st); break;
    case 4096: launch_rd_n<4096>(a, work, img, st); break;
    case 8192: launch_rd_n<8192>(a, work, img, st); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace sar
