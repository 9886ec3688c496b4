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

template <int N>
constexpr int rd_min_ctas() { return N >= 8192 ? 1 : N == 4096 ? 2 : (16 * 32) / (N / 16); }

// Azimuth DFT of every range bin, in place: row i of s [nr][N] (the range bin's N pulses) becomes
// its N-point spectrum in natural bin order.
template <int N>
__global__ void __launch_bounds__(N / 16, rd_min_ctas<N>()) rd_azfft_kernel(float2 *__restrict__ s, int nr, RdaArgs args)
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

// Normalised 8-tap sinc weights for fraction f in [0, 1]: w[k] for samples r - 3 + k.  The
// unnormalised weights (-1)^k W(f - k) prod_{j != k} (f - j) are those of the backprojection's
// sinc option (the common factors sin(pi f) / pi and prod_j (f - j) cancel in the normalisation).
__device__ __forceinline__ void sinc8_weights(float f, float (&w)[8])
{
    constexpr float r2 = 0.35355339059327376220f;             // sqrt(2) / 4
    constexpr float kC[8] = {r2, 0.0f, -r2, 0.5f, -r2, 0.0f, r2, -0.5f};
    constexpr float kS[8] = {r2, -0.5f, r2, 0.0f, -r2, 0.5f, -r2, 0.0f};
    constexpr float kH[8] = {-0.5f, 0.5f, -0.5f, 0.5f, -0.5f, 0.5f, -0.5f, 0.5f};
    float sq, cq;
    __sincosf(0.78539816339744830962f * f, &sq, &cq);
    float d[8], pre[8];
#pragma unroll
    for (int k = 0; k < 8; k++) d[k] = f + (float)(3 - k);
    pre[0] = 1.0f;
#pragma unroll
    for (int k = 1; k < 8; k++) pre[k] = pre[k - 1] * d[k - 1];
    float suf = 1.0f, sum = 0.0f;
#pragma unroll
    for (int k = 7; k >= 0; k--) {
        w[k] = fmaf(cq, kC[k], fmaf(sq, kS[k], kH[k])) * (pre[k] * suf);
        suf *= d[k];
        sum += w[k];
    }
    const float inv = __fdividef(1.0f, sum);
#pragma unroll
    for (int k = 0; k < 8; k++) w[k] *= inv;
}

// Migration correction, azimuth matched filter and azimuth IDFT of output range bin i: s [nr][N]
// holds the range-Doppler spectrum (row = range bin, natural Doppler order), img [nr][N] the image.
template <int N>
__global__ void __launch_bounds__(N / 16, rd_min_ctas<N>()) rd_compress_kernel(const float2 *__restrict__ s,
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
#pragma unroll
        for (int p = 0; p < 16; p++) {
            const int m = t + T * p;
            // migration: sample the range axis at q = i + (R0 / dr)(1/D_m - 1)
            const float q = (float)i + r_bins * __ldg(args.rcm + m);
            const float fl = floorf(q);
            const int r0 = (int)fl - 3;
            // the eight taps first (rows clamped into the axis, so every load is in bounds and none
            // waits on a branch), the weights while they are in flight; taps outside the axis
            // weigh zero
            float2 sv[8];
#pragma unroll
            for (int k = 0; k < 8; k++) sv[k] = __ldg(s + (int64_t)min(max(r0 + k, 0), nr - 1) * N + m);
            float w[8];
            sinc8_weights(q - fl, w);
            float2 v = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int k = 0; k < 8; k++) {
                const float wk = (r0 + k >= 0 && r0 + k < nr) ? w[k] : 0.0f;
                v.x = fmaf(wk, sv[k].x, v.x);
                v.y = fmaf(wk, sv[k].y, v.y);
            }
            // matched filter phase, turns: frac((2/lambda) R0) - (2/lambda)(1 - D_m) R0 (double-float)
            const float2 c = __ldg(args.phc + m);
            const float pr = c.x * r_hi;
            const float e = fmaf(c.x, r_lo, fmaf(c.y, r_hi, fmaf(c.x, r_hi, -pr)));
            float tq = (pr - rintf(pr)) + e;
            float turns = ph0 - tq;
            turns -= rintf(turns);
            float sn, cs;
            __sincosf(6.28318530717958648f * turns, &sn, &cs);
            // conjugate of the filtered value: the inverse DFT runs as conj(DFT(conj(.)))
            x[p] = make_float2(v.x * cs - v.y * sn, -(v.x * sn + v.y * cs));
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
