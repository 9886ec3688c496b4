// bp_kernel.cu -- time-domain backprojection ("GPU-accelerated backprojection
// SAR imaging", sections 1.1, 2.1-2.3 and 3.3): every pixel sums, over pulses,
// the linearly interpolated range-compressed echo at its range, multiplied by
// exp(+j 4 pi fc R / c0).
//
// Work decomposition.  One CTA owns a 32 x 32 pixel tile (warps run along x,
// the azimuth axis, so the 32 lanes of a warp read nearly the same range
// samples); each thread keeps four pixels' complex sums in registers for the
// whole pulse range.  The CTA walks the pulses in batches: for each pulse of a
// batch it first evaluates, in float64, the range R0 from the antenna to the
// tile centre, then stages the window of compressed samples the tile can touch
// in shared memory (section 2.3 of the same page stages echo data per image
// block the same way).
//
// Range and phase precision.  At X band the phase 4 pi R / lambda needs R to
// ~1e-5 m at R ~ 6 km, beyond float32 (the listing in section 3.3 computes the
// whole distance in float and loses ~0.1 rad).  Here each pixel's range is a
// float32 offset from the float64 tile-centre range: with d the pixel offset
// from the tile centre, w the antenna-to-centre vector and g = 2 w.d/R0 + |d|^2/R0,
//     R - R0 = g/2 - g^2/(8 R0) + g^3/(16 R0^2) - 5 g^4/(128 R0^3) + O(g^5/R0^4),
// evaluated by Horner's rule in range-bin units (the binomial series of
// R0 sqrt(1 + g/R0)).  |d| <= 11 m and R0 >= 100 tile half-diagonals keep the
// truncation below 1e-7 m.
//
// Interpolation and phase in one staged pair.  With q the pixel's fractional
// bin relative to the window origin o (half a bin shifted: qm = q - 1/2) and
// i = round(qm) = floor(q), the linear interpolation (1 - f) v_i + f v_{i+1},
// f = q - i, equals tau_i + qm sigma_i with sigma_i = v_{i+1} - v_i and
// tau_i = v_i - (i - 1/2) sigma_i.  The phase is 2 pi [(2/lambda) R_start +
// kappa (o + 1/2)] + 2 pi kappa qm, kappa = 2 dr / lambda, so the per-(tile,
// pulse) part is one angle theta and the per-pixel part one fused multiply-add.
// Per pixel and pulse that leaves: 2 FMA (range offset), 4 FMA (series),
// 1 add (round), 1 integer op (address), 1 shared 128-bit load, 2 FMA (interp),
// 1 FMA + sin/cos on the SFU (phase), 4 FMA (complex multiply-accumulate).
#include "sar_internal.cuh"

namespace sar {
namespace {

struct __align__(16) PulseParams {
    float a, b, c, q0m;       // g_bins = a dx + b dy + c |d|^2 ; qm0 = frac(bin of R0) - 1/2
    float c1, c2, c3, theta;  // series coefficients in bins; phase of the window origin (rad)
};

constexpr float kRoundMagic = 12582912.0f;                 // 1.5 * 2^23: x + magic rounds x to an integer
constexpr unsigned kRoundMagicBits = 0x4B400000u;

__device__ __forceinline__ float4 lds128(unsigned addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

template <bool kCheck>
__global__ void __launch_bounds__(kBpThreads, 3) bp_kernel(BpArgs args)
{
    extern __shared__ float4 smem4[];
    const int pb_max = args.pulses_per_batch;
    PulseParams *prm = reinterpret_cast<PulseParams *>(smem4);
    int *origin = reinterpret_cast<int *>(prm + pb_max);
    float4 *stage = smem4 + 2 * pb_max + (pb_max + 3) / 4;       // [pb_max][w] of (tau.re, tau.im, sigma.re, sigma.im)
    const int w = args.w, wh = args.wh;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tile_x = blockIdx.x, tile_y = blockIdx.y;
    // tile centre (float64) and this thread's pixel offsets from it (float32)
    const double cx = args.x0 + ((double)tile_x * kBpTileX + 0.5 * (kBpTileX - 1)) * args.dx;
    const double cy = args.y0 + ((double)tile_y * kBpTileY + 0.5 * (kBpTileY - 1)) * args.dy;
    const float ox = ((float)lane - 0.5f * (kBpTileX - 1)) * args.dxf;
    float oy[kBpRowsPerThread], od2[kBpRowsPerThread];
#pragma unroll
    for (int k = 0; k < kBpRowsPerThread; k++) {
        const int ly = warp * kBpRowsPerThread + k;
        oy[k] = ((float)ly - 0.5f * (kBpTileY - 1)) * args.dyf;
        od2[k] = fmaf(ox, ox, oy[k] * oy[k]);
    }
    float acc_re[kBpRowsPerThread], acc_im[kBpRowsPerThread];
#pragma unroll
    for (int k = 0; k < kBpRowsPerThread; k++) acc_re[k] = acc_im[k] = 0.0f;

    const unsigned stage_base = (unsigned)__cvta_generic_to_shared(stage);
    const int64_t ns = args.n_samples;

    for (int n0 = args.pulse_begin; n0 < args.pulse_end; n0 += pb_max) {
        const int pb = min(pb_max, args.pulse_end - n0);
        // ---- per-(tile, pulse) reference range in float64
        if (threadIdx.x < pb) {
            const int n = n0 + threadIdx.x;
            const double wx = cx - args.pos[3 * n + 0];
            const double wy = cy - args.pos[3 * n + 1];
            const double wz = args.z0 - args.pos[3 * n + 2];
            const double r2 = fma(wx, wx, fma(wy, wy, wz * wz));
            const float s0 = sqrtf((float)r2);
            const double s0d = (double)s0;
            const float res = (float)fma(-s0d, s0d, r2);                  // r2 - s0^2, exact enough in float
            const double r0 = s0d + (double)(res * (0.5f / s0));          // one Newton step
            const double qg = (r0 - args.range_start) * args.inv_dr;       // fractional global bin of the centre
            // Validity: finite, far enough for the range expansion (which bounds every pixel's offset
            // inside the staged window), and a representable window origin.  Otherwise flag the plan
            // and zero this pulse's parameters: every pixel then reads entry wh, inside the window.
            const bool ok = (r0 >= (double)args.min_range_tiles) && (fabs(qg) < 1.0e9);
            const double o = ok ? floor(qg) : 0.0;
            // 1 / (r0 dr) to float64 accuracy: float reciprocal refined by one Newton step
            const float inv_f = 1.0f / (float)r0;
            const double inv_r0d = (double)inv_f * fma(-r0, (double)inv_f, 2.0);
            const double k = inv_r0d * args.inv_dr;
            const float inv_r0 = (float)inv_r0d;
            const float e = args.dr * inv_r0;
            PulseParams p;
            p.a = (float)(2.0 * wx * k);          // each coefficient rounded to float once
            p.b = (float)(2.0 * wy * k);
            p.c = (float)k;
            p.q0m = (float)(qg - o) - 0.5f;
            p.c1 = -0.125f * e;
            p.c2 = 0.0625f * e * e;
            p.c3 = -0.0390625f * e * e * e;
            double t = fma(args.kappa, o + 0.5, args.phase0_turns);
            t -= rint(t);
            p.theta = (float)(6.283185307179586 * t);
            if (!ok) {
                p.a = p.b = p.c = p.q0m = p.c1 = p.c2 = p.c3 = p.theta = 0.0f;
                atomicOr(args.err, kDevErrGeometry);
            }
            prm[threadIdx.x] = p;
            origin[threadIdx.x] = (int)o;
        }
        __syncthreads();
        // ---- stage the windows: entry e <-> global bin origin + e - wh
        for (int p = warp; p < pb; p += kBpThreads / 32) {
            const float2 *line = args.rc + (int64_t)(n0 + p) * ns;
            const int64_t first = (int64_t)origin[p] - wh;
            float4 *row = stage + p * w;
            for (int e = lane; e < w; e += 32) {
                const int64_t I = first + e;
                const float2 v0 = (I >= 0 && I < ns) ? __ldg(line + I) : make_float2(0.0f, 0.0f);
                const float2 v1 = (I + 1 >= 0 && I + 1 < ns) ? __ldg(line + I + 1) : make_float2(0.0f, 0.0f);
                const float sr = v1.x - v0.x, si = v1.y - v0.y;
                const float im = (float)(e - wh) - 0.5f;
                row[e] = make_float4(fmaf(-im, sr, v0.x), fmaf(-im, si, v0.y), sr, si);
            }
        }
        __syncthreads();
        // ---- pixel x pulse inner loop
        for (int p = 0; p < pb; p++) {
            const PulseParams P = prm[p];
            // address of entry round(qm) + wh, from the bit pattern of qm + magic (32-bit wrap-around)
            const unsigned base = stage_base + (unsigned)(p * w) * 16u + 16u * (unsigned)wh - 16u * kRoundMagicBits;
            const float adx = P.a * ox;
#pragma unroll
            for (int k = 0; k < kBpRowsPerThread; k++) {
                const float g = fmaf(P.b, oy[k], fmaf(P.c, od2[k], adx));
                float t = fmaf(g, P.c3, P.c2);
                t = fmaf(g, t, P.c1);
                t = fmaf(g, t, 0.5f);
                const float qm = fmaf(g, t, P.q0m);
                const float rnd = __fadd_rn(qm, kRoundMagic);
                const unsigned addr = base + (__float_as_uint(rnd) << 4);
                if (kCheck) {
                    const int e = (int)(__float_as_uint(rnd) - kRoundMagicBits) + wh;
                    if (e < 0 || e >= w) {
                        atomicOr(args.err, kDevErrBounds);
                        continue;
                    }
                }
                const float4 v = lds128(addr);
                const float vr = fmaf(qm, v.z, v.x);
                const float vi = fmaf(qm, v.w, v.y);
                float s, c;
                __sincosf(fmaf(qm, args.two_pi_kappa, P.theta), &s, &c);
                acc_re[k] = fmaf(vr, c, acc_re[k]);
                acc_re[k] = fmaf(-vi, s, acc_re[k]);
                acc_im[k] = fmaf(vr, s, acc_im[k]);
                acc_im[k] = fmaf(vi, c, acc_im[k]);
            }
        }
        __syncthreads();
    }
    // ---- store
    const int ix = tile_x * kBpTileX + lane;
#pragma unroll
    for (int k = 0; k < kBpRowsPerThread; k++) {
        const int iy = tile_y * kBpTileY + warp * kBpRowsPerThread + k;
        if (ix < args.nx && iy < args.ny) {
            float2 *dst = args.image + (int64_t)iy * args.nx + ix;
            float2 v = make_float2(acc_re[k], acc_im[k]);
            if (args.accumulate) {
                const float2 old = *dst;
                v.x += old.x;
                v.y += old.y;
            }
            *dst = v;
        }
    }
}

}  // namespace

size_t bp_smem_bytes(int w, int pulses_per_batch)
{
    const int pb = pulses_per_batch;
    return (size_t)(2 * pb + (pb + 3) / 4) * sizeof(float4) + (size_t)pb * w * sizeof(float4);
}

cudaError_t bp_configure()
{
    cudaError_t e = cudaFuncSetAttribute(bp_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(bp_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
}

cudaError_t launch_bp(const BpArgs &a, bool check_bounds, cudaStream_t s)
{
    if (a.pulse_end <= a.pulse_begin) return cudaSuccess;
    const dim3 grid(a.tiles_x, a.tiles_y);
    const size_t smem = bp_smem_bytes(a.w, a.pulses_per_batch);
    if (check_bounds) bp_kernel<true><<<grid, kBpThreads, smem, s>>>(a);
    else bp_kernel<false><<<grid, kBpThreads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace sar
