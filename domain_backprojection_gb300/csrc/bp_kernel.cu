// bp_kernel.cu -- time-domain backprojection ("GPU-accelerated backprojection
// SAR imaging", sections 1.1, 2.1-2.3 and 3.3): every pixel sums, over pulses,
// the linearly interpolated range-compressed echo at its range, multiplied by
// exp(+j 4 pi fc R / c0).
//
// Work decomposition.  One CTA owns a 64 x 32 pixel tile, long in azimuth (x):
// pixels that differ only in x lie at nearly the same range, so the window of
// compressed samples a tile touches grows with its range (y) extent only and
// staging it is shared by twice as many pixels.  Warps run along x, so the 32
// lanes of a warp read nearly the same samples; each thread keeps four pixels'
// complex sums in registers for the whole pulse range.  The CTA walks the
// pulses in batches: for each pulse of a batch it first evaluates, in float64,
// the range R0 from the antenna to the tile centre, then stages the window of
// compressed samples the tile can touch in shared memory (section 2.3 of the
// same page stages echo data per image block the same way).  Long pulse ranges
// are split into slices (gridDim.z) whose partial images a second kernel adds
// in slice order, so that small images and the last wave still fill the GPU.
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

constexpr float kRoundMagic = 12582912.0f;                 // 1.5 * 2^23: x + magic rounds x to an integer
constexpr unsigned kRoundMagicBits = 0x4B400000u;

__device__ __forceinline__ float4 lds128(unsigned addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

// One pulse's contribution to this thread's pixels (one column, kBpRowsPerThread rows).
template <bool kCheck>
__device__ __forceinline__ void pixel_pulse(const float4 pa, const float4 pc, const int4 wv, const unsigned base,
                                            const float adx, const float *oy, const float *od2, float *acc_re,
                                            float *acc_im, const BpArgs &args)
{
#pragma unroll
    for (int k = 0; k < kBpRowsPerThread; k++) {
        const float g = fmaf(pa.y, oy[k], fmaf(pa.z, od2[k], adx));
        float t = fmaf(g, fmaf(g, pc.z, pc.y), pc.x);
        t = fmaf(g, t, 0.5f);
        const float qm = fmaf(g, t, pa.w);
        const float rnd = __fadd_rn(qm, kRoundMagic);
        const unsigned addr = base + (__float_as_uint(rnd) << 4);
        if (kCheck) {
            const int e = (int)(__float_as_uint(rnd) - kRoundMagicBits) + args.wh;
            if (e < wv.y || e > wv.z) {
                atomicOr(args.err, kDevErrBounds);
                continue;
            }
        }
        const float4 v = lds128(addr);
        const float vr = fmaf(qm, v.z, v.x);
        const float vi = fmaf(qm, v.w, v.y);
        float sn, cs;
        __sincosf(fmaf(qm, args.two_pi_kappa, pc.w), &sn, &cs);
        acc_re[k] = fmaf(vr, cs, acc_re[k]);
        acc_re[k] = fmaf(-vi, sn, acc_re[k]);
        acc_im[k] = fmaf(vr, sn, acc_im[k]);
        acc_im[k] = fmaf(vi, cs, acc_im[k]);
    }
}

// Shared memory of one CTA: per pulse of the batch two float4 of parameters
//   (a, b, c, q0m): g_bins = a dx + b dy + c |d|^2, qm0 = frac(bin of R0) - 1/2
//   (c1, c2, c3, theta): series coefficients in bins, phase of the window origin (rad)
// one int4 (origin o, first and last staged entry, unused), then the staged windows
// [pulses_per_batch][w] of (tau.re, tau.im, sigma.re, sigma.im).
template <bool kCheck, bool kPlanar>
__global__ void __launch_bounds__(kBpThreads, 2) bp_kernel(BpArgs args)
{
    extern __shared__ float4 smem4[];
    const int pb_max = args.pulses_per_batch;
    float4 *prm = smem4;
    int4 *win = reinterpret_cast<int4 *>(smem4 + 2 * pb_max);
    float4 *stage = smem4 + 3 * pb_max;
    const int w = args.w, wh = args.wh;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kRowWarps = kBpTileY / kBpRowsPerThread;          // warps per column group (8)
    const int col = (warp / kRowWarps) * 32 + lane;                  // pixel column inside the tile
    const int row0 = (warp % kRowWarps) * kBpRowsPerThread;          // first of this thread's rows
    const int tile_x = blockIdx.x, tile_y = blockIdx.y, slice = blockIdx.z;
    const int p_begin = args.pulse_begin + slice * args.slice_len;
    const int p_end = min(args.pulse_end, p_begin + args.slice_len);
    // tile centre (float64) and this thread's pixel offsets from it (float32)
    const double cx = args.x0 + ((double)tile_x * kBpTileX + 0.5 * (kBpTileX - 1)) * args.dx;
    const double cy = args.y0 + ((double)tile_y * kBpTileY + 0.5 * (kBpTileY - 1)) * args.dy;
    const float hx = 0.5f * (kBpTileX - 1) * args.dxf, hy = 0.5f * (kBpTileY - 1) * args.dyf;
    const float ox = ((float)col - 0.5f * (kBpTileX - 1)) * args.dxf;
    float oy[kBpRowsPerThread], od2[kBpRowsPerThread];
#pragma unroll
    for (int k = 0; k < kBpRowsPerThread; k++) {
        const int ly = row0 + k;
        oy[k] = ((float)ly - 0.5f * (kBpTileY - 1)) * args.dyf;
        od2[k] = fmaf(ox, ox, oy[k] * oy[k]);
    }
    float acc_re[kBpRowsPerThread], acc_im[kBpRowsPerThread];
#pragma unroll
    for (int k = 0; k < kBpRowsPerThread; k++) acc_re[k] = acc_im[k] = 0.0f;

    // entry e of pulse row p lives at stage_row0 + 16 (p w + e); the address of entry round(qm) + wh
    // is formed from the bit pattern of qm + magic with 32-bit wrap-around
    const unsigned stage_row0 = (unsigned)__cvta_generic_to_shared(stage) + 16u * (unsigned)wh - 16u * kRoundMagicBits;
    const int ns = args.n_samples;

    for (int n0 = p_begin; n0 < p_end; n0 += pb_max) {
        const int pb = min(pb_max, p_end - n0);
        // ---- per-(tile, pulse) reference range in float64, window extent in float32
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
            const double kk = inv_r0d * args.inv_dr;
            const float e = args.dr * (float)inv_r0d;
            float4 pa, pc;
            pa.x = (float)(2.0 * wx * kk);          // each coefficient rounded to float once
            pa.y = (float)(2.0 * wy * kk);
            pa.z = (float)kk;
            pa.w = (float)(qg - o) - 0.5f;
            pc.x = -0.125f * e;
            pc.y = 0.0625f * e * e;
            pc.z = -0.0390625f * e * e * e;
            double t = fma(args.kappa, o + 0.5, args.phase0_turns);
            t -= rint(t);
            pc.w = (float)(6.283185307179586 * t);
            // staged entries: the tile's nearest and farthest pixel ranges (float32 is ample here)
            // bound every pixel's bin; two entries of margin on each side
            const float wxf = (float)wx, wyf = (float)wy, wzf = (float)wz;
            const float nx_ = wxf + fminf(fmaxf(-wxf, -hx), hx), ny_ = wyf + fminf(fmaxf(-wyf, -hy), hy);
            const float fx = fabsf(wxf) + hx, fy = fabsf(wyf) + hy;
            const float rmin = sqrtf(fmaf(nx_, nx_, fmaf(ny_, ny_, wzf * wzf)));
            const float rmax = sqrtf(fmaf(fx, fx, fmaf(fy, fy, wzf * wzf)));
            const float r0f = (float)r0, qc = (float)(qg - o), idr = (float)args.inv_dr;
            int e_lo = (int)floorf(fmaf(rmin - r0f, idr, qc)) - 2 + wh;
            int e_hi = (int)floorf(fmaf(rmax - r0f, idr, qc)) + 2 + wh;
            e_lo = max(e_lo, 0);
            e_hi = min(e_hi, w - 1);
            if (!ok) {
                pa = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                pc = pa;
                e_lo = e_hi = wh;
                atomicOr(args.err, kDevErrGeometry);
            }
            prm[2 * threadIdx.x] = pa;
            prm[2 * threadIdx.x + 1] = pc;
            win[threadIdx.x] = make_int4((int)o, e_lo, e_hi, 0);
        }
        __syncthreads();
        // ---- stage the windows, one warp per pulse row: entry e <-> global bin o + e - wh holds
        // (tau, sigma) of samples v_I, v_{I+1}.  Lane j of a row handles the aligned sample pair
        // (a0 + 2j, a0 + 2j + 1) plus the next sample, which give two consecutive entries.
        if (kPlanar) {
            // polyphase planes: sample I at (I & u_mask) Nr + (I >> u_shift).  Each lane loads one sample;
            // the next one comes from the neighbouring lane (the last lane loads its own).
            for (int p = warp; p < pb; p += kBpThreads / 32) {
                const int4 wv = win[p];
                const float2 *line = args.rc + (int64_t)(n0 + p) * ns;
                const int first = wv.x - wh + wv.y;
                const int count = wv.z - wv.y + 1;
                float4 *row = stage + p * w + wv.y;
                const float im0 = (float)(wv.y - wh) - 0.5f;
                for (int c0 = 0; c0 <= count; c0 += 32) {
                    const int c = c0 + lane;
                    const int I = first + c;
                    float2 v0 = make_float2(0.0f, 0.0f), v1;
                    if (c <= count && I >= 0 && I < ns)
                        v0 = __ldg(line + (I & args.u_mask) * args.n_range + (I >> args.u_shift));
                    v1.x = __shfl_down_sync(0xffffffffu, v0.x, 1);
                    v1.y = __shfl_down_sync(0xffffffffu, v0.y, 1);
                    if (lane == 31) {
                        const int J = I + 1;
                        v1 = (c < count && J >= 0 && J < ns)
                                 ? __ldg(line + (J & args.u_mask) * args.n_range + (J >> args.u_shift))
                                 : make_float2(0.0f, 0.0f);
                    }
                    if (c < count) {
                        const float sr = v1.x - v0.x, si = v1.y - v0.y;
                        const float im = im0 + (float)c;
                        row[c] = make_float4(fmaf(-im, sr, v0.x), fmaf(-im, si, v0.y), sr, si);
                    }
                }
            }
        } else
        for (int p = warp; p < pb; p += kBpThreads / 32) {
            const int4 wv = win[p];
            const float2 *line = args.rc + (int64_t)(n0 + p) * ns;
            const int first = wv.x - wh + wv.y;                 // global bin of entry e_lo
            const int count = wv.z - wv.y + 1;                  // entries to stage
            const int a0 = first & ~1;                          // even, so the pair load is 16-byte aligned
            const int off = first - a0;
            const int npairs = (count + 1 + off) >> 1;
            const bool inside = a0 >= 0 && a0 + 2 * npairs < ns;
            float4 *row = stage + p * w + wv.y;
            float im = (float)(wv.y - wh) - 0.5f + (float)(2 * lane - off);   // (entry - wh) - 1/2
            for (int j = lane; j < npairs; j += 32, im += 64.0f) {
                const int s = a0 + 2 * j;
                float2 va, vb, vc;
                if (inside) {
                    const float4 ab = __ldg(reinterpret_cast<const float4 *>(line + s));
                    va = make_float2(ab.x, ab.y);
                    vb = make_float2(ab.z, ab.w);
                    vc = __ldg(line + s + 2);
                } else {
                    const float2 z = make_float2(0.0f, 0.0f);
                    va = (s >= 0 && s < ns) ? __ldg(line + s) : z;
                    vb = (s + 1 >= 0 && s + 1 < ns) ? __ldg(line + s + 1) : z;
                    vc = (s + 2 >= 0 && s + 2 < ns) ? __ldg(line + s + 2) : z;
                }
                const int c = 2 * j - off;                      // entry of the pair's first sample
                if (c >= 0) {
                    const float sr = vb.x - va.x, si = vb.y - va.y;
                    row[c] = make_float4(fmaf(-im, sr, va.x), fmaf(-im, si, va.y), sr, si);
                }
                if (c + 1 < count) {
                    const float sr = vc.x - vb.x, si = vc.y - vb.y, im1 = im + 1.0f;
                    row[c + 1] = make_float4(fmaf(-im1, sr, vb.x), fmaf(-im1, si, vb.y), sr, si);
                }
            }
        }
        __syncthreads();
        // ---- pixel x pulse inner loop
#pragma unroll 2
        for (int p = 0; p < pb; p++) {
            const float4 pa = prm[2 * p], pc = prm[2 * p + 1];
            const int4 wv = kCheck ? win[p] : make_int4(0, 0, 0, 0);
            const unsigned base = stage_row0 + (unsigned)(p * w) * 16u;
            const float adx = pa.x * ox;
            pixel_pulse<kCheck>(pa, pc, wv, base, adx, oy, od2, acc_re, acc_im, args);
        }
        __syncthreads();
    }
    // ---- store: straight into the image with one slice, else into this slice's partial image
    const int ix = tile_x * kBpTileX + col;
    const bool direct = gridDim.z == 1;
    float2 *out = direct ? args.image : args.partial + (int64_t)slice * args.nx * args.ny;
#pragma unroll
    for (int k = 0; k < kBpRowsPerThread; k++) {
        const int iy = tile_y * kBpTileY + row0 + k;
        if (ix < args.nx && iy < args.ny) {
            float2 *dst = out + (int64_t)iy * args.nx + ix;
            float2 v = make_float2(acc_re[k], acc_im[k]);
            if (direct && args.accumulate) {
                const float2 old = *dst;
                v.x += old.x;
                v.y += old.y;
            }
            *dst = v;
        }
    }
}

// image = (accumulate ? image : 0) + partial_0 + partial_1 + ... in slice order, so the result does
// not depend on which slice finished first
__global__ void bp_reduce_kernel(const float2 *__restrict__ partial, int slices, int64_t npix, float2 *image,
                                 int accumulate)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < npix; i += (int64_t)gridDim.x * blockDim.x) {
        float2 acc = accumulate ? image[i] : make_float2(0.0f, 0.0f);
        for (int s = 0; s < slices; s++) {
            const float2 v = __ldg(partial + s * npix + i);
            acc.x += v.x;
            acc.y += v.y;
        }
        image[i] = acc;
    }
}

}  // namespace

size_t bp_smem_bytes(int w, int pulses_per_batch)
{
    return (size_t)pulses_per_batch * (3 + (size_t)w) * sizeof(float4);
}

cudaError_t bp_configure(int smem_bytes)
{
    const void *fns[] = {(const void *)bp_kernel<false, false>, (const void *)bp_kernel<false, true>,
                         (const void *)bp_kernel<true, false>, (const void *)bp_kernel<true, true>};
    for (const void *f : fns) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

int bp_ctas_per_sm(int smem_bytes)
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, bp_kernel<false, true>, kBpThreads, smem_bytes) != cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}

cudaError_t launch_bp(const BpArgs &a, int slices, bool check_bounds, cudaStream_t s)
{
    if (a.pulse_end <= a.pulse_begin) return cudaSuccess;
    const dim3 grid(a.tiles_x, a.tiles_y, slices);
    const size_t smem = bp_smem_bytes(a.w, a.pulses_per_batch);
    if (check_bounds) {
        if (a.planar) bp_kernel<true, true><<<grid, kBpThreads, smem, s>>>(a);
        else bp_kernel<true, false><<<grid, kBpThreads, smem, s>>>(a);
    } else {
        if (a.planar) bp_kernel<false, true><<<grid, kBpThreads, smem, s>>>(a);
        else bp_kernel<false, false><<<grid, kBpThreads, smem, s>>>(a);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || slices == 1) return e;
    const int64_t npix = (int64_t)a.nx * a.ny;
    const int blocks = (int)((npix + 255) / 256 < 4096 ? (npix + 255) / 256 : 4096);
    bp_reduce_kernel<<<blocks, 256, 0, s>>>(a.partial, slices, npix, a.image, a.accumulate);
    return cudaGetLastError();
}

}  // namespace sar
