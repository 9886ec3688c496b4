// bp_kernel.cu -- time-domain backprojection ("GPU-accelerated backprojection
// SAR imaging", sections 1.1, 2.1-2.3 and 3.3): every pixel sums, over pulses,
// the linearly interpolated range-compressed echo at its range, multiplied by
// exp(+j 4 pi fc R / c0).
//
// Work decomposition.  One CTA owns a tile of 2048 pixels, long in azimuth (x): 128 x 16, 64 x 32
// or 32 x 64 pixels, the longest whose half-diagonal stays within the range-series bound (the plan
// picks it).  Pixels that differ only in x lie at nearly the same range, so the window of
// compressed samples a tile touches grows with its range (y) extent only and staging it is shared
// by more pixels.  Warps run along x, so the 32 lanes of a warp read nearly the same samples; each
// thread keeps eight pixels' complex sums (one column, eight consecutive rows) in registers for
// the whole pulse range.  A prep kernel first evaluates, per (tile, pulse) and in double-float
// arithmetic, the range R0 from the antenna to the tile centre and the parameters derived from
// it; the CTA then walks the pulses in batches, reading those parameters and staging the window
// of compressed samples the tile can touch in shared memory (section 2.3 of the same page stages
// echo data per image block the same way).  Long pulse ranges are split into slices (gridDim.z)
// whose partial images a second kernel adds in slice order, so that small images and the last
// wave still fill the GPU.
//
// Range and phase precision.  At X band the phase 4 pi R / lambda needs R to
// ~1e-5 m at R ~ 6 km, beyond float32 (the listing in section 3.3 computes the
// whole distance in float and loses ~0.1 rad).  Here each pixel's range is a
// float32 offset from the float64 tile-centre range: with d the pixel offset
// from the tile centre, w the antenna-to-centre vector and g = 2 w.d/R0 + |d|^2/R0,
//     R - R0 = g/2 - g^2/(8 R0) + g^3/(16 R0^2) - 5 g^4/(128 R0^3) + O(g^5/R0^4),
// evaluated by Horner's rule in range-bin units (the binomial series of
// R0 sqrt(1 + g/R0)).  |d| <= h (the tile half-diagonal, at most 32 m) and R0 >= 100 h
// keep the truncation below 9e-9 h, 3e-7 m (below 1e-9 m for 16 m tiles at 5.8 km).  The
// quartic term is evaluated only by CTAs whose slice has a (tile, pulse) where it can move the
// phase by 1e-6 rad or more (the prep kernel bounds it); elsewhere it is far below the float32
// rounding of the phase and the loop leaves it out.
//
// Interpolation and phase in one staged pair.  With q the pixel's fractional
// bin relative to the window origin o (half a bin shifted: qm = q - 1/2) and
// i = round(qm) = floor(q), the linear interpolation (1 - f) v_i + f v_{i+1},
// f = q - i, equals tau_i + qm sigma_i with sigma_i = v_{i+1} - v_i and
// tau_i = v_i - (i - 1/2) sigma_i.  The phase is 2 pi [(2/lambda) R_start +
// kappa (o + 1/2)] + 2 pi kappa qm, kappa = 2 dr / lambda, so the per-(tile,
// pulse) part is one angle theta and the per-pixel part one fused multiply-add.
// Per pixel and pulse that leaves: 2 FMA (range offset), 3 FMA (series; 4 with the quartic
// term), 1 add (round), 1 integer op (address), 1 shared 128-bit load, 2 FMA (interp),
// 1 FMA + sin/cos on the SFU (phase), 4 FMA (complex multiply-accumulate); the FMAs and adds of
// two pixel rows go as one paired instruction.
#include <cuda_fp16.h>
#include <cstring>
#include <type_traits>

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

__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }

// entry address = base + 16 * bits, one integer multiply-add (32-bit wrap-around)
__device__ __forceinline__ unsigned entry_addr(unsigned base, float rnd)
{
    unsigned a;
    asm("mad.lo.u32 %0, %1, 16, %2;" : "=r"(a) : "r"(__float_as_uint(rnd)), "r"(base));
    return a;
}

// One pulse's contribution to this thread's pixels, two pixel rows at a time: every per-pixel
// quantity of rows (2j, 2j + 1) is a register pair, so the range offset, the series, the rounding,
// the phase argument and the complex multiply-accumulate each take one paired (FFMA2 / FADD2)
// instruction for both pixels.  q4 points at the pulse's parameters, two float4 loads that every
// lane of the CTA shares: (a, b, c, q0m), (c1, c2, c3, theta); each becomes a pair (x, x) in
// registers (two loads per pulse instead of four of pre-duplicated pairs: measured on GB300,
// 2.961 -> 2.914 ms on the spotlight scene, the compensated variant 3.129 -> 3.004 ms).
template <bool kCheck, bool kQuartic>
__device__ __forceinline__ void pixel_pulse(const float4 *q4, const int4 wv, const unsigned base, const float2 ox2,
                                            const float2 *oyp, const float2 *odp, float2 *acc_r, float2 *acc_i,
                                            const BpArgs &args)
{
    const float4 Q0 = q4[0], Q1 = q4[1];
    const float2 A2 = f2(Q0.x, Q0.x), B2 = f2(Q0.y, Q0.y), C2 = f2(Q0.z, Q0.z), QM2 = f2(Q0.w, Q0.w);
    const float2 S1 = f2(Q1.x, Q1.x), S2 = f2(Q1.y, Q1.y), S3 = f2(Q1.z, Q1.z), TH = f2(Q1.w, Q1.w);
    const float2 half2 = f2(0.5f, 0.5f), magic2 = f2(kRoundMagic, kRoundMagic);
    const float2 tpk2 = f2(args.two_pi_kappa, args.two_pi_kappa);
    const float2 adx2 = __fmul2_rn(A2, ox2);
#pragma unroll
    for (int j = 0; j < kBpRowsPerThread / 2; j++) {
        const float2 g = __ffma2_rn(B2, oyp[j], __ffma2_rn(C2, odp[j], adx2));
        float2 t = kQuartic ? __ffma2_rn(g, __ffma2_rn(g, S3, S2), S1) : __ffma2_rn(g, S2, S1);
        t = __ffma2_rn(g, t, half2);
        const float2 qm = __ffma2_rn(g, t, QM2);
        const float2 rnd = __fadd2_rn(qm, magic2);
        const float2 ph = __ffma2_rn(qm, tpk2, TH);
        if (kCheck) {
            const int e0 = (int)(__float_as_uint(rnd.x) - kRoundMagicBits) + args.wh;
            const int e1 = (int)(__float_as_uint(rnd.y) - kRoundMagicBits) + args.wh;
            if (e0 < wv.y || e0 > wv.z || e1 < wv.y || e1 > wv.z) {
                atomicOr(args.err, kDevErrBounds);
                continue;
            }
        }
        const float4 v0 = lds128(entry_addr(base, rnd.x));
        const float4 v1 = lds128(entry_addr(base, rnd.y));
        const float2 vr = f2(fmaf(qm.x, v0.z, v0.x), fmaf(qm.y, v1.z, v1.x));
        const float2 vi = f2(fmaf(qm.x, v0.w, v0.y), fmaf(qm.y, v1.w, v1.y));
        float2 sn, cs;
        __sincosf(ph.x, &sn.x, &cs.x);
        __sincosf(ph.y, &sn.y, &cs.y);
        acc_r[j] = __ffma2_rn(vr, cs, acc_r[j]);
        acc_r[j] = __ffma2_rn(f2(-vi.x, -vi.y), sn, acc_r[j]);
        acc_i[j] = __ffma2_rn(vr, sn, acc_i[j]);
        acc_i[j] = __ffma2_rn(vi, cs, acc_i[j]);
    }
}

__device__ __forceinline__ uint2 lds64(unsigned addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ float2 half2_bits_to_float2(unsigned bits)
{
    __half2 h;
    memcpy(&h, &bits, sizeof(h));
    return __half22float2(h);
}

// entry address = base + 8 * bits (8-byte entries)
__device__ __forceinline__ unsigned entry_addr8(unsigned base, float rnd)
{
    unsigned a;
    asm("mad.lo.u32 %0, %1, 8, %2;" : "=r"(a) : "r"(__float_as_uint(rnd)), "r"(base));
    return a;
}

// The phase rotation and complex accumulation shared by the variants: acc += (vr + i vi) e^{i ph}.
__device__ __forceinline__ void rotate_accumulate(const float2 vr, const float2 vi, const float2 ph, float2 &acc_r,
                                                  float2 &acc_i)
{
    float2 sn, cs;
    __sincosf(ph.x, &sn.x, &cs.x);
    __sincosf(ph.y, &sn.y, &cs.y);
    acc_r = __ffma2_rn(vr, cs, acc_r);
    acc_r = __ffma2_rn(f2(-vi.x, -vi.y), sn, acc_r);
    acc_i = __ffma2_rn(vr, sn, acc_i);
    acc_i = __ffma2_rn(vi, cs, acc_i);
}

// Float16 entries: (m, s) with m = (v_i + v_{i+1}) / 2 and s = v_{i+1} - v_i as two half2
// (re, im) words.  With r = round(qm), the sample at q = qm + 1/2 is m_r + (qm - r) s_r: the
// interpolation variable stays within [-1/2, 1/2], so no large intercept (the tau of the float32
// entries) loses the float16 precision.  Arithmetic in float32.
template <bool kCheck, bool kQuartic>
__device__ __forceinline__ void pixel_pulse_half(const float4 *q4, const int4 wv, const unsigned base, const float2 ox2,
                                                 const float2 *oyp, const float2 *odp, float2 *acc_r, float2 *acc_i,
                                                 const BpArgs &args)
{
    const float4 Q0 = q4[0], Q1 = q4[1];
    const float2 A2 = f2(Q0.x, Q0.x), B2 = f2(Q0.y, Q0.y), C2 = f2(Q0.z, Q0.z), QM2 = f2(Q0.w, Q0.w);
    const float2 S1 = f2(Q1.x, Q1.x), S2 = f2(Q1.y, Q1.y), S3 = f2(Q1.z, Q1.z), TH = f2(Q1.w, Q1.w);
    const float2 half2v = f2(0.5f, 0.5f), magic2 = f2(kRoundMagic, kRoundMagic);
    const float2 tpk2 = f2(args.two_pi_kappa, args.two_pi_kappa);
    const float2 adx2 = __fmul2_rn(A2, ox2);
#pragma unroll
    for (int j = 0; j < kBpRowsPerThread / 2; j++) {
        const float2 g = __ffma2_rn(B2, oyp[j], __ffma2_rn(C2, odp[j], adx2));
        float2 t = kQuartic ? __ffma2_rn(g, __ffma2_rn(g, S3, S2), S1) : __ffma2_rn(g, S2, S1);
        t = __ffma2_rn(g, t, half2v);
        const float2 qm = __ffma2_rn(g, t, QM2);
        const float2 rnd = __fadd2_rn(qm, magic2);
        const float2 ph = __ffma2_rn(qm, tpk2, TH);
        if (kCheck) {
            const int e0 = (int)(__float_as_uint(rnd.x) - kRoundMagicBits) + args.wh;
            const int e1 = (int)(__float_as_uint(rnd.y) - kRoundMagicBits) + args.wh;
            if (e0 < wv.y || e0 > wv.z || e1 < wv.y || e1 > wv.z) {
                atomicOr(args.err, kDevErrBounds);
                continue;
            }
        }
        const float2 fm = __fadd2_rn(qm, f2(kRoundMagic - rnd.x, kRoundMagic - rnd.y));   // qm - round(qm)
        const uint2 e0 = lds64(entry_addr8(base, rnd.x));
        const uint2 e1 = lds64(entry_addr8(base, rnd.y));
        const float2 m0 = half2_bits_to_float2(e0.x), s0 = half2_bits_to_float2(e0.y);
        const float2 m1 = half2_bits_to_float2(e1.x), s1 = half2_bits_to_float2(e1.y);
        const float2 vr = f2(fmaf(fm.x, s0.x, m0.x), fmaf(fm.y, s1.x, m1.x));
        const float2 vi = f2(fmaf(fm.x, s0.y, m0.y), fmaf(fm.y, s1.y, m1.y));
        rotate_accumulate(vr, vi, ph, acc_r[j], acc_i[j]);
    }
}

// 8-tap sinc interpolation.  With q = qm + 1/2, r = floor(q) and f = q - r, taps k = -3 .. 4 read
// samples r + k with weights proportional to h(f - k), h(d) = sinc(d) (1 + cos(pi d / 4)) / 2 for
// |d| < 4, normalised to unit sum.  Since sin(pi (f - k)) = (-1)^k sin(pi f), the unnormalised
// weights are sin(pi f) / pi * (-1)^k W(f - k) / (f - k); the common factor drops out in the
// normalisation, and so does prod_j (f - j): the weights are proportional to
//     u_k = (-1)^k W(f - k) prod_{j != k} (f - j),
// which stays finite at f = 0 (only u_0 is nonzero there: the sample itself).  The taper W(f - k)
// comes from one sin/cos of pi f / 4 by the angle-sum identity.  Staged entries are float32
// samples; the row holds three samples before the window and four after.
template <bool kCheck, bool kQuartic>
__device__ __forceinline__ void pixel_pulse_sinc(const float4 *q4, const int4 wv, const unsigned base, const float2 ox2,
                                                 const float2 *oyp, const float2 *odp, float2 *acc_r, float2 *acc_i,
                                                 const BpArgs &args)
{
    const float4 Q0 = q4[0], Q1 = q4[1];
    const float2 A2 = f2(Q0.x, Q0.x), B2 = f2(Q0.y, Q0.y), C2 = f2(Q0.z, Q0.z), QM2 = f2(Q0.w, Q0.w);
    const float2 S1 = f2(Q1.x, Q1.x), S2 = f2(Q1.y, Q1.y), S3 = f2(Q1.z, Q1.z), TH = f2(Q1.w, Q1.w);
    const float2 half2v = f2(0.5f, 0.5f), magic2 = f2(kRoundMagic, kRoundMagic);
    const float2 tpk2 = f2(args.two_pi_kappa, args.two_pi_kappa);
    const float2 adx2 = __fmul2_rn(A2, ox2);
    // (-1)^k cos(pi k / 4) / 2, (-1)^k sin(pi k / 4) / 2 and (-1)^k / 2 for k = -3 .. 4
    constexpr float r2 = 0.35355339059327376220f;             // sqrt(2) / 4
    constexpr float kC[8] = {r2, 0.0f, -r2, 0.5f, -r2, 0.0f, r2, -0.5f};
    constexpr float kS[8] = {r2, -0.5f, r2, 0.0f, -r2, 0.5f, -r2, 0.0f};
    constexpr float kH[8] = {-0.5f, 0.5f, -0.5f, 0.5f, -0.5f, 0.5f, -0.5f, 0.5f};
#pragma unroll
    for (int j = 0; j < kBpRowsPerThread / 2; j++) {
        const float2 g = __ffma2_rn(B2, oyp[j], __ffma2_rn(C2, odp[j], adx2));
        float2 t = kQuartic ? __ffma2_rn(g, __ffma2_rn(g, S3, S2), S1) : __ffma2_rn(g, S2, S1);
        t = __ffma2_rn(g, t, half2v);
        const float2 qm = __ffma2_rn(g, t, QM2);
        const float2 rnd = __fadd2_rn(qm, magic2);
        const float2 ph = __ffma2_rn(qm, tpk2, TH);
        if (kCheck) {
            const int e0 = (int)(__float_as_uint(rnd.x) - kRoundMagicBits) + args.wh;
            const int e1 = (int)(__float_as_uint(rnd.y) - kRoundMagicBits) + args.wh;
            if (e0 < wv.y || e0 > wv.z || e1 < wv.y || e1 > wv.z) {
                atomicOr(args.err, kDevErrBounds);
                continue;
            }
        }
        // f = qm + 1/2 - round(qm), in [0, 1]
        const float2 f = __fadd2_rn(__fadd2_rn(qm, f2(kRoundMagic - rnd.x, kRoundMagic - rnd.y)), half2v);
        float2 cq, sq;
        __sincosf(0.78539816339744830962f * f.x, &sq.x, &cq.x);
        __sincosf(0.78539816339744830962f * f.y, &sq.y, &cq.y);
        // d_k = f - k; prefix and suffix products of the d's give prod_{j != k} d_j
        float2 d[8], pre[8];
#pragma unroll
        for (int k = 0; k < 8; k++) d[k] = __fadd2_rn(f, f2((float)(3 - k), (float)(3 - k)));
        pre[0] = f2(1.0f, 1.0f);
#pragma unroll
        for (int k = 1; k < 8; k++) pre[k] = __fmul2_rn(pre[k - 1], d[k - 1]);
        float2 suf = f2(1.0f, 1.0f), u[8], sum = f2(0.0f, 0.0f);
#pragma unroll
        for (int k = 7; k >= 0; k--) {
            const float2 wk = __ffma2_rn(cq, f2(kC[k], kC[k]), __ffma2_rn(sq, f2(kS[k], kS[k]), f2(kH[k], kH[k])));
            u[k] = __fmul2_rn(wk, __fmul2_rn(pre[k], suf));
            suf = __fmul2_rn(suf, d[k]);
            sum = __fadd2_rn(sum, u[k]);
        }
        const unsigned a0 = entry_addr8(base, rnd.x), a1 = entry_addr8(base, rnd.y);
        float2 v0 = f2(0.0f, 0.0f), v1 = f2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const uint2 s0 = lds64(a0 + 8u * (unsigned)(k - 3)), s1 = lds64(a1 + 8u * (unsigned)(k - 3));
            v0 = __ffma2_rn(f2(u[k].x, u[k].x), f2(__uint_as_float(s0.x), __uint_as_float(s0.y)), v0);
            v1 = __ffma2_rn(f2(u[k].y, u[k].y), f2(__uint_as_float(s1.x), __uint_as_float(s1.y)), v1);
        }
        const float n0 = __fdividef(1.0f, sum.x), n1 = __fdividef(1.0f, sum.y);
        rotate_accumulate(f2(v0.x * n0, v1.x * n1), f2(v0.y * n0, v1.y * n1), ph, acc_r[j], acc_i[j]);
    }
}

// ---------------------------------------------------------------------------
// Double-float arithmetic: a value is an unevaluated sum hi + lo of two floats
// with |lo| <= ulp(hi) / 2 (about 48 significant bits).  Error-free
// transformations: Knuth's two-sum, Dekker's fast two-sum (|a| >= |b|) and the
// FMA two-product.  Used for the per-(tile, pulse) reference range, whose phase
// needs ~1e-7 m at ~10 km; float64 runs at a small fraction of the float32 rate
// on this GPU, so the prep stays on the float32 pipe.
// ---------------------------------------------------------------------------
struct dflt {
    float hi, lo;
};
__device__ __forceinline__ dflt df_fast(float a, float b)
{
    const float s = __fadd_rn(a, b);
    return {s, __fadd_rn(b, -__fadd_rn(s, -a))};
}
__device__ __forceinline__ dflt df_two_sum(float a, float b)
{
    const float s = __fadd_rn(a, b);
    const float bb = __fadd_rn(s, -a);
    return {s, __fadd_rn(__fadd_rn(a, -__fadd_rn(s, -bb)), __fadd_rn(b, -bb))};
}
__device__ __forceinline__ dflt df_add(dflt x, dflt y)
{
    const dflt s = df_two_sum(x.hi, y.hi);
    return df_fast(s.hi, __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo)));
}
__device__ __forceinline__ dflt df_neg(dflt x) { return {-x.hi, -x.lo}; }
__device__ __forceinline__ dflt df_mul(dflt x, dflt y)
{
    const float p = __fmul_rn(x.hi, y.hi);
    float e = __fmaf_rn(x.hi, y.hi, -p);
    e = __fmaf_rn(x.hi, y.lo, e);
    e = __fmaf_rn(x.lo, y.hi, e);
    return df_fast(p, e);
}
__device__ __forceinline__ dflt df_mulf(dflt x, float y)
{
    const float p = __fmul_rn(x.hi, y);
    return df_fast(p, __fmaf_rn(x.lo, y, __fmaf_rn(x.hi, y, -p)));
}
// square root: correctly rounded float root refined by one Newton step in double-float
__device__ __forceinline__ dflt df_sqrt(dflt x)
{
    const float s = __fsqrt_rn(x.hi);
    const float p = __fmul_rn(s, s);
    const float r = __fadd_rn(__fadd_rn(__fadd_rn(x.hi, -p), -__fmaf_rn(s, s, -p)), x.lo);
    return df_fast(s, __fmul_rn(r, __fdiv_rn(0.5f, s)));
}
// reciprocal: correctly rounded float reciprocal refined by one Newton step
__device__ __forceinline__ dflt df_rcp(dflt x)
{
    const float y = __frcp_rn(x.hi);
    const dflt e = df_add({1.0f, 0.0f}, df_neg(df_mulf(x, y)));     // 1 - x y
    return df_fast(y, __fmul_rn(y, e.hi));
}
// floor and fraction of a double-float whose hi part is below 2^23
__device__ __forceinline__ float df_floor(dflt x, float &frac)
{
    float fl = floorf(x.hi);
    float fr = __fadd_rn(__fadd_rn(x.hi, -fl), x.lo);                 // x.hi - fl is exact
    if (fr < 0.0f) {
        fl -= 1.0f;
        fr += 1.0f;
    } else if (fr >= 1.0f) {
        fl += 1.0f;
        fr -= 1.0f;
    }
    frac = fr;
    return fl;
}

// A float64 value as a double-float (hi, lo) pair.
__device__ __forceinline__ dflt df_from_double(double v)
{
    const float hi = (float)v;
    return {hi, (float)(v - (double)hi)};
}

// Phase bound (radians) below which the series' quartic term is left out of a (tile, pulse).
constexpr float kBpQuarticPhase = 1.0e-6f;

// Per (tile, pulse) reference range (double-float) and window extent (float32), one thread each.
// Output: pa = (a, b, c, q0m), pc = (c1, c2, c3, theta),
// win = (origin o, first entry, last entry, 1 if the quartic term of the series is needed).
// (ax, ay, az): the pulse's antenna position in double-float.
__device__ __forceinline__ void tile_pulse_params(const BpArgs &args, int tile_x, int tile_y, const dflt ax,
                                                  const dflt ay, const dflt az, float4 &pa, float4 &pc, int4 &win)
{
    const int w = args.w, wh = args.wh;
    // tile centre: x0 + (tile * 64 + 31.5) dx, y0 + (tile * 32 + 15.5) dy (the float multipliers are exact)
    const dflt cx = df_add({args.x0s.x, args.x0s.y},
                           df_mulf({args.dxs.x, args.dxs.y}, (float)tile_x * args.tile_w + 0.5f * (args.tile_w - 1)));
    const dflt cy = df_add({args.y0s.x, args.y0s.y},
                           df_mulf({args.dys.x, args.dys.y}, (float)tile_y * args.tile_h + 0.5f * (args.tile_h - 1)));
    const float hx = 0.5f * (args.tile_w - 1) * args.dxf, hy = 0.5f * (args.tile_h - 1) * args.dyf;
    const dflt wx = df_add(cx, df_neg(ax)), wy = df_add(cy, df_neg(ay)), wz = df_add({args.z0s.x, args.z0s.y}, df_neg(az));
    const dflt r2 = df_add(df_mul(wx, wx), df_add(df_mul(wy, wy), df_mul(wz, wz)));
    const dflt r0 = df_sqrt(r2);
    // fractional global bin of the centre
    const dflt qg = df_mul(df_add(r0, df_neg({args.rss.x, args.rss.y})), {args.idrs.x, args.idrs.y});
    // Validity: finite, far enough for the range expansion (which bounds every pixel's offset
    // inside the staged window), and a representable window origin.  Otherwise flag the plan
    // and zero this pulse's parameters: every pixel then reads entry wh, inside the window.
    const bool ok = (r0.hi >= args.min_range_tiles) && (fabsf(qg.hi) < 4.0e6f);
    float qfrac = 0.0f;
    const float o = ok ? df_floor(qg, qfrac) : 0.0f;
    // coefficients of the range offset in bins: a = 2 wx / (r0 dr), b = 2 wy / (r0 dr), c = 1 / (r0 dr)
    const dflt k = df_mul(df_rcp(r0), {args.idrs.x, args.idrs.y});
    const float e = args.dr * __frcp_rn(r0.hi);
    pa.x = 2.0f * df_mul(wx, k).hi;
    pa.y = 2.0f * df_mul(wy, k).hi;
    pa.z = k.hi;
    pa.w = qfrac - 0.5f;
    pc.x = -0.125f * e;
    pc.y = 0.0625f * e * e;
    pc.z = -0.0390625f * e * e * e;
    // phase of the window origin (o + 1/2): frac((2/lambda) R_start + kappa (o + 1/2)) turns
    float tfrac;
    df_floor(df_add({args.ph0s.x, args.ph0s.y}, df_mulf({args.kps.x, args.kps.y}, o + 0.5f)), tfrac);
    if (tfrac >= 0.5f) tfrac -= 1.0f;
    pc.w = 6.28318530717958648f * tfrac;
    // staged entries: the tile's nearest and farthest pixel ranges (float32 is ample here)
    // bound every pixel's bin; two entries of margin on each side
    const float wxf = wx.hi, wyf = wy.hi, wzf = wz.hi;
    const float nx_ = wxf + fminf(fmaxf(-wxf, -hx), hx), ny_ = wyf + fminf(fmaxf(-wyf, -hy), hy);
    const float fx = fabsf(wxf) + hx, fy = fabsf(wyf) + hy;
    const float rmin = sqrtf(fmaf(nx_, nx_, fmaf(ny_, ny_, wzf * wzf)));
    const float rmax = sqrtf(fmaf(fx, fx, fmaf(fy, fy, wzf * wzf)));
    const float r0f = r0.hi, idr = args.idrs.x;
    int e_lo = (int)floorf(fmaf(rmin - r0f, idr, qfrac)) - 2 + wh;
    int e_hi = (int)floorf(fmaf(rmax - r0f, idr, qfrac)) + 2 + wh;
    e_lo = max(e_lo, 0);
    e_hi = min(e_hi, w - 1);
    // Whether the pixel kernel needs the series' quartic term: over the tile |g| is at most
    // G = |a| hx + |b| hy + c (hx^2 + hy^2), so the term moves a pixel's phase by at most
    // 2 pi kappa |c3| G^4.  Below kBpQuarticPhase it is left out; that is far below the float32
    // rounding of the phase argument (its last place is already 1e-6 rad at 8 rad).
    const float gb = fabsf(pa.x) * hx + fabsf(pa.y) * hy + pa.z * fmaf(hx, hx, hy * hy);
    int quartic = args.two_pi_kappa * fabsf(pc.z) * (gb * gb) * (gb * gb) > kBpQuarticPhase;
    if (!ok) {
        pa = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        pc = pa;
        e_lo = e_hi = wh;
        quartic = 0;
        atomicOr(args.err, kDevErrGeometry);
    }
    win = make_int4((int)o, e_lo, e_hi, quartic);
}

// The parameter table: entry (tile, pulse) at table + 3 (tile_index * pulse_count + pulse - pulse_begin).
// One thread per pulse and group of `group` consecutive tiles (pulses fastest, so that a warp's
// writes of one tile's entries are contiguous): the pulse's float64 position is split into
// double-float once per group (float64 runs at a small fraction of the float32 rate here).  The
// launcher makes groups of up to kBpPrepTiles tiles, fewer when that would leave the GPU short of
// threads (a small image).
constexpr int kBpPrepTiles = 16;

__global__ void __launch_bounds__(256) bp_prep_kernel(BpArgs args, int group)
{
    const int64_t npulses = args.pulse_end - args.pulse_begin;
    const int tiles = args.tiles_x * args.tiles_y;
    const int groups = (tiles + group - 1) / group;
    const int64_t total = npulses * groups;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int g = (int)(i / npulses);
        const int64_t pi = i - (int64_t)g * npulses;
        const double *ap = args.pos + 3 * (args.pulse_begin + pi);
        const dflt ax = df_from_double(__ldg(ap)), ay = df_from_double(__ldg(ap + 1)), az = df_from_double(__ldg(ap + 2));
        const int t_end = min(tiles, (g + 1) * group);
        for (int tile = g * group; tile < t_end; tile++) {
            float4 pa, pc;
            int4 win;
            tile_pulse_params(args, tile % args.tiles_x, tile / args.tiles_x, ax, ay, az, pa, pc, win);
            float4 *dst = args.table + 3 * ((int64_t)tile * npulses + pi);
            dst[0] = pa;
            dst[1] = pc;
            dst[2] = make_float4(__int_as_float(win.x), __int_as_float(win.y), __int_as_float(win.z), 0.0f);
        }
    }
}

// Kahan's compensated summation of x into (s, c), on a pair of independent sums: c carries the
// low-order part the previous additions lost, with the sign that makes s - c the better total.
__device__ __forceinline__ void kahan_add(float2 &s, float2 &c, const float2 x)
{
    const float2 y = __fadd2_rn(x, f2(-c.x, -c.y));
    const float2 t = __fadd2_rn(s, y);
    c = __fadd2_rn(__fadd2_rn(t, f2(-s.x, -s.y)), f2(-y.x, -y.y));
    s = t;
}

__device__ __forceinline__ void cp_async8(unsigned dst, const void *src, int src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async16(unsigned dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Shared memory of one CTA:
//   params [3][pulses_per_batch][2] float4 parameters (see pixel_pulse) and
//          [3][pulses_per_batch] int4 windows (origin o, first and last staged entry) -- for the
//          current batch and the next two;
//   raw    [batch][rw] float2 -- the next batch's compressed samples, gathered by
//          asynchronous copies while the current batch is computed;
//   stage  [pulses_per_batch][w] float4 -- the current batch's (tau, sigma) entries.
// Per batch: issue the copies for batch b+1, prefetch the parameters of batch b+2, run the pixel
// loop of batch b, then (one barrier later) turn the raw samples of b+1 into (tau, sigma) entries.
template <int kTileX, bool kCheck, bool kPlanar, int kMode>
__global__ void __launch_bounds__(kBpThreads, bp_mode_ctas(kMode)) bp_kernel(BpArgs args)
{
    constexpr int kTileY = kBpThreads * kBpRowsPerThread / kTileX;
    // staged entry: (tau, sigma) float4, (m, s) half2 pair, or one float32 sample (sinc rows hold
    // three samples before the window and four after)
    constexpr bool kSinc = kMode == kBpSinc8;
    constexpr unsigned kEb = (kMode == kBpHalfStage || kSinc) ? 8u : 16u;
    constexpr int kTapsBefore = kSinc ? 3 : 0;
    constexpr int kPulseUnroll = kMode == kBpLinear ? 8 : 4;           // pulses per unrolled loop step
    constexpr int kExtra = kSinc ? 7 : 1;                       // raw samples per row beyond its entries
    extern __shared__ float4 smem4[];
    constexpr int kWarps = kBpThreads / 32;
    const int pb_cap = args.pulses_per_batch;                                 // parameter slots per batch
    const int wh = args.wh;
    float4 *quads = smem4;                                                   // [3][pb_cap][2]
    int4 *wins = reinterpret_cast<int4 *>(smem4 + 6 * pb_cap);               // [3][pb_cap]
    float4 *dyn = smem4 + kBpParamSlots * pb_cap;                            // raw rows, then stage rows
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kRowWarps = kTileY / kBpRowsPerThread;            // warps per column group
    const int col = (warp / kRowWarps) * 32 + lane;                  // pixel column inside the tile
    const int row0 = (warp % kRowWarps) * kBpRowsPerThread;          // first of this thread's rows
    const int tile_x = blockIdx.x, tile_y = blockIdx.y, slice = blockIdx.z;
    const int p_begin = args.pulse_begin + slice * args.slice_len;
    const int p_end = min(args.pulse_end, p_begin + args.slice_len);
    // this thread's pixel offsets from the tile centre (float32), rows paired (2j, 2j + 1)
    const float ox = ((float)col - 0.5f * (kTileX - 1)) * args.dxf;
    const float2 ox2 = f2(ox, ox);
    float2 oyp[kBpRowsPerThread / 2], odp[kBpRowsPerThread / 2];
#pragma unroll
    for (int j = 0; j < kBpRowsPerThread / 2; j++) {
        const float y0 = ((float)(row0 + 2 * j) - 0.5f * (kTileY - 1)) * args.dyf;
        const float y1 = ((float)(row0 + 2 * j + 1) - 0.5f * (kTileY - 1)) * args.dyf;
        oyp[j] = f2(y0, y1);
        odp[j] = f2(fmaf(ox, ox, y0 * y0), fmaf(ox, ox, y1 * y1));
    }
    // complex sums of rows (2j, 2j + 1): real parts and imaginary parts
    float2 acc_r[kBpRowsPerThread / 2], acc_i[kBpRowsPerThread / 2];
#pragma unroll
    for (int j = 0; j < kBpRowsPerThread / 2; j++) acc_r[j] = acc_i[j] = f2(0.0f, 0.0f);
    // compensated variant: the batch sums above are folded after every batch into Kahan totals
    // (sum, compensation), so rounding grows with the batch length, not the pulse count
    float2 tot_r[kBpRowsPerThread / 2], tot_i[kBpRowsPerThread / 2], cmp_r[kBpRowsPerThread / 2],
        cmp_i[kBpRowsPerThread / 2];
#pragma unroll
    for (int j = 0; j < kBpRowsPerThread / 2; j++) tot_r[j] = tot_i[j] = cmp_r[j] = cmp_i[j] = f2(0.0f, 0.0f);

    const int ns = args.n_samples;
    // this tile's rows of the parameter table, indexed by pulse - pulse_begin
    const int64_t npulses = args.pulse_end - args.pulse_begin;
    const float4 *tab = args.table + 3 * (((int64_t)tile_y * args.tiles_x + tile_x) * npulses - args.pulse_begin);

    // Row sizes from the windows this CTA will actually stage (at most the diagonal bound w): the
    // widest window of the slice sets the stage row stride, and as many pulses as fit the shared
    // memory make a batch.
    // The same scan finds whether any pulse of the slice needs the series' quartic term (the
    // window's fourth word, set by the parameter kernel).
    __shared__ int s_extent, s_quartic;
    if (threadIdx.x == 0) {
        s_extent = 1;
        s_quartic = 0;
    }
    __syncthreads();
    {
        int m = 1, need = 0;
        for (int n = p_begin + (int)threadIdx.x; n < p_end; n += kBpThreads) {
            const float4 wf = __ldg(tab + 3 * (int64_t)n + 2);
            m = max(m, __float_as_int(wf.z) - __float_as_int(wf.y) + 1);
            need |= __float_as_int(wf.w);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        need = __any_sync(0xffffffffu, need != 0);
        if (lane == 0) {
            atomicMax(&s_extent, m);
            if (need) atomicOr(&s_quartic, 1);
        }
    }
    __syncthreads();
    const bool quartic = s_quartic != 0;
    const int stride = min(s_extent, args.w);                                // window entries per row
    const int row_n = kSinc ? ((stride + kExtra + 1) & ~1) : stride;        // stage entries per row
    const int rw = (stride + kExtra + 2) & ~1;                               // raw samples per row (even)
    const int pb_max = max(1, min(pb_cap, args.stage_bytes / (row_n * (int)kEb + rw * 8)));
    float2 *raw = reinterpret_cast<float2 *>(dyn);                           // [pb_max][rw]
    char *stage = reinterpret_cast<char *>(dyn) + (size_t)pb_max * rw * 8;   // [pb_max][row_n] entries

    // entry e of pulse row p lives at stage + p row_n + e - e_lo(p) + kTapsBefore (e_lo = win.y), and
    // the address of entry round(qm) + wh is formed from the bit pattern of qm + magic with 32-bit
    // wrap-around
    const unsigned stage_row0 = (unsigned)__cvta_generic_to_shared(stage) + kEb * (unsigned)wh - kEb * kRoundMagicBits;
    const unsigned raw_base = (unsigned)__cvta_generic_to_shared(raw);

    // asynchronous gather of batch rows [0, count) starting at pulse n into raw: sample j of row p is
    // the line's sample o - wh + e_lo + j (zero outside the line)
    auto issue_raw = [&](int n, int count, const int4 *win) {
        for (int p = warp; p < count; p += kWarps) {
            const int4 wv = win[p];
            const int first = wv.x - wh + wv.y - kTapsBefore;
            const int nsamp = min(wv.z - wv.y + 1 + kExtra, rw);        // never past the row
            const float2 *line = args.rc + (int64_t)(n + p) * ns;
            const unsigned dst = raw_base + (unsigned)(p * rw) * 8u;
            for (int j = lane; j < nsamp; j += 32) {
                const int I = first + j;
                const bool ok = I >= 0 && I < ns;
                const int off = kPlanar ? (I & args.u_mask) * args.n_range + (I >> args.u_shift) : I;
                cp_async8(dst + 8u * (unsigned)j, ok ? (const void *)(line + off) : (const void *)line, ok ? 8 : 0);
            }
        }
        cp_async_commit();
    };
    // raw samples -> staged entries: (tau, sigma) float4, (m, s) float16 pairs, or the samples
    // themselves (sinc); pulse n + p of the batch weighted by args.weights[n + p] when the plan has
    // pulse weights
    auto transform = [&](int n, int count, const int4 *win) {
        for (int p = warp; p < count; p += kWarps) {
            const int4 wv = win[p];
            const int e_lo = wv.y;
            const int nent = min(wv.z - e_lo + 1, stride);                  // stays inside both rows
            const float2 *rr = raw + p * rw;
            const float wgt = args.weights ? __ldg(args.weights + n + p) : 1.0f;
            if constexpr (kSinc) {
                float2 *row = reinterpret_cast<float2 *>(stage) + p * row_n;
                for (int c = lane; c < nent + kExtra; c += 32) {
                    const float2 v = rr[c];
                    row[c] = make_float2(wgt * v.x, wgt * v.y);
                }
            } else if constexpr (kMode == kBpHalfStage) {
                uint2 *row = reinterpret_cast<uint2 *>(stage) + p * row_n;
                for (int c = lane; c < nent; c += 32) {
                    const float2 v0 = rr[c], v1 = rr[c + 1];
                    const __half2 m = __floats2half2_rn(wgt * 0.5f * (v0.x + v1.x), wgt * 0.5f * (v0.y + v1.y));
                    const __half2 d = __floats2half2_rn(wgt * (v1.x - v0.x), wgt * (v1.y - v0.y));
                    uint2 e;
                    memcpy(&e.x, &m, 4);
                    memcpy(&e.y, &d, 4);
                    row[c] = e;
                }
            } else {
                float4 *row = reinterpret_cast<float4 *>(stage) + p * row_n;
                const float im0 = (float)(e_lo - wh) - 0.5f;
                for (int c = lane; c < nent; c += 32) {
                    const float2 v0 = rr[c], v1 = rr[c + 1];
                    const float sr = v1.x - v0.x, si = v1.y - v0.y;
                    const float im = im0 + (float)c;
                    row[c] = args.weights ? make_float4(wgt * fmaf(-im, sr, v0.x), wgt * fmaf(-im, si, v0.y), wgt * sr, wgt * si)
                                          : make_float4(fmaf(-im, sr, v0.x), fmaf(-im, si, v0.y), sr, si);
                }
            }
        }
    };
    // one pulse's table entry -> its two parameter slots and its window (the entry's words as they
    // are: the window's integers travel as float bit patterns)
    auto put_params = [&](int p, const float4 pa, const float4 pc, const float4 wf, float4 *quad, int4 *win) {
        quad[2 * p] = pa;
        quad[2 * p + 1] = pc;
        win[p] = make_int4(__float_as_int(wf.x), __float_as_int(wf.y), __float_as_int(wf.z), __float_as_int(wf.w));
    };
    auto load_params = [&](int n, int count, float4 *quad, int4 *win) {
        if ((int)threadIdx.x < count) {
            const float4 *src = tab + 3 * (int64_t)(n + threadIdx.x);
            put_params(threadIdx.x, __ldg(src), __ldg(src + 1), __ldg(src + 2), quad, win);
        }
    };

    // prologue: parameters of the first two batches, then the first batch's windows
    int pb = max(0, min(pb_max, p_end - p_begin));
    int pb1 = max(0, min(pb_max, p_end - (p_begin + pb)));
    load_params(p_begin, pb, quads, wins);
    load_params(p_begin + pb, pb1, quads + 2 * pb_cap, wins + pb_cap);
    __syncthreads();
    if (pb > 0) issue_raw(p_begin, pb, wins);
    cp_async_wait_all();
    __syncthreads();
    if (pb > 0) transform(p_begin, pb, wins);
    __syncthreads();

    int buf = 0;
    for (int n0 = p_begin; n0 < p_end; buf = (buf == 2) ? 0 : buf + 1) {
        const int buf1 = (buf == 2) ? 0 : buf + 1, buf2 = (buf1 == 2) ? 0 : buf1 + 1;
        const float4 *quad = quads + 2 * pb_cap * buf;
        const int4 *win = wins + pb_cap * buf;
        const int n1 = n0 + pb, n2 = n1 + pb1;
        const int pb2 = max(0, min(pb_max, p_end - n2));
        // the next batch's samples, copied while this batch is computed
        if (pb1 > 0) issue_raw(n1, pb1, wins + pb_cap * buf1);
        // the batch after next: its table entries copied into their slots while this batch is
        // computed (no registers held across the pixel loop)
        if ((int)threadIdx.x < pb2) {
            const float4 *src = tab + 3 * (int64_t)(n2 + threadIdx.x);
            const unsigned q = (unsigned)__cvta_generic_to_shared(quads + 2 * pb_cap * buf2 + 2 * threadIdx.x);
            cp_async16(q, src);
            cp_async16(q + 16u, src + 1);
            cp_async16((unsigned)__cvta_generic_to_shared(wins + pb_cap * buf2 + threadIdx.x), src + 2);
        }
        cp_async_commit();
        // ---- pixel x pulse inner loop, in the form with or without the series' quartic term for the
        // whole slice.  Eight pulses unrolled in the default variant, four in the others (measured on
        // GB300, spotlight scene: pixel kernel 2.720 ms with four, 2.691 with eight, 2.830 with
        // twelve, 2.762 with sixteen, curved-track scene 43.31 ms with four and 42.46 with eight;
        // whole backprojection calls, four against eight: compensated 2.916 against 2.947 ms,
        // float16 stage 3.538 against 3.551 ms; sinc, four against two and one: 13.157 against
        // 13.176 and 13.218 ms)
        auto pulse_loop = [&](auto tag) {
            constexpr bool kQ = decltype(tag)::value;
#pragma unroll(kPulseUnroll)
            for (int p = 0; p < pb; p++) {
                const int4 wv = win[p];
                const unsigned base = stage_row0 + (unsigned)(p * row_n - wv.y + kTapsBefore) * kEb;
                if constexpr (kSinc) pixel_pulse_sinc<kCheck, kQ>(quad + 2 * p, wv, base, ox2, oyp, odp, acc_r, acc_i, args);
                else if constexpr (kMode == kBpHalfStage)
                    pixel_pulse_half<kCheck, kQ>(quad + 2 * p, wv, base, ox2, oyp, odp, acc_r, acc_i, args);
                else pixel_pulse<kCheck, kQ>(quad + 2 * p, wv, base, ox2, oyp, odp, acc_r, acc_i, args);
            }
        };
        if (quartic) pulse_loop(std::true_type{});
        else pulse_loop(std::false_type{});
        if constexpr (kMode == kBpCompensated) {
#pragma unroll
            for (int j = 0; j < kBpRowsPerThread / 2; j++) {
                kahan_add(tot_r[j], cmp_r[j], acc_r[j]);
                kahan_add(tot_i[j], cmp_i[j], acc_i[j]);
                acc_r[j] = acc_i[j] = f2(0.0f, 0.0f);
            }
        }
        cp_async_wait_all();
        __syncthreads();
        if (pb1 > 0) transform(n1, pb1, wins + pb_cap * buf1);
        __syncthreads();
        n0 = n1;
        pb = pb1;
        pb1 = pb2;
    }
    // ---- store: straight into the image with one slice, else into this slice's partial image
    const int ix = tile_x * kTileX + col;
    const bool direct = gridDim.z == 1;
    float2 *out = direct ? args.image : args.partial + (int64_t)slice * args.nx * args.ny;
#pragma unroll
    for (int k = 0; k < kBpRowsPerThread; k++) {
        const int iy = tile_y * kTileY + row0 + k;
        if (ix < args.nx && iy < args.ny) {
            float2 *dst = out + (int64_t)iy * args.nx + ix;
            float2 v = (k & 1) ? make_float2(acc_r[k / 2].y, acc_i[k / 2].y) : make_float2(acc_r[k / 2].x, acc_i[k / 2].x);
            if constexpr (kMode == kBpCompensated) {
                // the total less its running compensation (the low part the last additions lost)
                v = (k & 1) ? make_float2(tot_r[k / 2].y - cmp_r[k / 2].y, tot_i[k / 2].y - cmp_i[k / 2].y)
                            : make_float2(tot_r[k / 2].x - cmp_r[k / 2].x, tot_i[k / 2].x - cmp_i[k / 2].x);
            }
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

size_t bp_smem_bytes(const BpArgs &a)
{
    return (size_t)kBpParamSlots * a.pulses_per_batch * sizeof(float4) + (size_t)a.stage_bytes;
}

template <int TX, int M>
cudaError_t bp_configure_mode(int smem_bytes)
{
    const void *fns[] = {(const void *)bp_kernel<TX, false, false, M>, (const void *)bp_kernel<TX, false, true, M>,
                         (const void *)bp_kernel<TX, true, false, M>, (const void *)bp_kernel<TX, true, true, M>};
    for (const void *f : fns) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int TX>
cudaError_t bp_configure_shape(int smem_bytes)
{
    cudaError_t e = bp_configure_mode<TX, kBpLinear>(smem_bytes);
    if (e == cudaSuccess) e = bp_configure_mode<TX, kBpCompensated>(smem_bytes);
    if (e == cudaSuccess) e = bp_configure_mode<TX, kBpHalfStage>(smem_bytes);
    if (e == cudaSuccess) e = bp_configure_mode<TX, kBpSinc8>(smem_bytes);
    return e;
}

cudaError_t bp_configure(int smem_bytes)
{
    cudaError_t e = bp_configure_shape<128>(smem_bytes);
    if (e == cudaSuccess) e = bp_configure_shape<64>(smem_bytes);
    if (e == cudaSuccess) e = bp_configure_shape<32>(smem_bytes);
    return e;
}

template <int TX, int M>
void launch_bp_mode(const BpArgs &a, dim3 grid, size_t smem, bool check_bounds, cudaStream_t s)
{
    if (check_bounds) {
        if (a.planar) bp_kernel<TX, true, true, M><<<grid, kBpThreads, smem, s>>>(a);
        else bp_kernel<TX, true, false, M><<<grid, kBpThreads, smem, s>>>(a);
    } else {
        if (a.planar) bp_kernel<TX, false, true, M><<<grid, kBpThreads, smem, s>>>(a);
        else bp_kernel<TX, false, false, M><<<grid, kBpThreads, smem, s>>>(a);
    }
}

template <int TX>
void launch_bp_shape(const BpArgs &a, dim3 grid, size_t smem, bool check_bounds, cudaStream_t s)
{
    switch (a.mode) {
    case kBpCompensated: launch_bp_mode<TX, kBpCompensated>(a, grid, smem, check_bounds, s); break;
    case kBpHalfStage: launch_bp_mode<TX, kBpHalfStage>(a, grid, smem, check_bounds, s); break;
    case kBpSinc8: launch_bp_mode<TX, kBpSinc8>(a, grid, smem, check_bounds, s); break;
    default: launch_bp_mode<TX, kBpLinear>(a, grid, smem, check_bounds, s); break;
    }
}

int bp_ctas_per_sm(int smem_bytes, int mode)
{
    int n = 0;
    const void *f = mode == kBpCompensated ? (const void *)bp_kernel<128, false, true, kBpCompensated>
                    : mode == kBpHalfStage ? (const void *)bp_kernel<128, false, true, kBpHalfStage>
                    : mode == kBpSinc8     ? (const void *)bp_kernel<128, false, true, kBpSinc8>
                                           : (const void *)bp_kernel<128, false, true, kBpLinear>;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, kBpThreads, smem_bytes) != cudaSuccess) return 1;
    return n > 0 ? n : 1;
}

cudaError_t launch_bp(const BpArgs &a, int slices, bool check_bounds, cudaStream_t s, cudaEvent_t main_begin,
                      cudaEvent_t main_end, cudaEvent_t image_wait, cudaEvent_t image_done)
{
    if (a.pulse_end <= a.pulse_begin) return cudaSuccess;
    const int npulse = a.pulse_end - a.pulse_begin;
    const int64_t tiles = (int64_t)a.tiles_x * a.tiles_y;
    // tiles per thread: up to kBpPrepTiles while that still leaves ~1024 threads per SM
    const int64_t per_thread = (tiles * npulse + 155647) / 155648;
    const int group = (int)(per_thread < 1 ? 1 : per_thread > kBpPrepTiles ? kBpPrepTiles : per_thread);
    const int64_t groups = (tiles + group - 1) / group;
    const int64_t prep_blocks = ((int64_t)npulse * groups + 255) / 256;
    bp_prep_kernel<<<(unsigned)(prep_blocks < (1 << 20) ? prep_blocks : (1 << 20)), 256, 0, s>>>(a, group);
    cudaError_t pe = cudaGetLastError();
    if (pe != cudaSuccess) return pe;
    const dim3 grid(a.tiles_x, a.tiles_y, slices);
    const size_t smem = bp_smem_bytes(a);
    if (slices == 1 && image_wait && (pe = cudaStreamWaitEvent(s, image_wait, 0)) != cudaSuccess) return pe;
    if (main_begin && (pe = cudaEventRecord(main_begin, s)) != cudaSuccess) return pe;
    if (a.tile_w == 128) launch_bp_shape<128>(a, grid, smem, check_bounds, s);
    else if (a.tile_w == 64) launch_bp_shape<64>(a, grid, smem, check_bounds, s);
    else launch_bp_shape<32>(a, grid, smem, check_bounds, s);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && main_end) e = cudaEventRecord(main_end, s);
    if (e == cudaSuccess && slices > 1) {
        const int64_t npix = (int64_t)a.nx * a.ny;
        const int blocks = (int)((npix + 255) / 256 < 4096 ? (npix + 255) / 256 : 4096);
        if (image_wait) e = cudaStreamWaitEvent(s, image_wait, 0);
        if (e == cudaSuccess) {
            bp_reduce_kernel<<<blocks, 256, 0, s>>>(a.partial, slices, npix, a.image, a.accumulate);
            e = cudaGetLastError();
        }
    }
    if (e == cudaSuccess && image_done) e = cudaEventRecord(image_done, s);
    return e;
}

}  // namespace sar
