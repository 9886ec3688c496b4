// fft_reg.cuh -- on-chip DFT building blocks shared by the range-compression and
// range-Doppler kernels: complex helpers, small radix-R DFTs in registers, the
// register-resident power-of-two Stockham transform (16 elements per thread,
// exchanges through padded shared memory), and line staging by bulk copy with a
// bounded mbarrier wait.  Everything here is device code with internal linkage;
// each translation unit that includes it gets its own copy.
#pragma once

#include "sar_internal.cuh"

namespace sar {
namespace {

// Complex sums as one paired instruction (FADD2) for the power-of-two butterflies, where it cut the
// transforms' issue slots (measured on GB300: 4096-point lines without upsampling 0.076 -> 0.070 ms,
// bit-identical results), and as two scalar adds for radices 3, 5, 6 and 10 (paired, the 6000-point
// kernel got 3% slower).
__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 csub(float2 a, float2 b) { return __fadd2_rn(a, make_float2(-b.x, -b.y)); }
__device__ __forceinline__ float2 cadd1(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 csub1(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }
__device__ __forceinline__ float2 cmul(float2 a, float2 b)
{
    return make_float2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.x, b.y, a.y * b.x));
}
__device__ __forceinline__ float2 cconj(float2 a) { return make_float2(a.x, -a.y); }
__device__ __forceinline__ float2 mul_minus_i(float2 a) { return make_float2(a.y, -a.x); }   // -i a
__device__ __forceinline__ float2 mul_plus_i(float2 a) { return make_float2(-a.y, a.x); }    // +i a
// -i a for a forward DFT, +i a for an inverse one
template <bool kInv>
__device__ __forceinline__ float2 mul_mi(float2 a) { return kInv ? mul_plus_i(a) : mul_minus_i(a); }
// a times w for a forward DFT, a times conj(w) for an inverse one
template <bool kInv>
__device__ __forceinline__ float2 cmul_c(float2 a, float wr, float wi) { return cmul(a, make_float2(wr, kInv ? -wi : wi)); }
__device__ __forceinline__ float2 cscale(float2 a, float s) { return make_float2(a.x * s, a.y * s); }

// DFTs of small sizes, in registers: y_k = sum_j a_j exp(-2 pi i j k / R) (forward), or with
// exp(+2 pi i j k / R) for kInv (radices 2, 4, 8 and 16; every constant conjugated, so that the
// inverse of a equals conj(forward(conj(a))) bit for bit).
template <int R, bool kInv = false> struct Dft;

template <bool kInv> struct Dft<2, kInv> {
    static __device__ __forceinline__ void run(float2 *a)
    {
        float2 t = a[0];
        a[0] = cadd(t, a[1]);
        a[1] = csub(t, a[1]);
    }
};

template <> struct Dft<3, false> {
    static __device__ __forceinline__ void run(float2 *a)
    {
        const float s = 0.86602540378443864676f;   // sin(2 pi / 3)
        float2 b = cadd1(a[1], a[2]);
        float2 d = csub1(a[1], a[2]);
        float2 t = make_float2(a[0].x - 0.5f * b.x, a[0].y - 0.5f * b.y);
        float2 v = mul_minus_i(cscale(d, s));
        a[0] = cadd1(a[0], b);
        a[1] = cadd1(t, v);
        a[2] = csub1(t, v);
    }
};

template <bool kInv> struct Dft<4, kInv> {
    static __device__ __forceinline__ void run(float2 *a)
    {
        float2 s02 = cadd(a[0], a[2]), d02 = csub(a[0], a[2]);
        float2 s13 = cadd(a[1], a[3]), d13 = mul_mi<kInv>(csub(a[1], a[3]));
        a[0] = cadd(s02, s13);
        a[2] = csub(s02, s13);
        a[1] = cadd(d02, d13);
        a[3] = csub(d02, d13);
    }
};

template <> struct Dft<5, false> {
    static __device__ __forceinline__ void run(float2 *a)
    {
        const float c1 = 0.30901699437494742410f;    // cos(2 pi / 5)
        const float c2 = -0.80901699437494742410f;   // cos(4 pi / 5)
        const float s1 = 0.95105651629515357212f;    // sin(2 pi / 5)
        const float s2 = 0.58778525229247312917f;    // sin(4 pi / 5)
        float2 b1 = cadd1(a[1], a[4]), d1 = csub1(a[1], a[4]);
        float2 b2 = cadd1(a[2], a[3]), d2 = csub1(a[2], a[3]);
        float2 t1 = make_float2(fmaf(c1, b1.x, fmaf(c2, b2.x, a[0].x)), fmaf(c1, b1.y, fmaf(c2, b2.y, a[0].y)));
        float2 t2 = make_float2(fmaf(c2, b1.x, fmaf(c1, b2.x, a[0].x)), fmaf(c2, b1.y, fmaf(c1, b2.y, a[0].y)));
        float2 u1 = make_float2(fmaf(s1, d1.x, s2 * d2.x), fmaf(s1, d1.y, s2 * d2.y));
        float2 u2 = make_float2(fmaf(s2, d1.x, -s1 * d2.x), fmaf(s2, d1.y, -s1 * d2.y));
        u1 = mul_minus_i(u1);
        u2 = mul_minus_i(u2);
        a[0] = cadd1(a[0], cadd1(b1, b2));
        a[1] = cadd1(t1, u1);
        a[4] = csub1(t1, u1);
        a[2] = cadd1(t2, u2);
        a[3] = csub1(t2, u2);
    }
};

// 6 = 2 x 3 and 10 = 2 x 5: DFTs of the even and the odd samples, the odd ones turned by
// exp(-2 pi i k / R), then sums and differences.
template <> struct Dft<6, false> {
    static __device__ __forceinline__ void run(float2 *a)
    {
        const float h = 0.86602540378443864676f;    // sin(2 pi / 6)
        float2 e[3] = {a[0], a[2], a[4]};
        float2 o[3] = {a[1], a[3], a[5]};
        Dft<3>::run(e);
        Dft<3>::run(o);
        o[1] = cmul(o[1], make_float2(0.5f, -h));
        o[2] = cmul(o[2], make_float2(-0.5f, -h));
#pragma unroll
        for (int k = 0; k < 3; k++) {
            a[k] = cadd1(e[k], o[k]);
            a[k + 3] = csub1(e[k], o[k]);
        }
    }
};

template <> struct Dft<10, false> {
    static __device__ __forceinline__ void run(float2 *a)
    {
        const float c1 = 0.80901699437494742410f, s1 = 0.58778525229247312917f;   // 2 pi / 10
        const float c2 = 0.30901699437494742410f, s2 = 0.95105651629515357212f;   // 4 pi / 10
        float2 e[5] = {a[0], a[2], a[4], a[6], a[8]};
        float2 o[5] = {a[1], a[3], a[5], a[7], a[9]};
        Dft<5>::run(e);
        Dft<5>::run(o);
        o[1] = cmul(o[1], make_float2(c1, -s1));
        o[2] = cmul(o[2], make_float2(c2, -s2));
        o[3] = cmul(o[3], make_float2(-c2, -s2));
        o[4] = cmul(o[4], make_float2(-c1, -s1));
#pragma unroll
        for (int k = 0; k < 5; k++) {
            a[k] = cadd1(e[k], o[k]);
            a[k + 5] = csub1(e[k], o[k]);
        }
    }
};

template <bool kInv> struct Dft<8, kInv> {
    static __device__ __forceinline__ void run(float2 *a)
    {
        const float r = 0.70710678118654752440f;
        float2 e[4] = {a[0], a[2], a[4], a[6]};
        float2 o[4] = {a[1], a[3], a[5], a[7]};
        Dft<4, kInv>::run(e);
        Dft<4, kInv>::run(o);
        // o_k *= exp(-2 pi i k / 8), or exp(+2 pi i k / 8)
        if constexpr (kInv) {
            o[1] = make_float2(r * (o[1].x - o[1].y), r * (o[1].y + o[1].x));
            o[3] = make_float2(-r * (o[3].x + o[3].y), r * (o[3].x - o[3].y));
        } else {
            o[1] = make_float2(r * (o[1].x + o[1].y), r * (o[1].y - o[1].x));
            o[3] = make_float2(r * (o[3].y - o[3].x), -r * (o[3].x + o[3].y));
        }
        o[2] = mul_mi<kInv>(o[2]);
#pragma unroll
        for (int k = 0; k < 4; k++) {
            a[k] = cadd(e[k], o[k]);
            a[k + 4] = csub(e[k], o[k]);
        }
    }
};

template <bool kInv> struct Dft<16, kInv> {
    static __device__ __forceinline__ void run(float2 *a)
    {
        // n = 4 n1 + n2, k = k1 + 4 k2: inner DFT4 over n1, twiddle w16^(n2 k1), outer DFT4 over n2
        float2 b[4][4];
#pragma unroll
        for (int n2 = 0; n2 < 4; n2++) {
            float2 t[4] = {a[n2], a[4 + n2], a[8 + n2], a[12 + n2]};
            Dft<4, kInv>::run(t);
#pragma unroll
            for (int k1 = 0; k1 < 4; k1++) b[n2][k1] = t[k1];
        }
        const float c = 0.92387953251128675613f, s = 0.38268343236508977173f, r = 0.70710678118654752440f;
        // w16^m = exp(-2 pi i m / 16) for m = n2 * k1 (conjugated for the inverse)
        b[1][1] = cmul_c<kInv>(b[1][1], c, -s);
        b[1][2] = cmul_c<kInv>(b[1][2], r, -r);
        b[1][3] = cmul_c<kInv>(b[1][3], s, -c);
        b[2][1] = cmul_c<kInv>(b[2][1], r, -r);
        b[2][2] = mul_mi<kInv>(b[2][2]);
        b[2][3] = cmul_c<kInv>(b[2][3], -r, -r);
        b[3][1] = cmul_c<kInv>(b[3][1], s, -c);
        b[3][2] = cmul_c<kInv>(b[3][2], -r, -r);
        b[3][3] = cmul_c<kInv>(b[3][3], -c, s);
#pragma unroll
        for (int k1 = 0; k1 < 4; k1++) {
            float2 t[4] = {b[0][k1], b[1][k1], b[2][k1], b[3][k1]};
            Dft<4, kInv>::run(t);
#pragma unroll
            for (int k2 = 0; k2 < 4; k2++) a[k1 + 4 * k2] = t[k2];
        }
    }
};

// 32 = 2 x 16: DFT16 of the even and of the odd samples, the odd ones turned by exp(-2 pi i k / 32),
// then sums and differences (forward only; the 8192-point line kernel inverts by the conjugate
// identity).
template <> struct Dft<32, false> {
    static __device__ __forceinline__ void run(float2 *a)
    {
        // cos and sin of 2 pi k / 32, k = 0 .. 8
        constexpr float c[9] = {1.0f, 0.98078528040323044913f, 0.92387953251128675613f, 0.83146961230254523708f,
                                0.70710678118654752440f, 0.55557023301960222474f, 0.38268343236508977173f,
                                0.19509032201612826785f, 0.0f};
        float2 e[16], o[16];
#pragma unroll
        for (int k = 0; k < 16; k++) {
            e[k] = a[2 * k];
            o[k] = a[2 * k + 1];
        }
        Dft<16>::run(e);
        Dft<16>::run(o);
        // o_k *= exp(-2 pi i k / 32) = cos - i sin, with both taken from the first quarter wave
#pragma unroll
        for (int k = 1; k < 16; k++) {
            if (k == 8) {
                o[k] = mul_minus_i(o[k]);
            } else {
                const float cs = k < 8 ? c[k] : -c[16 - k];   // cos(2 pi k / 32)
                const float sn = k < 8 ? c[8 - k] : c[k - 8]; // sin(2 pi k / 32)
                o[k] = cmul(o[k], make_float2(cs, -sn));
            }
        }
#pragma unroll
        for (int k = 0; k < 16; k++) {
            a[k] = cadd(e[k], o[k]);
            a[k + 16] = csub(e[k], o[k]);
        }
    }
};

// ---------------------------------------------------------------------------
// Register-resident transforms for power-of-two lines, Nr = 512 ... 8192.
// Each of the Nr/16 threads holds 16 elements, element t + T p in slot p
// (T = Nr/16).  A transform is radix-16 passes (the last one radix 2, 4 or 8
// when log2 Nr is not a multiple of 4) in the same self-sorting Stockham
// order as above; the first pass reads the thread's registers, the last pass
// leaves its results in registers in the same t + T p layout, and the passes
// in between exchange through two padded shared-memory buffers used in turn
// (one element of padding per 16 keeps the strided reads free of bank
// conflicts; alternating buffers leaves one barrier per exchange).  So the
// forward transform's output, the filter multiply and the inverse transforms'
// inputs never touch shared memory, and each transform costs log16(Nr) - 1
// exchanges.
// ---------------------------------------------------------------------------

__device__ __forceinline__ int pad16(int i) { return i + (i >> 4); }

// Twiddle load kept opaque to the compiler: the forward and inverse transforms of a line read the
// same twiddles, and merging their powers across the two would keep ~60 more registers live.
__device__ __forceinline__ float2 ld_twiddle(const float2 *p)
{
    float2 v;
    asm volatile("ld.global.nc.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
    return v;
}

// Raw-line load that leaves L1 to the filter, ramp and twiddle tables: each raw sample is read
// once, and letting the line stream through L1 evicts the tables that every line re-reads.
__device__ __forceinline__ float2 ld_raw(const float2 *p)
{
    float2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
    return v;
}

// w^p for p = 0 .. R-1 from w^1, multiplying powers of two (depth log2 R)
template <int R>
__device__ __forceinline__ void twiddle_powers(float2 w1, float2 *w)
{
    w[0] = make_float2(1.0f, 0.0f);
    w[1] = w1;
#pragma unroll
    for (int p = 2; p < R; p++) {
        const int hb = 1 << (31 - __clz(p));
        w[p] = (hb == p) ? cmul(w[p / 2], w[p / 2]) : cmul(w[hb], w[p - hb]);
    }
}

// One pass of radix R after L elements have been combined (L > 1): every
// thread loads its 16/R butterflies from `src`, transforms them and writes them
// to `dst` followed by a barrier, or keeps them in registers when kLast.  With
// one buffer (src == dst) a barrier also separates the loads from the stores.  An inverse pass
// (kInv) takes its twiddles from the conjugated table.
template <int N, int R, int L, bool kLast, bool kOneBuf, bool kTableTw, bool kInv = false>
__device__ __forceinline__ void reg_pass(float2 (&x)[16], const float2 *src, float2 *dst, const float2 *__restrict__ tw)
{
    constexpr int T = N / 16, SP = N / (L * R), NB = 16 / R;
    const int t = threadIdx.x;
#pragma unroll
    for (int i = 0; i < NB; i++) {
        const int b = t + T * i;
        const int jp = b % SP, kp = b / SP;
#pragma unroll
        for (int p = 0; p < R; p++) x[i * R + p] = src[pad16(kp * SP * R + jp + SP * p)];
    }
    if (kOneBuf && !kLast) __syncthreads();
#pragma unroll
    for (int i = 0; i < NB; i++) {
        const int b = t + T * i;
        const int jp = b % SP, kp = b / SP;
        float2 w[R];
        if constexpr (kTableTw && SP >= 8) {
            // at most four butterfly columns kp per warp: read every power w_N^(SP kp p) from the
            // table (SP kp p < N; the loads broadcast) instead of multiplying them out
            w[0] = make_float2(1.0f, 0.0f);
#pragma unroll
            for (int p = 1; p < R; p++) w[p] = ld_twiddle(tw + SP * kp * p);
        } else {
            twiddle_powers<R>(ld_twiddle(tw + SP * kp), w);
        }
#pragma unroll
        for (int p = 1; p < R; p++) x[i * R + p] = cmul(x[i * R + p], w[p]);
        Dft<R, kInv>::run(x + i * R);
        if (!kLast) {
#pragma unroll
            for (int q = 0; q < R; q++) dst[pad16((kp + L * q) * SP + jp)] = x[i * R + q];
        }
    }
    if (!kLast) __syncthreads();
    if (kLast && NB > 1) {
        // outputs (t + T i) + (N / R) q = t + T (i + NB q): move them to slot i + NB q
        float2 y[16];
#pragma unroll
        for (int i = 0; i < NB; i++)
#pragma unroll
            for (int q = 0; q < R; q++) y[i + NB * q] = x[i * R + q];
#pragma unroll
        for (int p = 0; p < 16; p++) x[p] = y[p];
    }
}

// Forward DFT of the line held as x[p] = element t + T p; result in the same layout.  With kInv
// the unnormalised inverse DFT instead, given the conjugated twiddle table: conjugated constants
// throughout, bit-identical to conjugating the input and the output of the forward transform.
// With two buffers (kTwoBuf) the exchanges alternate between them, so that each needs one
// barrier: every write goes to the buffer read two exchanges earlier, and the barrier of the
// exchange in between orders all of those reads before it.  The pair (a, b) carries the
// alternation from one transform to the next; `a` is the buffer the next exchange writes.  With
// one buffer (a == b) each exchange takes a second barrier before its stores, and the transform
// ends with one, so that the next transform may write the buffer.
template <int N, bool kTwoBuf, bool kTableTw = false, bool kInv = false>
__device__ __forceinline__ void reg_dft(float2 (&x)[16], float2 *&a, float2 *&b, const float2 *__restrict__ tw)
{
    constexpr int T = N / 16;
    constexpr bool k1 = !kTwoBuf;
    const int t = threadIdx.x;
    Dft<16, kInv>::run(x);                                      // pass 1: L = 1, no twiddles
#pragma unroll
    for (int q = 0; q < 16; q++) a[pad16(q * T + t)] = x[q];
    __syncthreads();
    if constexpr (N == 512) {
        reg_pass<N, 16, 16, false, k1, kTableTw, kInv>(x, a, b, tw);
        reg_pass<N, 2, 256, true, k1, kTableTw, kInv>(x, b, nullptr, tw);
    } else if constexpr (N == 1024) {
        reg_pass<N, 16, 16, false, k1, kTableTw, kInv>(x, a, b, tw);
        reg_pass<N, 4, 256, true, k1, kTableTw, kInv>(x, b, nullptr, tw);
    } else if constexpr (N == 2048) {
        reg_pass<N, 16, 16, false, k1, kTableTw, kInv>(x, a, b, tw);
        reg_pass<N, 8, 256, true, k1, kTableTw, kInv>(x, b, nullptr, tw);
    } else if constexpr (N == 4096) {
        reg_pass<N, 16, 16, false, k1, kTableTw, kInv>(x, a, b, tw);
        reg_pass<N, 16, 256, true, k1, kTableTw, kInv>(x, b, nullptr, tw);
    } else {
        static_assert(N == 8192, "unsupported line length");
        reg_pass<N, 16, 16, false, k1, kTableTw, kInv>(x, a, b, tw);
        reg_pass<N, 16, 256, false, k1, kTableTw, kInv>(x, b, a, tw);
        reg_pass<N, 2, 4096, true, k1, kTableTw, kInv>(x, a, nullptr, tw);
        float2 *c = a;                                          // three exchanges: the next one writes b
        a = b;
        b = c;
    }
    if constexpr (!kTwoBuf) __syncthreads();                    // the buffer is free for the next transform
}

// ---------------------------------------------------------------------------
// Line staging by the tensor memory accelerator: each CTA stays resident and
// loops over lines; while it transforms one line out of its registers, one
// bulk copy (cp.async.bulk, completion counted in bytes on an mbarrier)
// brings the next raw line into a shared-memory stage, so the load latency is
// hidden even with a single CTA per SM.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void stage_barrier_init(uint64_t *bar)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// One bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) into the stage,
// announced on the barrier as its expected transaction count.  Issued by one thread, after a
// CTA barrier that ended every generic-proxy read of the stage.
__device__ __forceinline__ void stage_line(uint64_t *bar, void *stage, const void *src, uint32_t bytes)
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(stage)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ bool stage_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Non-blocking test of the barrier phase of the given parity.
__device__ __forceinline__ bool stage_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return done != 0;
}

// Wait for the barrier phase of the given parity; false if limit_ns (or an iteration cap) passed
// first.  limit_ns = 0 tests the phase once without waiting (the plan's wait-limit knob, which
// lets a test make the wait run out).
__device__ __forceinline__ bool stage_wait(uint64_t *bar, uint32_t parity, unsigned long long limit_ns)
{
    if (limit_ns == 0) return stage_test_wait(bar, parity);
    if (stage_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 0; i < (1u << 30); i++) {
        if (stage_try_wait(bar, parity)) return true;
        if ((i & 63) == 63 && global_ns() - t0 > limit_ns) break;
    }
    return false;
}

}  // namespace
}  // namespace sar
