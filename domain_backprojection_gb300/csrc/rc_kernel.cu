// rc_kernel.cu -- fused range compression: per pulse, DFT -> multiply by the
// conjugate-chirp spectrum -> zero-padded upsampling -> IDFT, in one kernel
// with one HBM read of the raw line and one write of the compressed line.
//
// The fusion follows "Fused FFT -> filter -> IFFT for SAR on Apple Silicon",
// section 3.1 (one thread group per line, all intermediates on chip) and
// section 3.2 (IDFT(x) = conj(DFT(conj x)) / N, so the inverse reuses the
// forward transform).  The matched filter is the frequency-domain one of
// "GPU-accelerated backprojection SAR imaging", section 3.1.
//
// Upsampling by U never materialises the U Nr-point spectrum: with signed
// frequencies k_s in [-Nr/2, Nr/2), output sample U m + u of the zero-padded
// IDFT is
//     rc[U m + u] = (1/Nr) sum_k Y[k] exp(+j 2 pi k_s u / (U Nr)) exp(+j 2 pi k m / Nr),
// i.e. U Nr-point inverse transforms of the same on-chip spectrum, each with a
// per-u phase ramp (a polyphase split of the output index).
//
// Transforms are self-sorting mixed-radix Stockham passes (radices 16, 8, 5, 4,
// 3, 2) between two shared-memory buffers; the spectrum stays in a third.
#include "sar_internal.cuh"

namespace sar {
namespace {

__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 csub(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }
__device__ __forceinline__ float2 cmul(float2 a, float2 b)
{
    return make_float2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.x, b.y, a.y * b.x));
}
__device__ __forceinline__ float2 cconj(float2 a) { return make_float2(a.x, -a.y); }
__device__ __forceinline__ float2 mul_minus_i(float2 a) { return make_float2(a.y, -a.x); }   // -i a
__device__ __forceinline__ float2 cscale(float2 a, float s) { return make_float2(a.x * s, a.y * s); }

// Forward DFTs of small sizes, in registers: y_k = sum_j a_j exp(-2 pi i j k / R).
template <int R> struct Dft;

template <> struct Dft<2> {
    static __device__ __forceinline__ void run(float2 *a)
    {
        float2 t = a[0];
        a[0] = cadd(t, a[1]);
        a[1] = csub(t, a[1]);
    }
};

template <> struct Dft<3> {
    static __device__ __forceinline__ void run(float2 *a)
    {
        const float s = 0.86602540378443864676f;   // sin(2 pi / 3)
        float2 b = cadd(a[1], a[2]);
        float2 d = csub(a[1], a[2]);
        float2 t = make_float2(a[0].x - 0.5f * b.x, a[0].y - 0.5f * b.y);
        float2 v = mul_minus_i(cscale(d, s));
        a[0] = cadd(a[0], b);
        a[1] = cadd(t, v);
        a[2] = csub(t, v);
    }
};

template <> struct Dft<4> {
    static __device__ __forceinline__ void run(float2 *a)
    {
        float2 s02 = cadd(a[0], a[2]), d02 = csub(a[0], a[2]);
        float2 s13 = cadd(a[1], a[3]), d13 = mul_minus_i(csub(a[1], a[3]));
        a[0] = cadd(s02, s13);
        a[2] = csub(s02, s13);
        a[1] = cadd(d02, d13);
        a[3] = csub(d02, d13);
    }
};

template <> struct Dft<5> {
    static __device__ __forceinline__ void run(float2 *a)
    {
        const float c1 = 0.30901699437494742410f;    // cos(2 pi / 5)
        const float c2 = -0.80901699437494742410f;   // cos(4 pi / 5)
        const float s1 = 0.95105651629515357212f;    // sin(2 pi / 5)
        const float s2 = 0.58778525229247312917f;    // sin(4 pi / 5)
        float2 b1 = cadd(a[1], a[4]), d1 = csub(a[1], a[4]);
        float2 b2 = cadd(a[2], a[3]), d2 = csub(a[2], a[3]);
        float2 t1 = make_float2(fmaf(c1, b1.x, fmaf(c2, b2.x, a[0].x)), fmaf(c1, b1.y, fmaf(c2, b2.y, a[0].y)));
        float2 t2 = make_float2(fmaf(c2, b1.x, fmaf(c1, b2.x, a[0].x)), fmaf(c2, b1.y, fmaf(c1, b2.y, a[0].y)));
        float2 u1 = make_float2(fmaf(s1, d1.x, s2 * d2.x), fmaf(s1, d1.y, s2 * d2.y));
        float2 u2 = make_float2(fmaf(s2, d1.x, -s1 * d2.x), fmaf(s2, d1.y, -s1 * d2.y));
        u1 = mul_minus_i(u1);
        u2 = mul_minus_i(u2);
        a[0] = cadd(a[0], cadd(b1, b2));
        a[1] = cadd(t1, u1);
        a[4] = csub(t1, u1);
        a[2] = cadd(t2, u2);
        a[3] = csub(t2, u2);
    }
};

// 6 = 2 x 3 and 10 = 2 x 5: DFTs of the even and the odd samples, the odd ones turned by
// exp(-2 pi i k / R), then sums and differences.
template <> struct Dft<6> {
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
            a[k] = cadd(e[k], o[k]);
            a[k + 3] = csub(e[k], o[k]);
        }
    }
};

template <> struct Dft<10> {
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
            a[k] = cadd(e[k], o[k]);
            a[k + 5] = csub(e[k], o[k]);
        }
    }
};

template <> struct Dft<8> {
    static __device__ __forceinline__ void run(float2 *a)
    {
        const float r = 0.70710678118654752440f;
        float2 e[4] = {a[0], a[2], a[4], a[6]};
        float2 o[4] = {a[1], a[3], a[5], a[7]};
        Dft<4>::run(e);
        Dft<4>::run(o);
        // o_k *= exp(-2 pi i k / 8)
        o[1] = make_float2(r * (o[1].x + o[1].y), r * (o[1].y - o[1].x));
        o[2] = mul_minus_i(o[2]);
        o[3] = make_float2(r * (o[3].y - o[3].x), -r * (o[3].x + o[3].y));
#pragma unroll
        for (int k = 0; k < 4; k++) {
            a[k] = cadd(e[k], o[k]);
            a[k + 4] = csub(e[k], o[k]);
        }
    }
};

template <> struct Dft<16> {
    static __device__ __forceinline__ void run(float2 *a)
    {
        // n = 4 n1 + n2, k = k1 + 4 k2: inner DFT4 over n1, twiddle w16^(n2 k1), outer DFT4 over n2
        float2 b[4][4];
#pragma unroll
        for (int n2 = 0; n2 < 4; n2++) {
            float2 t[4] = {a[n2], a[4 + n2], a[8 + n2], a[12 + n2]};
            Dft<4>::run(t);
#pragma unroll
            for (int k1 = 0; k1 < 4; k1++) b[n2][k1] = t[k1];
        }
        const float c = 0.92387953251128675613f, s = 0.38268343236508977173f, r = 0.70710678118654752440f;
        // w16^m = exp(-2 pi i m / 16) for m = n2 * k1
        b[1][1] = cmul(b[1][1], make_float2(c, -s));
        b[1][2] = cmul(b[1][2], make_float2(r, -r));
        b[1][3] = cmul(b[1][3], make_float2(s, -c));
        b[2][1] = cmul(b[2][1], make_float2(r, -r));
        b[2][2] = mul_minus_i(b[2][2]);
        b[2][3] = cmul(b[2][3], make_float2(-r, -r));
        b[3][1] = cmul(b[3][1], make_float2(s, -c));
        b[3][2] = cmul(b[3][2], make_float2(-r, -r));
        b[3][3] = cmul(b[3][3], make_float2(-c, s));
#pragma unroll
        for (int k1 = 0; k1 < 4; k1++) {
            float2 t[4] = {b[0][k1], b[1][k1], b[2][k1], b[3][k1]};
            Dft<4>::run(t);
#pragma unroll
            for (int k2 = 0; k2 < 4; k2++) a[k1 + 4 * k2] = t[k2];
        }
    }
};

// One self-sorting Stockham pass of radix R.  Before the pass the buffer holds
// the length-L transforms A_j of the stride-S subsequences x[j + S n''] (S = N/L)
// at index k S + j; after it, the length-(L R) transforms of the stride-S'
// subsequences (S' = S / R) at index k S' + j.  Butterfly (j', k'):
//   B_{j'}[k' + L q] = sum_p w_R^{p q} w_{L R}^{p k'} A_{j' + S' p}[k'].
template <int R>
__device__ __forceinline__ void stockham_pass(const float2 *__restrict__ src, float2 *__restrict__ dst, int n, int L,
                                              const float2 *__restrict__ tw)
{
    const int sp = n / (L * R);
    const int nb = n / R;
    for (int b = threadIdx.x; b < nb; b += blockDim.x) {
        const int jp = b % sp, kp = b / sp;
        float2 a[R];
#pragma unroll
        for (int p = 0; p < R; p++) a[p] = src[kp * sp * R + jp + sp * p];
        if (L > 1) {
#pragma unroll
            for (int p = 1; p < R; p++) a[p] = cmul(a[p], __ldg(tw + sp * p * kp));   // w_N^(S' p k')
        }
        Dft<R>::run(a);
#pragma unroll
        for (int q = 0; q < R; q++) dst[(kp + L * q) * sp + jp] = a[q];
    }
}

// Full forward transform, ping-ponging between a and b; returns the buffer
// that holds the natural-order result.
__device__ float2 *dft_forward(float2 *a, float2 *b, const RcArgs &args)
{
    int L = 1;
    for (int s = 0; s < args.n_passes; s++) {
        const int r = args.radix[s];
        switch (r) {
        case 16: stockham_pass<16>(a, b, args.n, L, args.tw); break;
        case 8: stockham_pass<8>(a, b, args.n, L, args.tw); break;
        case 5: stockham_pass<5>(a, b, args.n, L, args.tw); break;
        case 4: stockham_pass<4>(a, b, args.n, L, args.tw); break;
        case 3: stockham_pass<3>(a, b, args.n, L, args.tw); break;
        default: stockham_pass<2>(a, b, args.n, L, args.tw); break;
        }
        __syncthreads();
        float2 *t = a;
        a = b;
        b = t;
        L *= r;
    }
    return a;
}

__global__ void __launch_bounds__(512) rc_fused_kernel(const float2 *__restrict__ raw, float2 *__restrict__ rc,
                                                       int64_t n_lines, RcArgs args)
{
    extern __shared__ float4 smem4[];
    float2 *sm = reinterpret_cast<float2 *>(smem4);
    const int n = args.n, U = args.u;
    // U = 1 needs no copy of the spectrum: two buffers (see rc_smem_bytes)
    float2 *A = sm, *B = sm + n, *Y = sm + 2 * n;
    const int un = U * n;
    const int lo_mask = (1 << args.ptw_lo_bits) - 1;

    for (int64_t line = blockIdx.x; line < n_lines; line += gridDim.x) {
        // load the raw line (16-byte vector loads; Nr is even)
        const float4 *src = reinterpret_cast<const float4 *>(raw + line * n);
        for (int i = threadIdx.x; i < n / 2; i += blockDim.x) reinterpret_cast<float4 *>(A)[i] = __ldg(src + i);
        __syncthreads();
        float2 *X = dft_forward(A, B, args);
        float2 *out = rc + line * (int64_t)un;
        if (U == 1) {
            // conj(X H) in place, transformed, conjugated on the way out
            for (int k = threadIdx.x; k < n; k += blockDim.x) X[k] = cconj(cmul(X[k], __ldg(args.h + k)));
            __syncthreads();
            const float2 *Z = dft_forward(X, X == A ? B : A, args);
            for (int i = threadIdx.x; i < n / 2; i += blockDim.x) {
                const float4 v = reinterpret_cast<const float4 *>(Z)[i];
                reinterpret_cast<float4 *>(out)[i] = make_float4(v.x, -v.y, v.z, -v.w);
            }
            __syncthreads();
            continue;
        }
        // matched filter: Y = X * conj(DFT(chirp))
        for (int k = threadIdx.x; k < n; k += blockDim.x) Y[k] = cmul(X[k], __ldg(args.h + k));
        __syncthreads();
        for (int u = 0; u < U; u++) {
            // conj(Z_u)[k] = conj(Y[k]) * exp(-j 2 pi k_s u / (U Nr))
            for (int k = threadIdx.x; k < n; k += blockDim.x) {
                float2 z = cconj(Y[k]);
                if (u != 0) {
                    const int ks = (2 * k >= n) ? k - n : k;
                    int t = (ks * u) % un;
                    if (t < 0) t += un;
                    const float2 w = cmul(__ldg(args.ptw_hi + (t >> args.ptw_lo_bits)), __ldg(args.ptw_lo + (t & lo_mask)));
                    z = cmul(z, w);
                }
                A[k] = z;
            }
            __syncthreads();
            float2 *Z = dft_forward(A, B, args);
            // rc[U m + u] = conj(DFT(conj Z_u))[m] (the 1 / Nr is in H)
            if (args.planar) {
                for (int m = threadIdx.x; m < n; m += blockDim.x) {
                    const float2 v = Z[m];
                    out[(int64_t)u * n + m] = cconj(v);
                }
            } else {
                for (int m = threadIdx.x; m < n; m += blockDim.x) {
                    const float2 v = Z[m];
                    out[(int64_t)U * m + u] = cconj(v);
                }
            }
            __syncthreads();
        }
    }
}

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
// one buffer (src == dst) a barrier also separates the loads from the stores.
template <int N, int R, int L, bool kLast, bool kOneBuf>
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
        twiddle_powers<R>(ld_twiddle(tw + SP * kp), w);
#pragma unroll
        for (int p = 1; p < R; p++) x[i * R + p] = cmul(x[i * R + p], w[p]);
        Dft<R>::run(x + i * R);
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

// Forward DFT of the line held as x[p] = element t + T p; result in the same layout.
// With two buffers (kTwoBuf) the exchanges alternate between them, so that each needs one
// barrier: every write goes to the buffer read two exchanges earlier, and the barrier of the
// exchange in between orders all of those reads before it.  The pair (a, b) carries the
// alternation from one transform to the next; `a` is the buffer the next exchange writes.  With
// one buffer (a == b) each exchange takes a second barrier before its stores, and the transform
// ends with one, so that the next transform may write the buffer.
template <int N, bool kTwoBuf>
__device__ __forceinline__ void reg_dft(float2 (&x)[16], float2 *&a, float2 *&b, const float2 *__restrict__ tw)
{
    constexpr int T = N / 16;
    constexpr bool k1 = !kTwoBuf;
    const int t = threadIdx.x;
    Dft<16>::run(x);                                            // pass 1: L = 1, no twiddles
#pragma unroll
    for (int q = 0; q < 16; q++) a[pad16(q * T + t)] = x[q];
    __syncthreads();
    if constexpr (N == 512) {
        reg_pass<N, 16, 16, false, k1>(x, a, b, tw);
        reg_pass<N, 2, 256, true, k1>(x, b, nullptr, tw);
    } else if constexpr (N == 1024) {
        reg_pass<N, 16, 16, false, k1>(x, a, b, tw);
        reg_pass<N, 4, 256, true, k1>(x, b, nullptr, tw);
    } else if constexpr (N == 2048) {
        reg_pass<N, 16, 16, false, k1>(x, a, b, tw);
        reg_pass<N, 8, 256, true, k1>(x, b, nullptr, tw);
    } else if constexpr (N == 4096) {
        reg_pass<N, 16, 16, false, k1>(x, a, b, tw);
        reg_pass<N, 16, 256, true, k1>(x, b, nullptr, tw);
    } else {
        static_assert(N == 8192, "unsupported line length");
        reg_pass<N, 16, 16, false, k1>(x, a, b, tw);
        reg_pass<N, 16, 256, false, k1>(x, b, a, tw);
        reg_pass<N, 2, 4096, true, k1>(x, a, nullptr, tw);
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

// Wait for the barrier phase of the given parity; false if kWaitLimitNs (or an iteration cap)
// passed first.
__device__ __forceinline__ bool stage_wait(uint64_t *bar, uint32_t parity)
{
    if (stage_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 0; i < (1u << 30); i++) {
        if (stage_try_wait(bar, parity)) return true;
        if ((i & 63) == 63 && global_ns() - t0 > kWaitLimitNs) break;
    }
    return false;
}

// Resident CTAs per SM each line kernel is built for: the register budget that __launch_bounds__
// enforces.  16 warps per SM for short lines; 3 CTAs for 4096-point lines without upsampling (no
// copy of the spectrum to keep), 2 with it; one 16-warp CTA for 8192-point lines.
template <int N, bool kMulti>
__host__ __device__ constexpr int rc_reg_min_ctas()
{
    return N == 8192 ? 1 : N == 4096 ? (kMulti ? 2 : 3) : (16 * 32) / (N / 16);
}

// Whether the (N, U) line kernel stages lines by bulk copy (persistent CTAs) or loads them
// straight into registers (one CTA per line).  Staging pays where a single CTA holds the SM
// (8192-point lines), so nothing else covers the load latency.  Where two or three CTAs share an
// SM, their loads overlap each other's transforms, and the stage's shared memory would instead
// take L1 capacity from the filter and ramp tables (measured on GB300: 4096-point lines without
// upsampling 0.081 ms unstaged against 0.085 ms staged, with upsampling 0.381 against 0.405 ms).
template <int N, bool kMulti>
__host__ __device__ constexpr bool rc_reg_staged() { return N == 8192; }

// Whether the (N, U) line kernel alternates two exchange buffers (one barrier per exchange) or
// uses one (two barriers per exchange, half the shared memory).  One buffer where three CTAs share
// an SM: their six buffers would leave L1 too little room for the filter table (measured on
// GB300: 4096-point lines without upsampling 0.081 ms with one buffer, 0.089 ms with two).
template <int N, bool kMulti>
__host__ __device__ constexpr bool rc_reg_two_buffers() { return rc_reg_min_ctas<N, kMulti>() < 3; }

// Exchange buffers of N + N/16 entries, then (staged kernels) the raw-line stage and its barrier.
template <int N, bool kMulti>
constexpr size_t rc_reg_smem()
{
    return (rc_reg_two_buffers<N, kMulti>() ? 2 : 1) * (size_t)(N + N / 16) * sizeof(float2) +
           (rc_reg_staged<N, kMulti>() ? (size_t)N * sizeof(float2) + 16 : 0);
}

// One line held in registers (x[p] = raw element t + T p): forward transform, matched filter,
// U inverse transforms, stores of the compressed line.
template <int N, bool kMulti>
__device__ __forceinline__ void rc_reg_line(float2 (&x)[16], float2 *&a, float2 *&b, float2 *__restrict__ out,
                                            const RcArgs &args)
{
    constexpr int T = N / 16;
    const int t = threadIdx.x;
    if constexpr (!kMulti) {
        // forward transform, filter and conjugate, inverse transform: one copy of the transform
        // code in a two-trip loop (two inlined copies spill)
#pragma unroll 1
        for (int k = 0; k < 2; k++) {
            reg_dft<N, rc_reg_two_buffers<N, kMulti>()>(x, a, b, args.tw);
            if (k == 0) {
#pragma unroll
                for (int p = 0; p < 16; p++) x[p] = cconj(cmul(x[p], __ldg(args.h + t + T * p)));
            }
        }
#pragma unroll
        for (int p = 0; p < 16; p++) out[t + T * p] = cconj(x[p]);
    } else {
        const int U = args.u;
        reg_dft<N, rc_reg_two_buffers<N, kMulti>()>(x, a, b, args.tw);
        // matched filter (with the IDFT's 1 / Nr)
        float2 y[16];
#pragma unroll
        for (int p = 0; p < 16; p++) y[p] = cmul(x[p], __ldg(args.h + t + T * p));
        for (int u = 0; u < U; u++) {
            // y = Y exp(+j 2 pi k_s u / (U N)); inverse transform by the conjugate identity
#pragma unroll
            for (int p = 0; p < 16; p++) x[p] = cconj(y[p]);
            reg_dft<N, rc_reg_two_buffers<N, kMulti>()>(x, a, b, args.tw);
            if (args.planar) {
                float2 *plane = out + (int64_t)u * N;
#pragma unroll
                for (int p = 0; p < 16; p++) plane[t + T * p] = cconj(x[p]);
            } else {
#pragma unroll
                for (int p = 0; p < 16; p++) out[(int64_t)U * (t + T * p) + u] = cconj(x[p]);
            }
            if (u + 1 < U) {
#pragma unroll
                for (int p = 0; p < 16; p++) y[p] = cmul(y[p], __ldg(args.ramp + t + T * p));
            }
        }
    }
}

template <int N, bool kMulti>
__global__ void __launch_bounds__(N / 16, (rc_reg_min_ctas<N, kMulti>()))
    rc_reg_kernel(const float2 *__restrict__ raw, float2 *__restrict__ rc, int64_t n_lines, RcArgs args)
{
    extern __shared__ float4 smem4[];
    constexpr int T = N / 16;
    float2 *a = reinterpret_cast<float2 *>(smem4);             // exchange buffers, N + N/16 entries each
    float2 *b = rc_reg_two_buffers<N, kMulti>() ? a + N + N / 16 : a;
    const int t = threadIdx.x;
    const int64_t line_elems = (int64_t)(kMulti ? args.u : 1) * N;
    int64_t line = blockIdx.x;
    if constexpr (!rc_reg_staged<N, kMulti>()) {
        for (; line < n_lines; line += gridDim.x) {
            float2 x[16];
            const float2 *src = raw + line * N;
#pragma unroll
            for (int p = 0; p < 16; p++) x[p] = ld_raw(src + t + T * p);
            rc_reg_line<N, kMulti>(x, a, b, rc + line * line_elems, args);
        }
    } else {
        float2 *stage = (rc_reg_two_buffers<N, kMulti>() ? b : a) + N + N / 16;   // raw line, N entries
                                                                // (16-byte aligned)
        uint64_t *bar = reinterpret_cast<uint64_t *>(stage + N);
        if (line >= n_lines) return;
        if (t == 0) stage_barrier_init(bar);
        __syncthreads();
        if (t == 0) stage_line(bar, stage, raw + line * N, N * sizeof(float2));
        uint32_t parity = 0;
        for (; line < n_lines; line += gridDim.x) {
            const bool ok = stage_wait(bar, parity);
            parity ^= 1u;
            float2 x[16];
#pragma unroll
            for (int p = 0; p < 16; p++) x[p] = stage[t + T * p];
            if (__syncthreads_or(!ok)) {                        // the stage is free again (or the copy never came)
                if (t == 0) atomicOr(args.err, kDevErrTimeout);
                return;
            }
            if (t == 0 && line + gridDim.x < n_lines)
                stage_line(bar, stage, raw + (line + gridDim.x) * N, N * sizeof(float2));
            rc_reg_line<N, kMulti>(x, a, b, rc + line * line_elems, args);
        }
    }
}

// ---------------------------------------------------------------------------
// Register-resident transform for Nr = 6000 = 2^4 3 5^3 (the non-power-of-two
// line of the range-only sweep): 200 threads of 30 elements, element t + T p in
// slot p (T = 200), and four Stockham passes of radix 10, 10, 10 and 6, each
// thread running 30 / R butterflies per pass.  As in the power-of-two kernel,
// the first pass reads registers, the last leaves its output in registers in
// the t + T p layout, and the passes in between exchange through shared memory.
// ---------------------------------------------------------------------------
template <int N, int E, int R, int L, bool kFirst, bool kLast, bool kOneBuf>
__device__ __forceinline__ void mixed_pass(float2 (&x)[E], const float2 *src, float2 *dst, const float2 *__restrict__ tw)
{
    constexpr int T = N / E, SP = N / (L * R), NB = E / R;
    static_assert(E % R == 0 && N % (L * R) == 0, "pass does not fit the layout");
    const int t = threadIdx.x;
    if (kFirst) {
        // butterfly i takes elements (t + T i) + (N / R) p = t + T (i + NB p): slot i + NB p
        float2 y[E];
#pragma unroll
        for (int i = 0; i < NB; i++)
#pragma unroll
            for (int p = 0; p < R; p++) y[i * R + p] = x[i + NB * p];
#pragma unroll
        for (int k = 0; k < E; k++) x[k] = y[k];
    } else {
#pragma unroll
        for (int i = 0; i < NB; i++) {
            const int b = t + T * i;
            const int jp = b % SP, kp = b / SP;
#pragma unroll
            for (int p = 0; p < R; p++) x[i * R + p] = src[kp * SP * R + jp + SP * p];
        }
        if (kOneBuf && !kLast) __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < NB; i++) {
        const int b = t + T * i;
        const int jp = b % SP, kp = b / SP;
        if (!kFirst) {
            float2 w[R];
            twiddle_powers<R>(ld_twiddle(tw + SP * kp), w);
#pragma unroll
            for (int p = 1; p < R; p++) x[i * R + p] = cmul(x[i * R + p], w[p]);
        }
        Dft<R>::run(x + i * R);
        if (!kLast) {
#pragma unroll
            for (int q = 0; q < R; q++) dst[(kp + L * q) * SP + jp] = x[i * R + q];
        }
    }
    if (!kLast) __syncthreads();
    if (kLast) {
        // outputs (t + T i) + (N / R) q = t + T (i + NB q): slot i + NB q
        float2 y[E];
#pragma unroll
        for (int i = 0; i < NB; i++)
#pragma unroll
            for (int q = 0; q < R; q++) y[i + NB * q] = x[i * R + q];
#pragma unroll
        for (int k = 0; k < E; k++) x[k] = y[k];
    }
}

// Forward DFT of the 6000-point line held as x[p] = element t + T p; result in the same layout.
// Exchanges use one or two buffers as in reg_dft; with two, there are three exchanges, so the
// next transform starts on the other buffer.
template <bool kTwoBuf>
__device__ __forceinline__ void mixed_dft6000(float2 (&x)[30], float2 *&a, float2 *&b, const float2 *__restrict__ tw)
{
    constexpr bool k1 = !kTwoBuf;
    mixed_pass<6000, 30, 10, 1, true, false, k1>(x, nullptr, a, tw);
    mixed_pass<6000, 30, 10, 10, false, false, k1>(x, a, b, tw);
    mixed_pass<6000, 30, 10, 100, false, false, k1>(x, b, a, tw);
    mixed_pass<6000, 30, 6, 1000, false, true, k1>(x, a, nullptr, tw);
    float2 *c = a;
    a = b;
    b = c;
    if constexpr (!kTwoBuf) __syncthreads();                    // the buffer is free for the next transform
}

constexpr int kRcMixedCtas = 1;     // with upsampling the 30-element layout and the spectrum copy want
                                    // ~250 registers; bounding them to fit 2 CTAs per SM spills.  Without
                                    // upsampling (no copy) 128 registers suffice and 2 CTAs fit.

// Whether the 6000-point kernel stages lines by bulk copy (persistent CTAs, one per SM: the stage
// does not fit beside two CTAs' exchange buffers) or loads them into registers (two CTAs per SM
// without upsampling).
__host__ __device__ constexpr bool rc_mixed_staged(bool multi) { return multi; }

// Two exchange buffers (one barrier per exchange), or one where two CTAs share an SM and two
// buffers each would leave L1 too little room for the 48 KB filter table.
__host__ __device__ constexpr bool rc_mixed_two_buffers(bool multi) { return multi; }

// Exchange buffers of 6000 entries, then (staged) the raw-line stage and its barrier.
__host__ __device__ constexpr size_t rc_mixed_smem(bool multi)
{
    return (rc_mixed_two_buffers(multi) ? 2 : 1) * 6000 * sizeof(float2) +
           (rc_mixed_staged(multi) ? 6000 * sizeof(float2) + 16 : 0);
}

template <bool kMulti>
__device__ __forceinline__ void rc_mixed_line(float2 (&x)[30], float2 *&a, float2 *&b, float2 *__restrict__ out,
                                              const RcArgs &args)
{
    constexpr int N = 6000, E = 30, T = N / E;
    const int t = threadIdx.x;
    if constexpr (!kMulti) {
        // forward transform, filter (with the IDFT's 1 / Nr) and conjugate, inverse transform
#pragma unroll 1
        for (int k = 0; k < 2; k++) {
            mixed_dft6000<rc_mixed_two_buffers(kMulti)>(x, a, b, args.tw);
            if (k == 0) {
#pragma unroll
                for (int p = 0; p < E; p++) x[p] = cconj(cmul(x[p], __ldg(args.h + t + T * p)));
            }
        }
#pragma unroll
        for (int p = 0; p < E; p++) out[t + T * p] = cconj(x[p]);
    } else {
        const int U = args.u;
        mixed_dft6000<rc_mixed_two_buffers(kMulti)>(x, a, b, args.tw);
        // matched filter (with the IDFT's 1 / Nr)
        float2 y[E];
#pragma unroll
        for (int p = 0; p < E; p++) y[p] = cmul(x[p], __ldg(args.h + t + T * p));
        for (int u = 0; u < U; u++) {
#pragma unroll
            for (int p = 0; p < E; p++) x[p] = cconj(y[p]);
            mixed_dft6000<rc_mixed_two_buffers(kMulti)>(x, a, b, args.tw);
            if (args.planar) {
                float2 *plane = out + (int64_t)u * N;
#pragma unroll
                for (int p = 0; p < E; p++) plane[t + T * p] = cconj(x[p]);
            } else {
#pragma unroll
                for (int p = 0; p < E; p++) out[(int64_t)U * (t + T * p) + u] = cconj(x[p]);
            }
            if (u + 1 < U) {
#pragma unroll
                for (int p = 0; p < E; p++) y[p] = cmul(y[p], __ldg(args.ramp + t + T * p));
            }
        }
    }
}

template <bool kMulti>
__global__ void __launch_bounds__(200, kMulti ? kRcMixedCtas : 2) rc_mixed6000_kernel(const float2 *__restrict__ raw, float2 *__restrict__ rc,
                                                           int64_t n_lines, RcArgs args)
{
    constexpr int N = 6000, E = 30, T = N / E;
    extern __shared__ float4 smem4[];
    float2 *a = reinterpret_cast<float2 *>(smem4);
    float2 *b = rc_mixed_two_buffers(kMulti) ? a + N : a;
    const int t = threadIdx.x;
    const int64_t line_elems = (int64_t)(kMulti ? args.u : 1) * N;
    int64_t line = blockIdx.x;
    if constexpr (!rc_mixed_staged(kMulti)) {
        for (; line < n_lines; line += gridDim.x) {
            float2 x[E];
            const float2 *src = raw + line * N;
#pragma unroll
            for (int p = 0; p < E; p++) x[p] = ld_raw(src + t + T * p);
            rc_mixed_line<kMulti>(x, a, b, rc + line * line_elems, args);
        }
    } else {
        float2 *stage = (rc_mixed_two_buffers(kMulti) ? b : a) + N;   // 48000 or 96000 bytes in: 16-byte aligned
        uint64_t *bar = reinterpret_cast<uint64_t *>(stage + N);
        if (line >= n_lines) return;
        if (t == 0) stage_barrier_init(bar);
        __syncthreads();
        if (t == 0) stage_line(bar, stage, raw + line * N, N * sizeof(float2));
        uint32_t parity = 0;
        for (; line < n_lines; line += gridDim.x) {
            const bool ok = stage_wait(bar, parity);
            parity ^= 1u;
            float2 x[E];
#pragma unroll
            for (int p = 0; p < E; p++) x[p] = stage[t + T * p];
            if (__syncthreads_or(!ok)) {
                if (t == 0) atomicOr(args.err, kDevErrTimeout);
                return;
            }
            if (t == 0 && line + gridDim.x < n_lines)
                stage_line(bar, stage, raw + (line + gridDim.x) * N, N * sizeof(float2));
            rc_mixed_line<kMulti>(x, a, b, rc + line * line_elems, args);
        }
    }
}

}  // namespace

int rc_block_threads(int n) { return n >= 4096 ? 512 : 256; }

size_t rc_smem_bytes(int n, int u) { return (size_t)(u == 1 ? 2 : 3) * n * sizeof(float2); }

namespace {

template <typename K>
int resident(K kernel, int threads, size_t smem, int dev)
{
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return per_sm * sms;
}

template <int N, bool kMulti>
cudaError_t set_reg_smem()
{
    return cudaFuncSetAttribute(rc_reg_kernel<N, kMulti>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)rc_reg_smem<N, kMulti>());
}

// Resident CTAs of a staged (persistent) line kernel; unstaged ones take one CTA per line.
template <int N, bool kMulti>
int reg_resident(int dev)
{
    if (!rc_reg_staged<N, kMulti>()) return 1 << 20;
    return resident(rc_reg_kernel<N, kMulti>, N / 16, rc_reg_smem<N, kMulti>(), dev);
}


}  // namespace

cudaError_t rc_configure(int)
{
    // every kernel gets its largest shared-memory size, so plans of any size can coexist
    cudaError_t e = cudaFuncSetAttribute(rc_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)rc_smem_bytes(8192, 2));
    if (e == cudaSuccess) e = set_reg_smem<512, false>();
    if (e == cudaSuccess) e = set_reg_smem<512, true>();
    if (e == cudaSuccess) e = set_reg_smem<1024, false>();
    if (e == cudaSuccess) e = set_reg_smem<1024, true>();
    if (e == cudaSuccess) e = set_reg_smem<2048, false>();
    if (e == cudaSuccess) e = set_reg_smem<2048, true>();
    if (e == cudaSuccess) e = set_reg_smem<4096, false>();
    if (e == cudaSuccess) e = set_reg_smem<4096, true>();
    if (e == cudaSuccess) e = set_reg_smem<8192, false>();
    if (e == cudaSuccess) e = set_reg_smem<8192, true>();
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rc_mixed6000_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)rc_mixed_smem(false));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rc_mixed6000_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)rc_mixed_smem(true));
    return e;
}

bool rc_has_reg_path(int n) { return n == 512 || n == 1024 || n == 2048 || n == 4096 || n == 8192; }

int rc_resident_ctas(int n, int u, int dev)
{
    const bool multi = u > 1;
    switch (n) {
    case 512: return multi ? reg_resident<512, true>(dev) : reg_resident<512, false>(dev);
    case 1024: return multi ? reg_resident<1024, true>(dev) : reg_resident<1024, false>(dev);
    case 2048: return multi ? reg_resident<2048, true>(dev) : reg_resident<2048, false>(dev);
    case 4096: return multi ? reg_resident<4096, true>(dev) : reg_resident<4096, false>(dev);
    case 8192: return multi ? reg_resident<8192, true>(dev) : reg_resident<8192, false>(dev);
    case 6000:
        if (!rc_mixed_staged(multi)) return 1 << 20;
        return multi ? resident(rc_mixed6000_kernel<true>, 200, rc_mixed_smem(true), dev)
                     : resident(rc_mixed6000_kernel<false>, 200, rc_mixed_smem(false), dev);
    default: return 1 << 20;     // the shared-memory kernel takes one CTA per line (grid-stride beyond 2^20)
    }
}

template <int N>
static void launch_reg(const RcArgs &a, const float2 *raw, float2 *rc, int64_t n_lines, unsigned grid, cudaStream_t s)
{
    if (a.u > 1) rc_reg_kernel<N, true><<<grid, N / 16, rc_reg_smem<N, true>(), s>>>(raw, rc, n_lines, a);
    else rc_reg_kernel<N, false><<<grid, N / 16, rc_reg_smem<N, false>(), s>>>(raw, rc, n_lines, a);
}

cudaError_t launch_rc(const RcArgs &a, const float2 *raw, float2 *rc, int64_t n_lines, cudaStream_t s)
{
    if (n_lines <= 0) return cudaSuccess;
    // staged line kernels are persistent: at most the resident CTAs, each looping over lines
    const int64_t cap = a.max_ctas > 0 ? a.max_ctas : 1;
    const unsigned grid = (unsigned)(n_lines < cap ? n_lines : cap);
    switch (a.n) {
    case 512: launch_reg<512>(a, raw, rc, n_lines, grid, s); break;
    case 1024: launch_reg<1024>(a, raw, rc, n_lines, grid, s); break;
    case 2048: launch_reg<2048>(a, raw, rc, n_lines, grid, s); break;
    case 4096: launch_reg<4096>(a, raw, rc, n_lines, grid, s); break;
    case 8192: launch_reg<8192>(a, raw, rc, n_lines, grid, s); break;
    case 6000:
        if (a.u == 1) rc_mixed6000_kernel<false><<<grid, 200, rc_mixed_smem(false), s>>>(raw, rc, n_lines, a);
        else rc_mixed6000_kernel<true><<<grid, 200, rc_mixed_smem(true), s>>>(raw, rc, n_lines, a);
        break;
    default: rc_fused_kernel<<<grid, rc_block_threads(a.n), rc_smem_bytes(a.n, a.u), s>>>(raw, rc, n_lines, a); break;
    }
    return cudaGetLastError();
}

}  // namespace sar
