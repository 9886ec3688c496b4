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
// in between exchange through one padded shared-memory buffer (one element of
// padding per 16 keeps the strided reads free of bank conflicts).  So the
// forward transform's output, the filter multiply and the inverse transforms'
// inputs never touch shared memory, and each transform costs log16(Nr) - 1
// exchanges.
// ---------------------------------------------------------------------------

__device__ __forceinline__ int pad16(int i) { return i + (i >> 4); }

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
// thread loads its 16/R butterflies from the buffer, then (after a barrier)
// writes them back transformed, or keeps them when kLast.
template <int N, int R, int L, bool kLast>
__device__ __forceinline__ void reg_pass(float2 (&x)[16], float2 *buf, const float2 *__restrict__ tw)
{
    constexpr int T = N / 16, SP = N / (L * R), NB = 16 / R;
    const int t = threadIdx.x;
#pragma unroll
    for (int i = 0; i < NB; i++) {
        const int b = t + T * i;
        const int jp = b % SP, kp = b / SP;
#pragma unroll
        for (int p = 0; p < R; p++) x[i * R + p] = buf[pad16(kp * SP * R + jp + SP * p)];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < NB; i++) {
        const int b = t + T * i;
        const int jp = b % SP, kp = b / SP;
        float2 w[R];
        twiddle_powers<R>(__ldg(tw + SP * kp), w);
#pragma unroll
        for (int p = 1; p < R; p++) x[i * R + p] = cmul(x[i * R + p], w[p]);
        Dft<R>::run(x + i * R);
        if (!kLast) {
#pragma unroll
            for (int q = 0; q < R; q++) buf[pad16((kp + L * q) * SP + jp)] = x[i * R + q];
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
template <int N>
__device__ __forceinline__ void reg_dft(float2 (&x)[16], float2 *buf, const float2 *__restrict__ tw)
{
    constexpr int T = N / 16;
    const int t = threadIdx.x;
    Dft<16>::run(x);                                            // pass 1: L = 1, no twiddles
#pragma unroll
    for (int q = 0; q < 16; q++) buf[pad16(q * T + t)] = x[q];
    __syncthreads();
    if constexpr (N == 512) {
        reg_pass<N, 16, 16, false>(x, buf, tw);
        reg_pass<N, 2, 256, true>(x, buf, tw);
    } else if constexpr (N == 1024) {
        reg_pass<N, 16, 16, false>(x, buf, tw);
        reg_pass<N, 4, 256, true>(x, buf, tw);
    } else if constexpr (N == 2048) {
        reg_pass<N, 16, 16, false>(x, buf, tw);
        reg_pass<N, 8, 256, true>(x, buf, tw);
    } else if constexpr (N == 4096) {
        reg_pass<N, 16, 16, false>(x, buf, tw);
        reg_pass<N, 16, 256, true>(x, buf, tw);
    } else {
        static_assert(N == 8192, "unsupported line length");
        reg_pass<N, 16, 16, false>(x, buf, tw);
        reg_pass<N, 16, 256, false>(x, buf, tw);
        reg_pass<N, 2, 4096, true>(x, buf, tw);
    }
    __syncthreads();                                            // the buffer is free for the next transform
}

template <int N>
__global__ void __launch_bounds__(N / 16, N == 4096 ? 2 : 1) rc_reg_kernel(const float2 *__restrict__ raw, float2 *__restrict__ rc,
                                                        int64_t n_lines, RcArgs args)
{
    extern __shared__ float4 smem4[];
    float2 *buf = reinterpret_cast<float2 *>(smem4);
    constexpr int T = N / 16;
    const int t = threadIdx.x;
    const int U = args.u;
    for (int64_t line = blockIdx.x; line < n_lines; line += gridDim.x) {
        float2 x[16], y[16];
        const float2 *src = raw + line * N;
#pragma unroll
        for (int p = 0; p < 16; p++) x[p] = __ldg(src + t + T * p);
        reg_dft<N>(x, buf, args.tw);
        // matched filter
#pragma unroll
        for (int p = 0; p < 16; p++) y[p] = cmul(x[p], __ldg(args.h + t + T * p));
        float2 *out = rc + line * (int64_t)(U * N);
        for (int u = 0; u < U; u++) {
            // y = Y exp(+j 2 pi k_s u / (U N)); inverse transform by the conjugate identity
#pragma unroll
            for (int p = 0; p < 16; p++) x[p] = cconj(y[p]);
            reg_dft<N>(x, buf, args.tw);
            if (args.planar || U == 1) {
                float2 *plane = out + (int64_t)u * N;
#pragma unroll
                for (int p = 0; p < 16; p++) plane[t + T * p] = cconj(x[p]);
            } else {
#pragma unroll
                for (int p = 0; p < 16; p++)
                    out[(int64_t)U * (t + T * p) + u] = cconj(x[p]);
            }
            if (u + 1 < U) {
#pragma unroll
                for (int p = 0; p < 16; p++) y[p] = cmul(y[p], __ldg(args.ramp + t + T * p));
            }
        }
    }
}

template <int N>
size_t rc_reg_smem() { return (size_t)(N + N / 16) * sizeof(float2); }

// ---------------------------------------------------------------------------
// Register-resident transform for Nr = 6000 = 2^4 3 5^3 (the non-power-of-two
// line of the range-only sweep): 200 threads of 30 elements, element t + T p in
// slot p (T = 200), and four Stockham passes of radix 10, 10, 10 and 6, each
// thread running 30 / R butterflies per pass.  As in the power-of-two kernel,
// the first pass reads registers, the last leaves its output in registers in
// the t + T p layout, and the passes in between exchange through shared memory.
// ---------------------------------------------------------------------------
template <int N, int E, int R, int L, bool kFirst, bool kLast>
__device__ __forceinline__ void mixed_pass(float2 (&x)[E], float2 *buf, const float2 *__restrict__ tw)
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
            for (int p = 0; p < R; p++) x[i * R + p] = buf[kp * SP * R + jp + SP * p];
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < NB; i++) {
        const int b = t + T * i;
        const int jp = b % SP, kp = b / SP;
        if (!kFirst) {
            float2 w[R];
            twiddle_powers<R>(__ldg(tw + SP * kp), w);
#pragma unroll
            for (int p = 1; p < R; p++) x[i * R + p] = cmul(x[i * R + p], w[p]);
        }
        Dft<R>::run(x + i * R);
        if (!kLast) {
#pragma unroll
            for (int q = 0; q < R; q++) buf[(kp + L * q) * SP + jp] = x[i * R + q];
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
__device__ __forceinline__ void mixed_dft6000(float2 (&x)[30], float2 *buf, const float2 *__restrict__ tw)
{
    mixed_pass<6000, 30, 10, 1, true, false>(x, buf, tw);
    mixed_pass<6000, 30, 10, 10, false, false>(x, buf, tw);
    mixed_pass<6000, 30, 10, 100, false, false>(x, buf, tw);
    mixed_pass<6000, 30, 6, 1000, false, true>(x, buf, tw);
    __syncthreads();                                            // the buffer is free for the next transform
}

constexpr int kRcMixedCtas = 1;     // the 30-element layout wants ~250 registers; bounding them to fit
                                    // 2 CTAs per SM spills and runs slower at U = 8

template <bool kMulti>
__global__ void __launch_bounds__(200, kRcMixedCtas) rc_mixed6000_kernel(const float2 *__restrict__ raw, float2 *__restrict__ rc,
                                                           int64_t n_lines, RcArgs args)
{
    constexpr int N = 6000, E = 30, T = N / E;
    extern __shared__ float4 smem4[];
    float2 *buf = reinterpret_cast<float2 *>(smem4);
    const int t = threadIdx.x;
    const int U = kMulti ? args.u : 1;
    for (int64_t line = blockIdx.x; line < n_lines; line += gridDim.x) {
        float2 x[E];
        const float2 *src = raw + line * N;
#pragma unroll
        for (int p = 0; p < E; p++) x[p] = __ldg(src + t + T * p);
        mixed_dft6000(x, buf, args.tw);
        // matched filter (with the IDFT's 1 / Nr)
#pragma unroll
        for (int p = 0; p < E; p++) x[p] = cmul(x[p], __ldg(args.h + t + T * p));
        float2 *out = rc + line * (int64_t)(U * N);
        if constexpr (!kMulti) {
#pragma unroll
            for (int p = 0; p < E; p++) x[p] = cconj(x[p]);
            mixed_dft6000(x, buf, args.tw);
#pragma unroll
            for (int p = 0; p < E; p++) out[t + T * p] = cconj(x[p]);
        } else {
            float2 y[E];
#pragma unroll
            for (int p = 0; p < E; p++) y[p] = x[p];
            for (int u = 0; u < U; u++) {
#pragma unroll
                for (int p = 0; p < E; p++) x[p] = cconj(y[p]);
                mixed_dft6000(x, buf, args.tw);
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
}

}  // namespace

int rc_block_threads(int n) { return n >= 4096 ? 512 : 256; }

size_t rc_smem_bytes(int n, int u) { return (size_t)(u == 1 ? 2 : 3) * n * sizeof(float2); }

cudaError_t rc_configure(int)
{
    // the largest supported line (8192 samples) sets the limit, so plans of any size can coexist
    cudaError_t e = cudaFuncSetAttribute(rc_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)rc_smem_bytes(8192, 2));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rc_reg_kernel<8192>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)rc_reg_smem<8192>());
    return e;
}

bool rc_has_reg_path(int n) { return n == 512 || n == 1024 || n == 2048 || n == 4096 || n == 8192; }

cudaError_t launch_rc(const RcArgs &a, const float2 *raw, float2 *rc, int64_t n_lines, cudaStream_t s)
{
    if (n_lines <= 0) return cudaSuccess;
    const int64_t max_grid = 1 << 20;
    const unsigned grid = (unsigned)(n_lines < max_grid ? n_lines : max_grid);
    switch (a.n) {
    case 512: rc_reg_kernel<512><<<grid, 512 / 16, rc_reg_smem<512>(), s>>>(raw, rc, n_lines, a); break;
    case 1024: rc_reg_kernel<1024><<<grid, 1024 / 16, rc_reg_smem<1024>(), s>>>(raw, rc, n_lines, a); break;
    case 2048: rc_reg_kernel<2048><<<grid, 2048 / 16, rc_reg_smem<2048>(), s>>>(raw, rc, n_lines, a); break;
    case 4096: rc_reg_kernel<4096><<<grid, 4096 / 16, rc_reg_smem<4096>(), s>>>(raw, rc, n_lines, a); break;
    case 8192: rc_reg_kernel<8192><<<grid, 8192 / 16, rc_reg_smem<8192>(), s>>>(raw, rc, n_lines, a); break;
    case 6000:
        if (a.u == 1) rc_mixed6000_kernel<false><<<grid, 200, 6000 * sizeof(float2), s>>>(raw, rc, n_lines, a);
        else rc_mixed6000_kernel<true><<<grid, 200, 6000 * sizeof(float2), s>>>(raw, rc, n_lines, a);
        break;
    default: rc_fused_kernel<<<grid, rc_block_threads(a.n), rc_smem_bytes(a.n, a.u), s>>>(raw, rc, n_lines, a); break;
    }
    return cudaGetLastError();
}

}  // namespace sar
