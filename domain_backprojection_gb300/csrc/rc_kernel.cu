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
// Kernels by line length Nr (launch_rc picks one):
//   - rc_reg_kernel<N, U>1>: powers of two 512 .. 8192 (8192 only with upsampling),
//     register-resident radix-16 transforms (fft_reg.cuh); 8192-point lines staged by
//     bulk copy;
//   - rc_reg32_kernel: Nr = 8192 without upsampling, 32 elements per thread;
//   - rc_mixed6000_kernel<U>1>: Nr = 6000, register-resident radix 10/10/10/6;
//   - rc_fused_kernel: other even 2^a 3^b 5^c lengths, mixed-radix Stockham passes
//     (16, 8, 5, 4, 3, 2) between two shared-memory buffers, the spectrum in a third;
//   - rc_blue_reg_kernel<M> (U = 1) and rc_bluestein_kernel (U > 1): any other
//     length up to 4096, as Bluestein transforms of a power-of-two length M;
//     rc_blue32_kernel: any other length from 4097 to 8192 (M = 16384).
#include "fft_reg.cuh"

namespace sar {
namespace {

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

// Full forward n-point transform (passes of the given radices, twiddles w_n^t),
// ping-ponging between a and b; returns the buffer that holds the natural-order
// result.
__device__ float2 *dft_forward_len(float2 *a, float2 *b, int n, int n_passes, const int *radix,
                                   const float2 *__restrict__ tw)
{
    int L = 1;
    for (int s = 0; s < n_passes; s++) {
        const int r = radix[s];
        switch (r) {
        case 16: stockham_pass<16>(a, b, n, L, tw); break;
        case 8: stockham_pass<8>(a, b, n, L, tw); break;
        case 5: stockham_pass<5>(a, b, n, L, tw); break;
        case 4: stockham_pass<4>(a, b, n, L, tw); break;
        case 3: stockham_pass<3>(a, b, n, L, tw); break;
        default: stockham_pass<2>(a, b, n, L, tw); break;
        }
        __syncthreads();
        float2 *t = a;
        a = b;
        b = t;
        L *= r;
    }
    return a;
}

__device__ float2 *dft_forward(float2 *a, float2 *b, const RcArgs &args)
{
    return dft_forward_len(a, b, args.n, args.n_passes, args.radix, args.tw);
}

// Forward N-point DFT of the N values at `in` (in == A or in == B) by Bluestein's chirp-z
// identity jk = (j^2 + k^2 - (k - j)^2) / 2 ("Ultra-high-resolution airborne SAR on CUDA",
// section 5.1): with w_t = exp(-i pi t^2 / N),
//     X[k] = w_k sum_j (x_j w_j) conj(w_{k-j}),
// a linear convolution evaluated as an M-point circular one (M >= 2N - 1, a power of two):
// FFT_M of the zero-padded x w, times Bf = FFT_M(conj w, wrapped) / M (a plan table), then the
// inverse transform by the conjugate identity.  Returns the buffer (A or B) whose first N entries
// hold X in natural order.
__device__ float2 *bluestein_forward(const float2 *in, float2 *A, float2 *B, const RcArgs &args)
{
    const int n = args.n, m = args.bm;
    for (int j = threadIdx.x; j < m; j += blockDim.x)
        A[j] = j < n ? cmul(in[j], __ldg(args.bw + j)) : make_float2(0.0f, 0.0f);
    __syncthreads();
    float2 *P = dft_forward_len(A, B, m, args.bm_passes, args.bm_radix, args.btw);
    for (int k = threadIdx.x; k < m; k += blockDim.x) P[k] = cconj(cmul(P[k], __ldg(args.bf + k)));
    __syncthreads();
    float2 *Q = dft_forward_len(P, P == A ? B : A, m, args.bm_passes, args.bm_radix, args.btw);
    for (int k = threadIdx.x; k < n; k += blockDim.x) Q[k] = cmul(cconj(Q[k]), __ldg(args.bw + k));
    __syncthreads();
    return Q;
}

// Range compression of lines whose length N has prime factors other than 2, 3 and 5 (or is odd),
// N <= 4096: every N-point transform of the fused kernel below runs as a Bluestein transform of
// length M.  Shared memory: two M-entry buffers, plus the N-entry filtered spectrum when U > 1.
// Plain 8-byte accesses (odd N leaves lines 8-byte aligned only).
__global__ void __launch_bounds__(512) rc_bluestein_kernel(const float2 *__restrict__ raw, float2 *__restrict__ rc,
                                                           int64_t n_lines, RcArgs args)
{
    extern __shared__ float4 smem4[];
    float2 *sm = reinterpret_cast<float2 *>(smem4);
    const int n = args.n, U = args.u, m = args.bm;
    float2 *A = sm, *B = sm + m, *Y = sm + 2 * m;
    const int un = U * n;
    const int lo_mask = (1 << args.ptw_lo_bits) - 1;
    for (int64_t line = blockIdx.x; line < n_lines; line += gridDim.x) {
        const float2 *src = raw + line * n;
        for (int j = threadIdx.x; j < n; j += blockDim.x) A[j] = __ldg(src + j);
        __syncthreads();
        float2 *X = bluestein_forward(A, A, B, args);
        float2 *out = rc + line * (int64_t)un;
        if (U == 1) {
            for (int k = threadIdx.x; k < n; k += blockDim.x) X[k] = cconj(cmul(X[k], __ldg(args.h + k)));
            __syncthreads();
            const float2 *Z = bluestein_forward(X, A, B, args);
            for (int j = threadIdx.x; j < n; j += blockDim.x) out[j] = cconj(Z[j]);
            __syncthreads();
            continue;
        }
        for (int k = threadIdx.x; k < n; k += blockDim.x) Y[k] = cmul(X[k], __ldg(args.h + k));
        __syncthreads();
        for (int u = 0; u < U; u++) {
            // conj(Z_u)[k] = conj(Y[k]) * exp(-j 2 pi k_s u / (U Nr)), as in rc_fused_kernel
            for (int k = threadIdx.x; k < n; k += blockDim.x) {
                float2 z = cconj(Y[k]);
                if (u != 0) {
                    const int ks = (2 * k >= n) ? k - n : k;
                    int t = (ks * u) % un;
                    if (t < 0) t += un;
                    z = cmul(z, cmul(__ldg(args.ptw_hi + (t >> args.ptw_lo_bits)), __ldg(args.ptw_lo + (t & lo_mask))));
                }
                A[k] = z;
            }
            __syncthreads();
            const float2 *Z = bluestein_forward(A, A, B, args);
            if (args.planar) {
                for (int j = threadIdx.x; j < n; j += blockDim.x) out[(int64_t)u * n + j] = cconj(Z[j]);
            } else {
                for (int j = threadIdx.x; j < n; j += blockDim.x) out[(int64_t)U * j + u] = cconj(Z[j]);
            }
            __syncthreads();
        }
    }
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

// Resident CTAs per SM each line kernel is built for: the register budget that __launch_bounds__
// enforces.  16 warps per SM for short lines; 4 CTAs (64 registers, no spills) for 4096-point lines
// without upsampling (no copy of the spectrum to keep; measured on GB300: 0.0759 ms for 4096 lines
// against 0.0813 ms at 3 CTAs), 2 with it; one 16-warp CTA for 8192-point lines.
template <int N, bool kMulti>
__host__ __device__ constexpr int rc_reg_min_ctas()
{
    return N == 8192 ? 1 : N == 4096 ? (kMulti ? 2 : 4) : (16 * 32) / (N / 16);
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
        // with upsampling, passes with at most four butterfly columns per warp read their twiddle
        // powers from the table (measured on GB300 at 4096 points, U = 8: 0.369 -> 0.357 ms; without
        // upsampling the same change was slower, and at 8192 points it spills)
        reg_dft<N, rc_reg_two_buffers<N, kMulti>(), (N < 8192)>(x, a, b, args.tw);
        // matched filter (with the IDFT's 1 / Nr)
        float2 y[16];
#pragma unroll
        for (int p = 0; p < 16; p++) y[p] = cmul(x[p], __ldg(args.h + t + T * p));
        for (int u = 0; u < U; u++) {
            // y = Y exp(+j 2 pi k_s u / (U N)), then its inverse transform (conjugated twiddles)
#pragma unroll
            for (int p = 0; p < 16; p++) x[p] = y[p];
            reg_dft<N, rc_reg_two_buffers<N, kMulti>(), (N < 8192), true>(x, a, b, args.twi);
            if (args.planar) {
                float2 *plane = out + (int64_t)u * N;
#pragma unroll
                for (int p = 0; p < 16; p++) plane[t + T * p] = x[p];
            } else {
#pragma unroll
                for (int p = 0; p < 16; p++) out[(int64_t)U * (t + T * p) + u] = x[p];
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
            const uint32_t ph = parity;
            const bool ok = stage_wait(bar, ph, args.wait_limit_ns);
            parity ^= 1u;
            float2 x[16];
#pragma unroll
            for (int p = 0; p < 16; p++) x[p] = stage[t + T * p];
            if (__syncthreads_or(!ok)) {                        // the stage is free again (or the copy never came)
                if (t == 0) {
                    atomicOr(args.err, kDevErrTimeout);
                    stage_wait(bar, ph, kWaitLimitNs);          // let the copy in flight land before the CTA exits
                }
                return;
            }
            if (t == 0 && line + gridDim.x < n_lines)
                stage_line(bar, stage, raw + (line + gridDim.x) * N, N * sizeof(float2));
            rc_reg_line<N, kMulti>(x, a, b, rc + line * line_elems, args);
        }
    }
}

// ---------------------------------------------------------------------------
// Register-resident transforms with E elements per thread, element t + T p in
// slot p (T = N / E), each thread running E / R butterflies per pass:
//   - Nr = 6000 = 2^4 3 5^3 (the non-power-of-two line of the range-only sweep):
//     200 threads of 30 elements, four passes of radix 10, 10, 10 and 6;
//   - Nr = 8192 without upsampling: 256 threads of 32 elements, three passes of
//     radix 16, 16 and 32 (two exchanges, against three for 16 elements per
//     thread).
// As in the 16-element kernel, the first pass reads registers, the last leaves
// its output in registers in the t + T p layout, and the passes in between
// exchange through shared memory.  kPad32 adds one entry of padding per 32 to
// the exchange indices, which keeps the radix-32 pass's stride-32 reads free of
// bank conflicts.
// ---------------------------------------------------------------------------
template <bool kPad32>
__device__ __forceinline__ int xpad(int i) { return kPad32 ? i + (i >> 5) : i; }

template <int N, int E, int R, int L, bool kFirst, bool kLast, bool kOneBuf, bool kPad32 = false>
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
            for (int p = 0; p < R; p++) x[i * R + p] = src[xpad<kPad32>(kp * SP * R + jp + SP * p)];
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
            for (int q = 0; q < R; q++) dst[xpad<kPad32>((kp + L * q) * SP + jp)] = x[i * R + q];
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
            const uint32_t ph = parity;
            const bool ok = stage_wait(bar, ph, args.wait_limit_ns);
            parity ^= 1u;
            float2 x[E];
#pragma unroll
            for (int p = 0; p < E; p++) x[p] = stage[t + T * p];
            if (__syncthreads_or(!ok)) {
                if (t == 0) {
                    atomicOr(args.err, kDevErrTimeout);
                    stage_wait(bar, ph, kWaitLimitNs);          // let the copy in flight land before the CTA exits
                }
                return;
            }
            if (t == 0 && line + gridDim.x < n_lines)
                stage_line(bar, stage, raw + (line + gridDim.x) * N, N * sizeof(float2));
            rc_mixed_line<kMulti>(x, a, b, rc + line * line_elems, args);
        }
    }
}

// 8192-point lines without upsampling: 256 threads of 32 elements (one CTA per line, 2 per SM at
// 128 registers), passes of radix 16, 16 and 32 with two exchanges through one padded buffer, the
// inverse transform by the conjugate identity (one copy of the transform code in a two-trip loop).
// Measured on GB300, 4096 lines: 0.167 ms against 0.191 ms for 512 threads of 16 elements (three
// exchanges, one 16-warp CTA per SM with bulk-copy staging).  Each CTA asks L2 for the line of the
// CTA that will take its place (args.prefetch_ahead lines on, the kernel's resident CTAs): the
// load of a new line then finds its data in L2 (0.174 -> 0.167 ms).
constexpr int kRc8192Threads = 256, kRc8192Elems = 32;

__host__ __device__ constexpr size_t rc8192_smem() { return (size_t)(8192 + 8192 / 32) * sizeof(float2); }

__global__ void __launch_bounds__(kRc8192Threads, 2)
    rc_reg32_kernel(const float2 *__restrict__ raw, float2 *__restrict__ rc, int64_t n_lines, RcArgs args)
{
    constexpr int N = 8192, E = kRc8192Elems, T = kRc8192Threads;
    extern __shared__ float4 smem4[];
    float2 *buf = reinterpret_cast<float2 *>(smem4);
    const int t = threadIdx.x;
    for (int64_t line = blockIdx.x; line < n_lines; line += gridDim.x) {
        const int64_t ahead = line + args.prefetch_ahead;
        if (ahead < n_lines) {
            // two 128-byte lines per thread cover the 64 KB raw line
            const float2 *q = raw + ahead * N + 16 * t;
            asm volatile("prefetch.global.L2 [%0];" ::"l"(q));
            asm volatile("prefetch.global.L2 [%0];" ::"l"(q + 16 * T));
        }
        float2 x[E];
        const float2 *src = raw + line * N;
#pragma unroll
        for (int p = 0; p < E; p++) x[p] = ld_raw(src + t + T * p);
#pragma unroll 1
        for (int trip = 0; trip < 2; trip++) {
            mixed_pass<N, E, 16, 1, true, false, true, true>(x, nullptr, buf, args.tw);
            mixed_pass<N, E, 16, 16, false, false, true, true>(x, buf, buf, args.tw);
            mixed_pass<N, E, 32, 256, false, true, true, true>(x, buf, nullptr, args.tw);
            __syncthreads();                                    // the buffer is free for the next transform
            if (trip == 0) {
                // filter (with the IDFT's 1 / Nr) and conjugate
#pragma unroll
                for (int p = 0; p < E; p++) x[p] = cconj(cmul(x[p], __ldg(args.h + t + T * p)));
            }
        }
        float2 *out = rc + line * N;
#pragma unroll
        for (int p = 0; p < E; p++) out[t + T * p] = cconj(x[p]);
    }
}

// Bluestein lines without upsampling, register-resident: the four M-point transforms of a line
// (M = 512 .. 8192) are reg_dft passes over the thread's 16 elements t + T p (T = M / 16), the
// line's samples in the first N positions.
// 2 CTAs of 512 threads at M = 8192 (64 registers, a small spill): 4096 lines of 4094 samples
// 0.4215 -> 0.3876 ms against one CTA.
template <int M>
constexpr int rc_blue_min_ctas() { return M >= 8192 ? 2 : M == 4096 ? 2 : (16 * 32) / (M / 16); }

template <int M>
__global__ void __launch_bounds__(M / 16, rc_blue_min_ctas<M>())
    rc_blue_reg_kernel(const float2 *__restrict__ raw, float2 *__restrict__ rc, int64_t n_lines, RcArgs args)
{
    extern __shared__ float4 smem4[];
    constexpr int T = M / 16;
    float2 *a = reinterpret_cast<float2 *>(smem4), *b = a;
    const int t = threadIdx.x, n = args.n;
    for (int64_t line = blockIdx.x; line < n_lines; line += gridDim.x) {
        const float2 *src = raw + line * n;
        float2 x[16];
#pragma unroll
        for (int p = 0; p < 16; p++) {
            const int k = t + T * p;
            x[p] = k < n ? cmul(__ldg(src + k), __ldg(args.bw + k)) : make_float2(0.0f, 0.0f);
        }
        // four transforms, one copy of the transform code: after transforms 0 and 2 the convolution
        // spectrum is multiplied by Bf (and conjugated for the inverse), after transform 1 the line's
        // spectrum X is filtered and prepared for the inverse Bluestein transform
#pragma unroll 1
        for (int trip = 0; trip < 4; trip++) {
            reg_dft<M, false>(x, a, b, args.btw);
            if (trip == 1) {
#pragma unroll
                for (int p = 0; p < 16; p++) {
                    const int k = t + T * p;
                    if (k < n) {
                        const float2 w = __ldg(args.bw + k);
                        const float2 X = cmul(w, cconj(x[p]));                   // spectrum bin k
                        x[p] = cmul(cconj(cmul(X, __ldg(args.h + k))), w);      // conj(X H) w
                    } else {
                        x[p] = make_float2(0.0f, 0.0f);
                    }
                }
            } else if (trip != 3) {
#pragma unroll
                for (int p = 0; p < 16; p++) x[p] = cconj(cmul(x[p], __ldg(args.bf + t + T * p)));
            }
        }
        float2 *out = rc + line * (int64_t)n;
#pragma unroll
        for (int p = 0; p < 16; p++) {
            const int k = t + T * p;
            if (k < n) out[k] = cconj(cmul(__ldg(args.bw + k), cconj(x[p])));
        }
    }
}

template <int M>
size_t rc_blue_reg_smem() { return (size_t)(M + M / 16) * sizeof(float2); }

// Bluestein lines of 4097 .. 8192 samples, both without and with upsampling (convolution length
// M = 16384): 512 threads of 32 elements, element t + T p in slot p (T = 512), M-point transforms
// of radix 32, 16 and 32 with two exchanges through one padded buffer (135 KB, one CTA per SM).
// Without upsampling four transforms per line, as in rc_blue_reg_kernel.  With upsampling the
// filtered spectrum Y waits in shared memory (each thread reads back only its own bins) and every
// polyphase component u runs one forward Bluestein transform of conj(Y) exp(-j 2 pi k_s u / (U Nr)),
// as in rc_bluestein_kernel.
constexpr int kBlue32M = 16384, kBlue32Threads = 512, kBlue32Elems = 32;

__host__ __device__ constexpr size_t rc_blue32_smem(bool multi)
{
    return (size_t)(kBlue32M + kBlue32M / 32) * sizeof(float2) + (multi ? (size_t)8192 * sizeof(float2) : 0);
}

// forward M-point DFT of the elements held as x[p] = element t + T p; result in the same layout
__device__ __forceinline__ void blue32_dft(float2 (&x)[kBlue32Elems], float2 *buf, const float2 *__restrict__ tw)
{
    constexpr int M = kBlue32M, E = kBlue32Elems;
    mixed_pass<M, E, 32, 1, true, false, true, true>(x, nullptr, buf, tw);
    mixed_pass<M, E, 16, 32, false, false, true, true>(x, buf, buf, tw);
    mixed_pass<M, E, 32, 512, false, true, true, true>(x, buf, nullptr, tw);
    __syncthreads();                                            // the buffer is free for the next transform
}

// x <- conj(x Bf): the convolution with the chirp, ready for the transform that inverts it
__device__ __forceinline__ void blue32_filter(float2 (&x)[kBlue32Elems], const RcArgs &args)
{
#pragma unroll
    for (int p = 0; p < kBlue32Elems; p++) x[p] = cconj(cmul(x[p], __ldg(args.bf + threadIdx.x + kBlue32Threads * p)));
}

template <bool kMulti>
__global__ void __launch_bounds__(kBlue32Threads, 1)
    rc_blue32_kernel(const float2 *__restrict__ raw, float2 *__restrict__ rc, int64_t n_lines, RcArgs args)
{
    constexpr int T = kBlue32Threads, E = kBlue32Elems;
    extern __shared__ float4 smem4[];
    float2 *buf = reinterpret_cast<float2 *>(smem4);
    float2 *ysm = buf + kBlue32M + kBlue32M / 32;              // [Nr] filtered spectrum (with upsampling)
    const int t = threadIdx.x, n = args.n;
    const int U = kMulti ? args.u : 1, un = U * n;
    const int lo_mask = (1 << args.ptw_lo_bits) - 1;
    // z_u = conj(Y) exp(-j 2 pi k_s u / (U Nr)) bw, the input of component u's forward transform
    auto component_input = [&](float2 (&x)[E], int u) {
#pragma unroll
        for (int p = 0; p < E; p++) {
            const int k = t + T * p;
            float2 z = make_float2(0.0f, 0.0f);
            if (k < n) {
                z = cconj(ysm[k]);
                if (u != 0) {
                    const int ks = (2 * k >= n) ? k - n : k;
                    int tt = (ks * u) % un;
                    if (tt < 0) tt += un;
                    z = cmul(z, cmul(__ldg(args.ptw_hi + (tt >> args.ptw_lo_bits)), __ldg(args.ptw_lo + (tt & lo_mask))));
                }
                z = cmul(z, __ldg(args.bw + k));
            }
            x[p] = z;
        }
    };
    for (int64_t line = blockIdx.x; line < n_lines; line += gridDim.x) {
        const float2 *src = raw + line * n;
        float2 *out = rc + line * (int64_t)un;
        float2 x[E];
#pragma unroll
        for (int p = 0; p < E; p++) {
            const int k = t + T * p;
            x[p] = k < n ? cmul(__ldg(src + k), __ldg(args.bw + k)) : make_float2(0.0f, 0.0f);
        }
        // one copy of the transform code: every Bluestein transform is two M-point transforms with
        // the chirp filter between them (even trips); after the odd trips the line's spectrum is
        // filtered (trip 1), or a result is stored (later odd trips)
        const int trips = kMulti ? 2 + 2 * U : 4;
#pragma unroll 1
        for (int trip = 0; trip < trips; trip++) {
            blue32_dft(x, buf, args.btw);
            if ((trip & 1) == 0) {
                blue32_filter(x, args);
            } else if (trip == 1) {
                // X[k] = bw[k] conj(x[k]); Y = X H
#pragma unroll
                for (int p = 0; p < E; p++) {
                    const int k = t + T * p;
                    if (k < n) {
                        const float2 w = __ldg(args.bw + k);
                        const float2 y = cmul(cmul(w, cconj(x[p])), __ldg(args.h + k));
                        if constexpr (kMulti) ysm[k] = y;
                        else x[p] = cmul(cconj(y), w);              // conj(Y) bw: the inverse transform's input
                    } else {
                        x[p] = make_float2(0.0f, 0.0f);
                    }
                }
                if constexpr (kMulti) component_input(x, 0);
            } else {
                // a finished inverse transform: sample U m + u = conj(bw conj(x)) = x conj(bw)
                const int u = kMulti ? (trip - 3) / 2 : 0;
#pragma unroll
                for (int p = 0; p < E; p++) {
                    const int k = t + T * p;
                    if (k < n) {
                        const float2 v = cmul(x[p], cconj(__ldg(args.bw + k)));
                        if (!kMulti || args.planar) out[(int64_t)u * n + k] = v;
                        else out[(int64_t)U * k + u] = v;
                    }
                }
                if (kMulti && u + 1 < U) component_input(x, u + 1);
            }
        }
    }
}

}  // namespace

int rc_block_threads(int n) { return n >= 4096 ? 512 : 256; }

size_t rc_smem_bytes(int n, int u) { return (size_t)(u == 1 ? 2 : 3) * n * sizeof(float2); }

size_t rc_bluestein_smem(int n, int u, int m) { return (2 * (size_t)m + (u > 1 ? (size_t)n : 0)) * sizeof(float2); }

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
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rc_bluestein_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)rc_bluestein_smem(4096, 2, 8192));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rc_blue_reg_kernel<4096>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)rc_blue_reg_smem<4096>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rc_blue_reg_kernel<8192>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)rc_blue_reg_smem<8192>());
    if (e == cudaSuccess) e = set_reg_smem<512, false>();
    if (e == cudaSuccess) e = set_reg_smem<512, true>();
    if (e == cudaSuccess) e = set_reg_smem<1024, false>();
    if (e == cudaSuccess) e = set_reg_smem<1024, true>();
    if (e == cudaSuccess) e = set_reg_smem<2048, false>();
    if (e == cudaSuccess) e = set_reg_smem<2048, true>();
    if (e == cudaSuccess) e = set_reg_smem<4096, false>();
    if (e == cudaSuccess) e = set_reg_smem<4096, true>();
    if (e == cudaSuccess) e = set_reg_smem<8192, true>();
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rc_reg32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rc8192_smem());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rc_blue32_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)rc_blue32_smem(false));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rc_blue32_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)rc_blue32_smem(true));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rc_mixed6000_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)rc_mixed_smem(false));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(rc_mixed6000_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)rc_mixed_smem(true));
    return e;
}

int rc_prefetch_ahead(int n, int u, int dev)
{
    if (n == 8192 && u == 1) return resident(rc_reg32_kernel, kRc8192Threads, rc8192_smem(), dev);
    return 0;
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
    case 8192: return multi ? reg_resident<8192, true>(dev) : 1 << 20;    // U = 1: one CTA per line
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
    else if constexpr (N != 8192) rc_reg_kernel<N, false><<<grid, N / 16, rc_reg_smem<N, false>(), s>>>(raw, rc, n_lines, a);
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
    case 8192:
        if (a.u == 1) rc_reg32_kernel<<<grid, kRc8192Threads, rc8192_smem(), s>>>(raw, rc, n_lines, a);
        else launch_reg<8192>(a, raw, rc, n_lines, grid, s);
        break;
    case 6000:
        if (a.u == 1) rc_mixed6000_kernel<false><<<grid, 200, rc_mixed_smem(false), s>>>(raw, rc, n_lines, a);
        else rc_mixed6000_kernel<true><<<grid, 200, rc_mixed_smem(true), s>>>(raw, rc, n_lines, a);
        break;
    default:
        if (a.bm == kBlue32M) {
            if (a.u == 1) rc_blue32_kernel<false><<<grid, kBlue32Threads, rc_blue32_smem(false), s>>>(raw, rc, n_lines, a);
            else rc_blue32_kernel<true><<<grid, kBlue32Threads, rc_blue32_smem(true), s>>>(raw, rc, n_lines, a);
        } else if (a.bm > 0 && a.u == 1) {
            switch (a.bm) {
            case 512: rc_blue_reg_kernel<512><<<grid, 32, rc_blue_reg_smem<512>(), s>>>(raw, rc, n_lines, a); break;
            case 1024: rc_blue_reg_kernel<1024><<<grid, 64, rc_blue_reg_smem<1024>(), s>>>(raw, rc, n_lines, a); break;
            case 2048: rc_blue_reg_kernel<2048><<<grid, 128, rc_blue_reg_smem<2048>(), s>>>(raw, rc, n_lines, a); break;
            case 4096: rc_blue_reg_kernel<4096><<<grid, 256, rc_blue_reg_smem<4096>(), s>>>(raw, rc, n_lines, a); break;
            default: rc_blue_reg_kernel<8192><<<grid, 512, rc_blue_reg_smem<8192>(), s>>>(raw, rc, n_lines, a); break;
            }
        } else if (a.bm > 0)
            rc_bluestein_kernel<<<grid, 512, rc_bluestein_smem(a.n, a.u, a.bm), s>>>(raw, rc, n_lines, a);
        else
            rc_fused_kernel<<<grid, rc_block_threads(a.n), rc_smem_bytes(a.n, a.u), s>>>(raw, rc, n_lines, a);
        break;
    }
    return cudaGetLastError();
}

}  // namespace sar
