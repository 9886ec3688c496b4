// sar_internal.cuh -- declarations shared by the library's translation units
// (plan / ABI code, the range-compression kernel and the backprojection kernel).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sar.h"

namespace sar {

constexpr double kC0 = 299792458.0;
constexpr int kMaxPasses = 16;

// Device-side error flags (bit mask in the plan's error word).
enum : int {
    kDevErrBounds = 1,       // a staged-window index fell outside the window (bounds-checked build)
    kDevErrGeometry = 2,     // a tile came too close to the antenna for the range expansion
    kDevErrTimeout = 4,      // a bounded wait for an asynchronous copy ran out
};

// Longest a kernel waits for one of its own asynchronous copies before it gives up, sets
// kDevErrTimeout and returns (nanoseconds of the GPU's global timer).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// ----------------------------------------------------------- range compression
struct RcArgs {
    int n;                   // samples per line, Nr
    int u;                   // upsampling factor U
    int n_passes;            // Stockham passes of the Nr-point transform
    int radix[kMaxPasses];   // radix of each pass (product = Nr)
    int ptw_lo_bits;         // polyphase twiddle t = hi * 2^bits + lo
    const float2 *h;         // matched filter spectrum H[k] = conj(DFT_N chirp)[k] / Nr (the IDFT's
                             // scaling U * 1/(U Nr) folded in), natural order
    const float2 *tw;        // w_N^t = exp(-2 pi i t / Nr), t in [0, Nr)
    const float2 *ptw_hi;    // exp(-2 pi i (hi << bits) / (U Nr))
    const float2 *ptw_lo;    // exp(-2 pi i lo / (U Nr)), lo < 2^bits
    const float2 *ramp;      // exp(+2 pi i k_s / (U Nr)) for k in [0, Nr), k_s the signed frequency
    const float2 *twi;       // conj(w_N^t): the inverse transforms' twiddles
    int planar;              // output layout: 0 natural (sample U m + u at U m + u), 1 planes (at u Nr + m)
    // Bluestein transforms (lengths other than 2^a 3^b 5^c, or odd): bm = 0 when unused
    int bm;                  // convolution length M (a power of two >= 2 Nr - 1)
    int bm_passes;
    int bm_radix[kMaxPasses];
    const float2 *btw;       // exp(-2 pi i t / M), t in [0, M)
    const float2 *bw;        // exp(-i pi t^2 / Nr), t in [0, Nr)
    const float2 *bf;        // FFT_M of the wrapped conj(bw), divided by M
    unsigned long long wait_limit_ns;   // bound of the staged kernels' waits (kWaitLimitNs unless the
                                        // SAR_WAIT_LIMIT_NS knob sets another; 0 = test once)
    int max_ctas;            // CTAs of the line kernel resident on the whole device (its grid cap)
    int prefetch_ahead;      // lines ahead whose raw samples a line kernel asks L2 for (0: none)
    int *err;                // device error word
};

int rc_block_threads(int n);
bool rc_has_reg_path(int n);
size_t rc_smem_bytes(int n, int u);
size_t rc_bluestein_smem(int n, int u, int m);
cudaError_t rc_configure(int n);
// CTAs of the line kernel for (n, u) that fit on device `dev` at once (0 on error).
int rc_resident_ctas(int n, int u, int dev);
// Lines ahead of its own whose raw samples a one-CTA-per-line kernel prefetches into L2 (the CTAs
// resident on device `dev`, so that each CTA fetches the line of the CTA that will replace it), or 0.
int rc_prefetch_ahead(int n, int u, int dev);
cudaError_t launch_rc(const RcArgs &a, const float2 *raw, float2 *rc, int64_t n_lines, cudaStream_t s);

// ----------------------------------------------------------- range-Doppler
struct RdaArgs {
    int na, nr;              // pulses (the azimuth transform length) and range bins
    const float2 *tw;        // exp(-2 pi i t / Na), t in [0, Na)
    const float *rcm;        // [Na] 1 / D_m - 1 (range migration factor), natural Doppler order
    const float2 *phc;       // [Na] (2 / lambda)(1 - D_m) as (hi, lo) floats, turns per metre of range
    double range_start;      // m, range of bin 0
    double dr;               // m, c0 / (2 fs)
    double two_over_lambda;  // turns per metre
    float inv_na;            // 1 / Na
};

bool rd_supported_pulses(int na);
cudaError_t rd_configure();
// rc [Na][Nr] compressed lines -> (work [Nr][Na] transposed, then spectra) -> img [Nr][Na]
cudaError_t launch_rd(const RdaArgs &a, const float2 *rc, float2 *work, float2 *img, cudaStream_t s);

// ----------------------------------------------------------- backprojection
constexpr int kBpRowsPerThread = 8;   // pixel rows each thread accumulates
constexpr int kBpThreads = 256;        // threads per CTA: a tile of kBpThreads * kBpRowsPerThread pixels,
                                       // 128 x 16, 64 x 32 or 32 x 64 (x along azimuth), chosen per plan
constexpr int kBpCtasPerSm = 3;        // resident CTAs per SM the kernel is built for (registers, shared memory)
constexpr int kBpParamSlots = 9;       // float4 slots of shared memory per batch pulse: 3 batches x (2 parameters + window)
constexpr int kBpMaxSlices = 32;

// Backprojection variants (one at a time; a plan selects one with its option setters).
enum BpMode : int {
    kBpLinear = 0,           // linear interpolation, (tau, sigma) float32 entries, plain float32 sums
    kBpCompensated = 1,      // as kBpLinear, per-batch sums folded into Kahan-compensated totals
    kBpHalfStage = 2,        // linear interpolation from float16 (midpoint, slope) entries
    kBpSinc8 = 3,            // 8-tap Hann-tapered sinc interpolation of float32 samples
};
constexpr int kBpModes = 4;
// Resident CTAs per SM each variant is built for (the heavier variants need more registers).
constexpr int bp_mode_ctas(int mode) { return mode == kBpLinear || mode == kBpHalfStage ? kBpCtasPerSm : 2; }

struct BpArgs {
    // grid
    double x0, y0, z0;
    double dx, dy;           // pixel spacing (float64: tile centres must not inherit float32 rounding)
    float dxf, dyf;          // the same spacing in float32, for offsets inside a tile
    int nx, ny, tiles_x, tiles_y;
    int tile_w, tile_h;      // tile shape in pixels (tile_w * tile_h = kBpThreads * kBpRowsPerThread)
    // range axis
    double range_start;      // m
    double inv_dr;           // 1 / dr_U (bins per metre)
    float dr;                // dr_U, m
    int n_samples;           // U * Nr
    // phase: exp(+j 2 pi [ (2/lambda) R_start + kappa Q ]) for a fractional global bin Q
    double phase0_turns;     // frac((2 / lambda) * range_start)
    double kappa;            // 2 dr_U / lambda, turns per bin
    float two_pi_kappa;      // 2 pi kappa (rad per bin)
    // staged window: entries e in [0, w) hold local bins i = e - wh
    int wh, w;               // every pixel of a tile reads entries within [0, w) of its pulse's window
    int pulses_per_batch;    // parameter slots per batch (the batch may be smaller)
    int stage_bytes;         // shared memory for raw and staged rows of one batch
    float min_range_tiles;   // geometry validity: range >= this (m) per tile
    // pulse slicing: slice s of gridDim.z sums pulses [pulse_begin + s * slice_len, ...) into
    // partial + s * nx * ny (or straight into image when there is one slice)
    int slice_len;
    float2 *partial;
    // per (tile, pulse) parameters written by the prep kernel: 3 float4 per entry
    float4 *table;
    // double-float (hi, lo) copies of the float64 constants the prep kernel needs
    float2 x0s, y0s, z0s, dxs, dys, rss, idrs, ph0s, kps;
    // data
    const float2 *rc;        // [Na][U Nr], natural order or polyphase planes (planar != 0)
    int planar, u_shift, u_mask, n_range;   // planes: sample I of a line at (I & u_mask) Nr + (I >> u_shift)
    const double *pos;       // [Na][3]
    const float *weights;    // [Na] real pulse weights, or null for 1
    int mode;                // BpMode
    float2 *image;           // [ny][nx]
    int pulse_begin, pulse_end;
    int accumulate;
    int *err;                // device error word
};

size_t bp_smem_bytes(const BpArgs &a);
cudaError_t bp_configure(int smem_bytes);
int bp_ctas_per_sm(int smem_bytes, int mode);
// main_begin / main_end (may be null): events recorded on s right around the pixel kernel.
// image_wait (may be null): s waits for it right before the first launch that writes the image
// (the slice sum, or the pixel kernel itself without slices); image_done (may be null) is
// recorded on s right after that launch.  Two calls on different streams over disjoint pulses,
// tables and partial images then overlap everywhere but in their writes of the image.
cudaError_t launch_bp(const BpArgs &a, int slices, bool check_bounds, cudaStream_t s,
                      cudaEvent_t main_begin = nullptr, cudaEvent_t main_end = nullptr,
                      cudaEvent_t image_wait = nullptr, cudaEvent_t image_done = nullptr);

}  // namespace sar
