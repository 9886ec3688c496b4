/*
 * sar.h -- C ABI of the GB300 (sm_103a) SAR image-formation library: fused
 * range compression and time-domain backprojection.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Complex samples are complex64: interleaved (re, im) float32 pairs.
 *  - Device buffers are CUDA device pointers on the plan's device, 16-byte
 *    aligned, dense (no row padding).  The caller owns them; the library never
 *    frees or retains them past the call.
 *  - Every call that launches work enqueues it on `stream` (a cudaStream_t;
 *    NULL = the legacy default stream) and returns without synchronising,
 *    except where stated.  Argument errors are detected before anything is
 *    launched.  Device-side error flags (bounds checks, geometry validity)
 *    are reported by sar_plan_sync.
 *  - Errors are return codes only; nothing aborts, traps or throws.  The
 *    library prints nothing, except a trace of plan parameters, kernel
 *    choices and device flags on stderr when SAR_LOG=1 is in the environment.
 *  - A plan may be used from one host thread at a time.  Calls on different
 *    streams that share one plan are serialised by the caller.
 *
 * Geometry: x along-track, y ground range, z up (metres).  Pixel (ix, iy) sits
 * at (x0 + ix dx, y0 + iy dy, z0); images are [ny][nx], x fastest.  Antenna
 * positions are one (x, y, z) float64 triple per pulse (stop-and-go).
 */
#ifndef SAR_H
#define SAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct sar_plan_s *sar_plan;

typedef enum {
    SAR_OK = 0,
    SAR_ERR_INVALID_ARG = 1,   /* NULL, non-positive or non-finite values, misaligned pointers, bad ranges */
    SAR_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels handle (see each entry) */
    SAR_ERR_NO_MEMORY = 3,     /* a device or host allocation failed */
    SAR_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    SAR_ERR_TIMEOUT = 5,       /* a bounded device-side wait ran out */
    SAR_ERR_INTERNAL = 6       /* a device-side bounds check fired (bug) */
} sar_status;

/* Radar and sampling parameters.
 * The transmitted pulse is a baseband linear-FM up-chirp exp(j pi K t^2),
 * K = bandwidth / pulse_width, on -pulse_width/2 <= t < pulse_width/2; echoes are
 * sampled at fs starting at two-way time 2 range_start / c0.  Range compression
 * ("GPU-accelerated backprojection SAR imaging", section 3.1; "Fused FFT ->
 * filter -> IFFT for SAR on Apple Silicon", section 3.1) produces upsample x
 * oversampled compressed lines. */
typedef struct {
    double fc;            /* carrier frequency, Hz (> 0) */
    double bandwidth;     /* chirp bandwidth B, Hz (> 0) */
    double pulse_width;   /* chirp duration Tp, s (> 0); Tp * fs must not exceed n_range */
    double fs;            /* complex sampling rate, Hz (> 0) */
    double range_start;   /* slant range of sample 0, m */
    int32_t n_pulses;     /* pulses Na (>= 1) */
    int32_t n_range;      /* samples per pulse Nr: 16 <= Nr <= 8192 when even and of the form
                             2^a 3^b 5^c (mixed-radix transforms); any other 16 <= Nr <= 8192
                             (Bluestein / chirp-z transforms of length up to 16384,
                             "Ultra-high-resolution airborne SAR on CUDA", section 5.1) */
    int32_t upsample;     /* range upsampling U in {1, 2, 4, 8} */
} sar_radar;

/* The image grid of pixel centres ("GPU-accelerated backprojection SAR imaging",
 * section 3.3: pixels on a plane z = z0, mapped from thread indices). */
typedef struct {
    double x0, y0, z0;    /* position of pixel (0, 0), m */
    double dx, dy;        /* pixel spacing, m (> 0) */
    int32_t nx, ny;       /* pixels per row and rows (>= 1) */
} sar_grid;

/* Create a plan on CUDA device `device`: validates the parameters, builds the
 * matched-filter spectrum conj(DFT_Nr(chirp)) and the transform tables in
 * float64 on the host, uploads them, and allocates the plan's small device
 * state.  `grid` may be NULL for a range-compression-only plan.
 * Returns SAR_ERR_INVALID_ARG / SAR_ERR_UNSUPPORTED for bad parameters,
 * SAR_ERR_NO_MEMORY or SAR_ERR_CUDA on allocation / runtime failure.  On
 * success *out owns everything the plan allocated. */
sar_status sar_plan_create(const sar_radar *radar, const sar_grid *grid, int device, sar_plan *out);

/* Free everything the plan owns (synchronises the plan's device first).
 * NULL is accepted and ignored. */
sar_status sar_plan_destroy(sar_plan plan);

/* Bytes of caller-provided workspace sar_form_image needs: the compressed
 * lines, Na * U * Nr complex64, rounded up to 256 bytes. */
sar_status sar_workspace_size(sar_plan plan, size_t *bytes);

/* Range compression of n_lines pulses, each fused into one kernel pass
 * ("Fused FFT -> filter -> IFFT for SAR on Apple Silicon", sections 3.1-3.2;
 * "GPU-accelerated backprojection SAR imaging", section 3.1):
 *   X = DFT_Nr(raw_n); Y = X * conj(DFT_Nr(chirp)); Y zero-padded to U Nr
 *   points (bins k with 2k >= Nr at the negative-frequency end);
 *   rc_n = U * IDFT_{U Nr}(Y')   (so rc_n[U m] is the plain compressed sample m).
 * raw: device [n_lines][Nr] complex64.  rc: device [n_lines][U Nr] complex64.
 * 1 <= n_lines; raw and rc must not overlap. */
sar_status sar_range_compress(sar_plan plan, const void *raw, void *rc, int64_t n_lines, void *stream);

/* Time-domain backprojection of pulses [pulse_begin, pulse_begin + pulse_count)
 * ("GPU-accelerated backprojection SAR imaging", sections 1.1, 2.2, 3.3): for
 * every pixel p,
 *   I(p) = sum_n L_n((|p - a_n| - range_start) / dr_U) * exp(+j 4 pi fc |p - a_n| / c0)
 * with dr_U = c0 / (2 fs U), L_n the linear interpolation of compressed line n,
 * and samples outside [0, U Nr) taken as zero.  accumulate != 0 adds into image
 * instead of overwriting it.  The sum over pulses runs in float32.
 * rc: device [Na][U Nr] complex64 (full plan-sized array; lines outside the
 * pulse range are not read).  pos: device [Na][3] float64.  image: device
 * [ny][nx] complex64.  Needs a plan created with a grid; SAR_ERR_UNSUPPORTED
 * otherwise.  The kernel computes each pixel's range as a float32 offset
 * from a float64 range to the centre of its pixel tile; sar_plan_sync reports
 * SAR_ERR_UNSUPPORTED if a tile came closer to the antenna than the
 * expansion allows (range below 100 tile half-diagonals).  Tiles hold 2048
 * pixels (128 x 16, 64 x 32 or 32 x 64, the longest in x whose half-diagonal
 * stays within clamp(range_start / 150, 20 m, 32 m)), so every tile centre at
 * max(2 km, 2/3 range_start) or beyond is in range. */
sar_status sar_backproject(sar_plan plan, const void *rc, const double *pos, int32_t pulse_begin,
                           int32_t pulse_count, void *image, int accumulate, void *stream);

/* Range compression of all Na pulses into `workspace`, then backprojection of
 * all pulses into `image` (overwritten).  workspace: device, at least
 * sar_workspace_size bytes.  raw: device [Na][Nr] complex64; pos: device
 * [Na][3] float64; image: device [ny][nx] complex64. */
sar_status sar_form_image(sar_plan plan, const void *raw, const double *pos, void *image,
                          void *workspace, size_t workspace_bytes, void *stream);

/* The same image formation from HOST buffers: copies raw and pos to device
 * buffers the plan owns (allocated on the first call), forms the image and
 * copies it back to image_host, then synchronises `stream`.  From 512 pulses on
 * the pulses go in 3 growing chunks: while one is range compressed and backprojected on
 * `stream` (accumulating into the image), the next is copied on a stream the
 * plan owns, so the host-to-device copy overlaps the kernels; every other
 * chunk's kernels run on a second stream the plan owns, ordered after `stream`'s
 * earlier work, and `stream` waits for them before the read-back.  The image then
 * equals sar_form_image's up to the float32 summation order of the chunks.
 * Host buffers should be pinned for full copy bandwidth.  raw_host: [Na][Nr]
 * complex64; pos_host: [Na][3] float64; image_host: [ny][nx] complex64. */
sar_status sar_form_image_host(sar_plan plan, const void *raw_host, const double *pos_host, void *image_host,
                               void *stream);

/* Layout of compressed lines with U > 1, for sar_range_compress's output and
 * sar_backproject's input.  SAR_RC_NATURAL (the default): sample j = U m + u of
 * a line at index j.  SAR_RC_POLYPHASE: at index u Nr + m, i.e. U contiguous
 * planes of Nr samples, plane u holding the samples with j mod U = u -- each
 * of the U inverse transforms of range compression then writes one contiguous
 * plane, which halves the kernel's memory traffic compared with interleaved
 * stores.  The two layouts coincide for U = 1.  sar_form_image uses the
 * polyphase layout for its workspace regardless of this setting. */
typedef enum { SAR_RC_NATURAL = 0, SAR_RC_POLYPHASE = 1 } sar_rc_layout;

/* Set the plan's compressed-line layout (SAR_ERR_INVALID_ARG for other values). */
sar_status sar_plan_set_rc_layout(sar_plan plan, sar_rc_layout layout);

/* Image formation that allocates nothing (the pages have no counterpart: this
 * is a deployment variant of sar_form_image).  For callers that cannot call
 * cudaMalloc when they form an image -- processing loops whose device memory
 * is fixed at start-up, or hosts whose device memory belongs to an allocator
 * this library cannot use.  The compressed lines go to a 32 MiB array compiled
 * into the library, which every device that loads the library holds until the
 * process exits; the caller passes only inputs and outputs (raw, pos, image as
 * in sar_form_image).  Plans whose Na * U * Nr * 8 bytes exceed 32 MiB get
 * SAR_ERR_UNSUPPORTED before anything is launched.  The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress, once per device);
 * make that first call before any stream capture.  All calls share the one
 * array: calls whose work overlaps on the GPU (other streams, other plans)
 * race on it and must be serialised by the caller.  Nothing in it needs
 * clearing between calls. */
sar_status sar_form_image_noalloc(sar_plan plan, const void *raw, const double *pos, void *image, void *stream);

/* Synchronise `stream`, then read and clear the plan's device error flags:
 * SAR_ERR_INTERNAL if a bounds check fired, SAR_ERR_TIMEOUT if a kernel gave
 * up waiting (about 1 s) for one of its own asynchronous line copies and
 * returned early (its output is then incomplete), SAR_ERR_UNSUPPORTED if a
 * geometry validity check failed, SAR_ERR_CUDA on an asynchronous CUDA error. */
sar_status sar_plan_sync(sar_plan plan, void *stream);

/* Static, NUL-terminated description of a status code. */
const char *sar_status_string(sar_status status);

/* Number of kernel launches the last call on this plan enqueued (for
 * accounting in benchmarks); 0 for a NULL plan. */
int32_t sar_plan_last_launches(sar_plan plan);

/* Range weighting of the matched filter ("GPU-accelerated backprojection SAR
 * imaging", section 3.1: the unweighted filter leaves range sidelobes of about
 * -13 dB; weighting lowers them and widens the main lobe 1.3-1.5 times).  The
 * weight multiplies the Nchirp samples i = 0 .. Nchirp-1 of the reference chirp:
 *   SAR_WINDOW_NONE     w = 1 (the plan's default);
 *   SAR_WINDOW_HAMMING  w = 0.54 - 0.46 cos(2 pi i / (Nchirp - 1));
 *   SAR_WINDOW_TAYLOR   Taylor's distribution with taylor_nbar terms and peak
 *                       sidelobes taylor_sll_db below the main lobe, sampled at
 *                       x = (i - (Nchirp - 1)/2) / Nchirp (e.g. nbar 4, 35 dB). */
typedef enum { SAR_WINDOW_NONE = 0, SAR_WINDOW_HAMMING = 1, SAR_WINDOW_TAYLOR = 2 } sar_window;

/* Rebuild the plan's matched filter with `window` (taylor_* are read for
 * SAR_WINDOW_TAYLOR only: 2 <= taylor_nbar <= 64, 0 < taylor_sll_db <= 120;
 * SAR_ERR_INVALID_ARG otherwise).  Synchronises the device first, so that work
 * already queued keeps the filter it was queued with; later range compressions
 * (and image formations) use the new one.  SAR_ERR_CUDA if the upload fails. */
sar_status sar_plan_set_range_window(sar_plan plan, sar_window window, int32_t taylor_nbar, double taylor_sll_db);

/* Azimuth (pulse) weighting of the backprojection: with weights non-NULL, every
 * later backprojection on this plan sums weights[n] * L_n(...) * exp(...) over
 * pulses n, i.e. pulse n's compressed line scaled by a real weight (an aperture
 * taper such as Hamming or Taylor over the pulses lowers the azimuth sidelobes
 * the way range weighting lowers the range ones).  weights: device [Na] float32,
 * 4-byte aligned, owned by the caller, read by the kernels and left unchanged;
 * it must stay valid while backprojections that use it are in flight.  NULL
 * restores unit weights.  The weights are applied while the compressed samples
 * are staged, so they cost nothing per pixel.  SAR_ERR_UNSUPPORTED for a plan
 * without a grid. */
sar_status sar_plan_set_pulse_weights(sar_plan plan, const float *weights);

/* Backprojection variants.  Each option below selects another version of the
 * pixel kernel for every later backprojection (and image formation) on the
 * plan.  At most one option differs from its default at a time: setting a
 * second non-default option returns SAR_ERR_UNSUPPORTED and changes nothing
 * (reset the first to its default before).  All three return
 * SAR_ERR_INVALID_ARG for a NULL plan or an unknown value, SAR_ERR_UNSUPPORTED
 * for a plan without a grid.  None of them launches work. */

/* Accumulation of the pulse sum ("GPU-accelerated backprojection SAR imaging",
 * sections 2.2 and 4.3: float32 sums over thousands of pulses gather rounding
 * error; Kahan's compensated summation keeps it small):
 *   SAR_ACCUM_FP32         plain float32 sums in pulse order (default);
 *   SAR_ACCUM_COMPENSATED  float32 sums over each staged batch of at most 48
 *                          pulses, added into a Kahan-compensated running total,
 *                          so the rounding error grows with the batch length
 *                          rather than the pulse count. */
typedef enum { SAR_ACCUM_FP32 = 0, SAR_ACCUM_COMPENSATED = 1 } sar_accumulation;
sar_status sar_plan_set_accumulation(sar_plan plan, sar_accumulation accumulation);

/* Precision of the compressed samples staged in shared memory ("Fused FFT ->
 * filter -> IFFT for SAR on Apple Silicon", section 7, on half-precision
 * storage with single-precision arithmetic):
 *   SAR_STAGE_FP32  (tau, sigma) float32 interpolation entries (default);
 *   SAR_STAGE_FP16  each entry holds the midpoint (v_i + v_i+1)/2 and the slope
 *                   v_i+1 - v_i of the compressed line as float16, halving the
 *                   staged bytes; arithmetic stays float32.  Compressed samples
 *                   (times the pulse weights) must stay below 65504 in
 *                   magnitude, float16's largest finite value. */
typedef enum { SAR_STAGE_FP32 = 0, SAR_STAGE_FP16 = 1 } sar_stage_precision;
sar_status sar_plan_set_stage_precision(sar_plan plan, sar_stage_precision precision);

/* Interpolation of the compressed line at each pixel's range ("GPU-accelerated
 * backprojection SAR imaging", section 2.2: nearest, linear or sinc
 * interpolation, sinc being the accurate and costly choice):
 *   SAR_INTERP_LINEAR  linear between the two neighbouring samples (default);
 *   SAR_INTERP_SINC8   truncated sinc over 8 samples: with q the fractional
 *                      sample index, r = floor(q) and f = q - r, sample r + k
 *                      (k = -3 .. 4) has weight h(f - k) / sum_j h(f - j),
 *                      h(d) = sinc(d) (1 + cos(pi d / 4)) / 2 (a Hann taper
 *                      that reaches zero at the ends of the 8-sample support).
 *                      Samples outside the line count as zero. */
typedef enum { SAR_INTERP_LINEAR = 0, SAR_INTERP_SINC8 = 1 } sar_interpolation;
sar_status sar_plan_set_interpolation(sar_plan plan, sar_interpolation interpolation);

/* Range-Doppler image formation, a second image-formation path for a straight,
 * uniformly sampled track ("Fused FFT -> filter -> IFFT for SAR on Apple
 * Silicon", sections 2.1 and 5.1; "Ultra-high-resolution airborne SAR on
 * CUDA", section 2): range compression, azimuth DFT of every range bin,
 * range cell migration correction by interpolation across range bins,
 * multiplication by the azimuth matched filter, azimuth IDFT.  With dr =
 * c0 / (2 fs), du the along-track distance between pulses, m the Doppler bin
 * (m_s its signed value, the Nyquist bin negative), k_m = m_s / (Na du) and
 * D_m = sqrt(1 - (lambda k_m / 2)^2), output range bin i (R0 = range_start +
 * i dr) takes the compressed spectrum S(m, .) at range bin
 * i + R0 (1/D_m - 1) / dr (8-tap sinc interpolation, as SAR_INTERP_SINC8;
 * bins outside [0, Nr) count as zero), multiplies it by
 * exp(+j 4 pi R0 D_m / lambda) and transforms back with 1/Na:
 *   image [Nr][Na] complex64, row i = slant range R0, column n = the
 *   along-track position of pulse n.
 * A point target of complex amplitude a focuses at its closest-approach range
 * and along-track position with phase arg(a) - pi/4 (stationary phase of the
 * azimuth chirp).  The plan needs upsample 1 and n_pulses a power of two from
 * 512 to 8192 (SAR_ERR_UNSUPPORTED otherwise). */

/* Build the plan's azimuth tables for pulses `pulse_spacing` metres apart
 * (finite, > 0: SAR_ERR_INVALID_ARG otherwise; SAR_ERR_UNSUPPORTED when
 * lambda / (4 pulse_spacing) >= 1, where D_m is not real).  Synchronises the
 * device first; SAR_ERR_CUDA if an allocation or upload fails. */
sar_status sar_plan_set_range_doppler(sar_plan plan, double pulse_spacing);

/* Workspace bytes sar_range_doppler needs: 2 Na Nr 8 (the compressed lines and
 * their transpose).  SAR_ERR_UNSUPPORTED before sar_plan_set_range_doppler. */
sar_status sar_range_doppler_workspace_size(sar_plan plan, size_t *bytes);

/* Form the range-Doppler image of raw [Na][Nr] complex64 into image [Nr][Na]
 * complex64, using `workspace` (device, at least
 * sar_range_doppler_workspace_size bytes, owned by the caller, contents
 * overwritten).  Four launches on `stream`, no synchronisation.  All device
 * pointers 16-byte aligned and not overlapping.  SAR_ERR_INVALID_ARG for NULL
 * or misaligned pointers or a short workspace, SAR_ERR_UNSUPPORTED before
 * sar_plan_set_range_doppler. */
sar_status sar_range_doppler(sar_plan plan, const void *raw, void *image, void *workspace, size_t workspace_bytes,
                             void *stream);

/* Kernel timing, for benchmarks (no counterpart in the pages).  With enable != 0,
 * each later range-compression call records a pair of CUDA events on its stream
 * around the transform kernel, and each backprojection around the pixel kernel
 * alone (not its small per-tile parameter and slice-sum launches); at most
 * 4096 calls of each kind are recorded until the next read.  The events belong
 * to the plan.  enable = 0 stops recording.  Errors: SAR_ERR_INVALID_ARG for a
 * NULL plan. */
sar_status sar_plan_set_timing(sar_plan plan, int enable);

/* Wait for the recorded events, then return the summed kernel durations in
 * milliseconds and the number of calls recorded since timing was enabled or
 * last read, for range compression (rc_*) and backprojection (bp_*), and forget
 * them.  All four pointers are host pointers and must be non-NULL
 * (SAR_ERR_INVALID_ARG otherwise); SAR_ERR_CUDA if an event could not be read. */
sar_status sar_plan_kernel_times(sar_plan plan, double *rc_ms, int32_t *rc_calls, double *bp_ms, int32_t *bp_calls);

#ifdef __cplusplus
}
#endif

#endif /* SAR_H */
