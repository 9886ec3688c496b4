// sar_api.cu -- the C ABI declared in include/sar.h: plan creation (argument
// validation, matched-filter and transform tables in float64 on the host),
// range compression, backprojection and image formation entry points.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <utility>
#include <vector>

#include "sar_internal.cuh"

struct sar_plan_s {
    int device = 0;
    sar_radar radar{};
    sar_grid grid{};
    bool has_grid = false;
    bool check_bounds = false;
    int rc_layout = SAR_RC_NATURAL;
    // range compression
    sar::RcArgs rc{};
    float2 *d_tables = nullptr;       // H | tw | ptw_hi | ptw_lo | ramp | twi in one allocation
    float2 *d_blue = nullptr;         // Bluestein tables (lengths the mixed-radix kernels do not take)
    // backprojection
    sar::BpArgs bp{};
    int bp_slots = 1;                 // CTAs of bp_kernel resident on the whole device at once
    int sms = 1;                      // multiprocessors of the plan's device
    int bp_max_slices = 1;            // pulse slices the partial-image buffer can hold
    float2 *d_partial = nullptr;      // [bp_max_slices][ny][nx] partial images
    float4 *d_table = nullptr;        // [tiles][n_pulses] x 48 B per-(tile, pulse) parameters
    // range-Doppler (sar_plan_set_range_doppler): azimuth twiddles | phase coefficients | migration factors
    sar::RdaArgs rd{};
    void *d_rd_tables = nullptr;
    bool rd_ready = false;
    // device error word and its pinned host mirror
    int *d_err = nullptr;
    int *h_err = nullptr;
    // buffers for the host-pointer entry point (allocated on first use)
    void *d_raw = nullptr, *d_pos = nullptr, *d_rc = nullptr, *d_img = nullptr;
    cudaStream_t copy_stream = nullptr;    // host path: host-to-device copies, overlapped with compute
    cudaEvent_t host_ev[5] = {};           // host path: call entry, then one per pulse chunk copied
    cudaStream_t aux_stream = nullptr;     // host path: every other pulse chunk's kernels
    cudaEvent_t img_ev[4] = {};            // host path: one per chunk, its last write of the image
    float2 *d_partial2 = nullptr;          // host path: the aux stream's partial images
    int32_t last_launches = 0;
    // kernel timing (sar_plan_set_timing): event pairs around the main kernel of each call
    bool timing = false;
    std::vector<cudaEvent_t> ev_pool;           // created on demand, destroyed with the plan
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> ev_rc, ev_bp;
    size_t ev_used = 0;
};

namespace {

using sar::kC0;

struct DeviceGuard {
    int prev = -1;
    cudaError_t status = cudaSuccess;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) status = cudaSetDevice(dev);
    }
    ~DeviceGuard()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

bool finite_pos(double v) { return std::isfinite(v) && v > 0.0; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Optional trace on stderr (SAR_LOG=1 in the environment when the library first logs): plan
// parameters and the kernels chosen, device-side flags.  Silent otherwise.
void sar_log(const char *fmt, ...)
{
    static const int on = [] {
        const char *v = std::getenv("SAR_LOG");
        return v && v[0] == '1' ? 1 : 0;
    }();
    if (!on) return;
    va_list ap;
    va_start(ap, fmt);
    std::fputs("[sar] ", stderr);
    std::vfprintf(stderr, fmt, ap);
    std::fputc('\n', stderr);
    va_end(ap);
}

// Fault-injection hook for tests: with SAR_INJECT_ALLOC_FAILURE=1 in the environment every device
// allocation the library makes reports cudaErrorMemoryAllocation without calling CUDA, so the
// SAR_ERR_NO_MEMORY paths (and the clean-up behind them) run on any machine.
cudaError_t dev_alloc(void **p, size_t bytes)
{
    const char *inj = std::getenv("SAR_INJECT_ALLOC_FAILURE");
    if (inj && inj[0] == '1') {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaMalloc(p, bytes);
}
template <typename T>
cudaError_t dev_alloc(T **p, size_t bytes)
{
    void *v = nullptr;
    const cudaError_t e = dev_alloc(&v, bytes);
    *p = static_cast<T *>(v);
    return e;
}

bool factor_235(int n)
{
    for (int p : {2, 3, 5})
        while (n % p == 0) n /= p;
    return n == 1;
}

// Radix sequence for the Stockham passes: 16s first, then 8, 4, 5, 3, 2.
int plan_radices(int n, int *radix)
{
    int np = 0;
    while (n % 16 == 0 && n > 16) { radix[np++] = 16; n /= 16; }
    for (int r : {16, 8, 4, 5, 3, 2})
        while (n % r == 0 && n > 1) { radix[np++] = r; n /= r; }
    return np;
}

// Lines the mixed-radix kernels transform directly: even, 2^a 3^b 5^c, up to 8192 samples.  Other
// lengths from 16 to 8192 go through Bluestein transforms of length M <= 16384.
bool direct_length(int n) { return n >= 16 && n <= 8192 && (n & 1) == 0 && factor_235(n); }
bool bluestein_length(int n) { return !direct_length(n) && n >= 16 && n <= 8192; }

// In-place radix-2 DFT of length m (a power of two), sign -1, float64 (host tables only).
void host_fft(std::vector<double> &re, std::vector<double> &im)
{
    const size_t m = re.size();
    for (size_t i = 1, j = 0; i < m; i++) {
        size_t bit = m >> 1;
        for (; j & bit; bit >>= 1) j ^= bit;
        j ^= bit;
        if (i < j) {
            std::swap(re[i], re[j]);
            std::swap(im[i], im[j]);
        }
    }
    for (size_t len = 2; len <= m; len <<= 1) {
        for (size_t k = 0; k < len / 2; k++) {
            const double a = -2.0 * M_PI * (double)k / (double)len, c = std::cos(a), sn = std::sin(a);
            for (size_t s0 = 0; s0 < m; s0 += len) {
                const size_t i0 = s0 + k, i1 = i0 + len / 2;
                const double vr = re[i1] * c - im[i1] * sn, vi = re[i1] * sn + im[i1] * c;
                re[i1] = re[i0] - vr;
                im[i1] = im[i0] - vi;
                re[i0] += vr;
                im[i0] += vi;
            }
        }
    }
}

int chirp_samples(const sar_radar &r)
{
    const double x = r.pulse_width * r.fs;
    const double k = std::nearbyint(x);
    return (int)(std::fabs(x - k) < 1e-6 ? k : std::floor(x));
}

sar_status cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return SAR_OK;
    if (e == cudaErrorMemoryAllocation) return SAR_ERR_NO_MEMORY;
    return SAR_ERR_CUDA;
}

// The matched-filter spectrum conj(DFT_N(h)), h the centred up-chirp on the
// integer samples s with -nc/2 <= s < nc/2, stored circularly; the DFT is a
// direct sum over the nc nonzero samples, in float64.
// Weights of the nc reference-chirp samples ("GPU-accelerated backprojection SAR imaging",
// section 3.1: weighting the matched filter trades the ~-13 dB range sidelobes of the unweighted
// one for a wider main lobe).  Hamming: 0.54 - 0.46 cos(2 pi i / (nc - 1)).  Taylor (nbar terms,
// sidelobes sll_db below the peak): the line-source distribution 1 + 2 sum_m F_m cos(2 pi m x) at
// x = (i - (nc - 1) / 2) / nc, with A = acosh(10^(sll/20)) / pi, sigma^2 = nbar^2 / (A^2 +
// (nbar - 1/2)^2) and F_m = (-1)^(m+1)/2 prod_n (1 - m^2 / (sigma^2 (A^2 + (n - 1/2)^2))) /
// prod_{n != m} (1 - m^2 / n^2), n = 1 .. nbar - 1.
std::vector<double> range_weights(int kind, int nc, int nbar, double sll_db)
{
    std::vector<double> w((size_t)nc, 1.0);
    if (kind == SAR_WINDOW_HAMMING) {
        for (int i = 0; i < nc; i++) w[i] = 0.54 - 0.46 * std::cos(2.0 * M_PI * i / (nc - 1));
    } else if (kind == SAR_WINDOW_TAYLOR) {
        const double A = std::acosh(std::pow(10.0, sll_db / 20.0)) / M_PI;
        const double s2 = nbar * (double)nbar / (A * A + (nbar - 0.5) * (nbar - 0.5));
        std::vector<double> F((size_t)nbar, 0.0);
        for (int m = 1; m < nbar; m++) {
            double num = 1.0, den = 1.0;
            for (int k = 1; k < nbar; k++) {
                num *= 1.0 - m * (double)m / (s2 * (A * A + (k - 0.5) * (k - 0.5)));
                if (k != m) den *= 1.0 - m * (double)m / (k * (double)k);
            }
            F[m] = (m % 2 ? 0.5 : -0.5) * num / den;
        }
        for (int i = 0; i < nc; i++) {
            const double x = (i - 0.5 * (nc - 1)) / nc;
            double v = 1.0;
            for (int m = 1; m < nbar; m++) v += 2.0 * F[m] * std::cos(2.0 * M_PI * m * x);
            w[i] = v;
        }
    }
    return w;
}

void build_matched_filter(const sar_radar &r, int n, std::vector<float2> &H, int window = SAR_WINDOW_NONE,
                          int nbar = 4, double sll_db = 35.0)
{
    const int nc = chirp_samples(r);
    const double K = r.bandwidth / r.pulse_width;
    const std::vector<double> w = range_weights(window, nc, nbar, sll_db);
    std::vector<double> hre, him;
    std::vector<int> hs;
    for (int s = -nc; s <= nc; s++) {
        if (2 * s < -nc || 2 * s >= nc) continue;
        const double tau = s / r.fs;
        const double ph = M_PI * K * tau * tau;
        const double a = w[(size_t)(s + nc / 2)];                 // sample s - s_first, s_first = -(nc / 2)
        hs.push_back(((s % n) + n) % n);
        hre.push_back(a * std::cos(ph));
        him.push_back(a * std::sin(ph));
    }
    H.resize(n);
    for (int k = 0; k < n; k++) {
        double re = 0.0, im = 0.0;
        for (size_t j = 0; j < hs.size(); j++) {
            const long long t = ((long long)hs[j] * k) % n;
            const double a = -2.0 * M_PI * (double)t / n;
            const double c = std::cos(a), s = std::sin(a);
            re += hre[j] * c - him[j] * s;
            im += hre[j] * s + him[j] * c;
        }
        H[k] = make_float2((float)(re / n), (float)(-im / n));     // conjugate, with the IDFT's 1 / Nr
    }
}

sar_status validate_radar(const sar_radar *r)
{
    if (!r) return SAR_ERR_INVALID_ARG;
    if (!finite_pos(r->fc) || !finite_pos(r->bandwidth) || !finite_pos(r->pulse_width) || !finite_pos(r->fs) ||
        !std::isfinite(r->range_start))
        return SAR_ERR_INVALID_ARG;
    if (r->n_pulses < 1 || r->n_range < 1 || r->upsample < 1) return SAR_ERR_INVALID_ARG;
    if (!direct_length(r->n_range) && !bluestein_length(r->n_range)) return SAR_ERR_UNSUPPORTED;
    if (r->upsample != 1 && r->upsample != 2 && r->upsample != 4 && r->upsample != 8) return SAR_ERR_UNSUPPORTED;
    const int nc = chirp_samples(*r);
    if (nc < 1 || nc > r->n_range) return SAR_ERR_UNSUPPORTED;
    return SAR_OK;
}

sar_status validate_grid(const sar_grid *g)
{
    if (!std::isfinite(g->x0) || !std::isfinite(g->y0) || !std::isfinite(g->z0)) return SAR_ERR_INVALID_ARG;
    if (!finite_pos(g->dx) || !finite_pos(g->dy) || g->nx < 1 || g->ny < 1) return SAR_ERR_INVALID_ARG;
    return SAR_OK;
}

sar_status setup_rc(sar_plan p)
{
    const sar_radar &r = p->radar;
    const int n = r.n_range, U = r.upsample, un = n * U;
    sar::RcArgs &a = p->rc;
    a.n = n;
    a.u = U;
    a.n_passes = plan_radices(n, a.radix);
    int bits = 0;
    while ((1 << (2 * bits)) < un) bits++;                      // lo table ~ sqrt(U N) entries
    a.ptw_lo_bits = bits;
    const int n_lo = 1 << bits, n_hi = (un + n_lo - 1) / n_lo;

    std::vector<float2> host;
    build_matched_filter(r, n, host);                           // [0, n)
    for (int t = 0; t < n; t++) {                               // [n, 2n)
        const double ang = -2.0 * M_PI * t / n;
        host.push_back(make_float2((float)std::cos(ang), (float)std::sin(ang)));
    }
    for (int t = 0; t < n_hi; t++) {                            // [2n, 2n + n_hi)
        const double ang = -2.0 * M_PI * ((double)t * n_lo) / un;
        host.push_back(make_float2((float)std::cos(ang), (float)std::sin(ang)));
    }
    for (int t = 0; t < n_lo; t++) {                            // then n_lo
        const double ang = -2.0 * M_PI * (double)t / un;
        host.push_back(make_float2((float)std::cos(ang), (float)std::sin(ang)));
    }
    for (int k = 0; k < n; k++) {                               // then n: exp(+2 pi i k_s / (U N))
        const int ks = (2 * k >= n) ? k - n : k;
        const double ang = 2.0 * M_PI * (double)ks / un;
        host.push_back(make_float2((float)std::cos(ang), (float)std::sin(ang)));
    }
    for (int t = 0; t < n; t++) {                               // then n: conj(w_N^t), the inverse twiddles
        const float2 w = host[n + t];
        host.push_back(make_float2(w.x, -w.y));
    }
    cudaError_t e = dev_alloc(&p->d_tables, host.size() * sizeof(float2));
    if (e != cudaSuccess) return cuda_status(e);
    e = cudaMemcpy(p->d_tables, host.data(), host.size() * sizeof(float2), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_status(e);
    a.h = p->d_tables;
    a.tw = p->d_tables + n;
    a.ptw_hi = p->d_tables + 2 * n;
    a.ptw_lo = p->d_tables + 2 * n + n_hi;
    a.ramp = p->d_tables + 2 * n + n_hi + n_lo;
    a.twi = p->d_tables + 3 * n + n_hi + n_lo;
    a.planar = 0;
    a.err = p->d_err;
    a.wait_limit_ns = sar::kWaitLimitNs;
    if (const char *wl = std::getenv("SAR_WAIT_LIMIT_NS")) a.wait_limit_ns = std::strtoull(wl, nullptr, 10);
    a.bm = 0;
    if (bluestein_length(n)) {
        // Bluestein tables: M-point twiddles, w_t = exp(-i pi t^2 / N) (t^2 reduced mod 2N so the
        // angle stays small), and Bf = FFT_M(b) / M with b_t = conj(w_t) at t and M - t
        int m = 512;                                            // the register transforms start at 512
        while (m < 2 * n - 1) m <<= 1;
        a.bm = m;
        a.bm_passes = plan_radices(m, a.bm_radix);
        std::vector<float2> bt;
        for (int t = 0; t < m; t++) {
            const double ang = -2.0 * M_PI * t / m;
            bt.push_back(make_float2((float)std::cos(ang), (float)std::sin(ang)));
        }
        std::vector<double> br(m, 0.0), bi(m, 0.0);
        for (int t = 0; t < n; t++) {
            const long long t2 = ((long long)t * t) % (2LL * n);
            const double ang = -M_PI * (double)t2 / n;
            bt.push_back(make_float2((float)std::cos(ang), (float)std::sin(ang)));
            br[t] = std::cos(ang);
            bi[t] = -std::sin(ang);
            if (t > 0) {
                br[m - t] = br[t];
                bi[m - t] = bi[t];
            }
        }
        host_fft(br, bi);
        for (int k = 0; k < m; k++) bt.push_back(make_float2((float)(br[k] / m), (float)(bi[k] / m)));
        e = dev_alloc(&p->d_blue, bt.size() * sizeof(float2));
        if (e == cudaSuccess) e = cudaMemcpy(p->d_blue, bt.data(), bt.size() * sizeof(float2), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_status(e);
        a.btw = p->d_blue;
        a.bw = p->d_blue + m;
        a.bf = p->d_blue + m + n;
    }
    e = sar::rc_configure(n);
    if (e != cudaSuccess) return cuda_status(e);
    a.max_ctas = sar::rc_resident_ctas(n, U, p->device);
    a.prefetch_ahead = sar::rc_prefetch_ahead(n, U, p->device);
    return a.max_ctas > 0 ? SAR_OK : SAR_ERR_CUDA;
}

// Pulse slices for a backprojection of `pulses` pulses: the tiles x slices work units should fill
// the resident CTA slots in whole waves without making the slices so short that the CTAs' fixed
// cost dominates; each slice keeps at least 16 pulses.
int bp_pick_slices(sar_plan p, int pulses)
{
    // Time of a call with S slices ~ waves(S) * (pulses / S + P0): the CTAs of tiles * S units run
    // in waves of `slots`, each CTA walks pulses / S pulses, and P0 ~ 8 pulses' worth of time is
    // a CTA's fixed cost (its first batches' parameters, gather and barriers).  Fewer slices win
    // ties within 0.5% (less partial-image traffic).  For 512 tiles on 456 slots and 4096 pulses
    // that is 8 slices (9 waves of 512-pulse CTAs) rather than 7 (8 waves of 585).
    constexpr double kCtaFixedPulses = 8.0;
    const long long tiles = (long long)p->bp.tiles_x * p->bp.tiles_y;
    const long long slots = p->bp_slots > 0 ? p->bp_slots : 1;
    int cap = pulses / 16;
    if (cap > sar::kBpMaxSlices) cap = sar::kBpMaxSlices;
    auto cost = [&](int sl) {
        return (double)((tiles * sl + slots - 1) / slots) * ((double)pulses / sl + kCtaFixedPulses);
    };
    int best = 1;
    double best_cost = cost(1);
    for (int sl = 2; sl <= cap; sl++) {
        const double c = cost(sl);
        if (c < 0.995 * best_cost) {
            best = sl;
            best_cost = c;
        }
    }
    return best;
}

float2 split_double(double v)
{
    const float hi = (float)v;
    return make_float2(hi, (float)(v - (double)hi));
}

sar_status setup_bp(sar_plan p)
{
    const sar_radar &r = p->radar;
    const sar_grid &g = p->grid;
    sar::BpArgs &a = p->bp;
    a.x0 = g.x0;
    a.y0 = g.y0;
    a.z0 = g.z0;
    a.dx = g.dx;
    a.dy = g.dy;
    a.dxf = (float)g.dx;
    a.dyf = (float)g.dy;
    a.nx = g.nx;
    a.ny = g.ny;
    // tile shape: the longest in azimuth (x) whose half-diagonal h stays within
    // clamp(R_start / 150, 20 m, 32 m) and whose staged window fits the shared memory.  The range
    // expansion about the tile centre holds for tiles at least 100 h away (the prep kernel checks
    // every tile and pulse), so down to 2/3 of the range window's start (a grid may reach nearer
    // than the swath), and never closer than 2 km for a 20 m tile.  Shorter tiles in range stage narrower windows: 128 x 16 pixels at
    // 0.5 m stage half the samples per pulse of 64 x 32 (measured on GB300, 512 x 512 pixels, 1024
    // pulses: 0.211 against 0.238 ms).
    const double dr = kC0 / (2.0 * r.fs * r.upsample);
    const double h_max = std::min(32.0, std::max(20.0, r.range_start / 150.0));
    // 216 KB of shared memory per SM, split between the resident CTAs: 48 pulses' parameters, the
    // rest for raw and staged rows; the kernel sizes its rows from the windows it actually stages
    const int pulses_per_batch = 48;
    const int stage_bytes = 216 * 1024 / sar::kBpCtasPerSm - sar::kBpParamSlots * pulses_per_batch * (int)sizeof(float4);
    // When no shape stays within h_max: the one with the smallest half-diagonal, and of equal ones
    // the longest in azimuth.  Pixels carry their range as a float32 offset from the tile centre, so
    // a tile short in range also keeps the offsets' rounding small: at X band about 1.5e-3 rad of
    // phase for the 27 m range half-extent of a 32 x 64 tile of 1 m pixels, half that for 64 x 32
    // (measured against the oracle on images of noise, where it shows undamped).
    a.tile_w = 0;
    int fallback_w = 32;
    double fallback_h = 1e300;
    for (int tw : {128, 64, 32}) {
        const int th = sar::kBpThreads * sar::kBpRowsPerThread / tw;
        const double h = 0.5 * std::hypot((tw - 1) * g.dx, (th - 1) * g.dy);
        const int w = 2 * ((int)std::ceil(h / dr) + 3) + 1;
        if (w * 16 + ((w + 3) & ~1) * 8 > stage_bytes) continue;
        if (h <= h_max) {
            a.tile_w = tw;
            break;
        }
        if (h < fallback_h) {
            fallback_h = h;
            fallback_w = tw;
        }
    }
    if (a.tile_w == 0) a.tile_w = fallback_w;
    a.tile_h = sar::kBpThreads * sar::kBpRowsPerThread / a.tile_w;
    a.tiles_x = (g.nx + a.tile_w - 1) / a.tile_w;
    a.tiles_y = (g.ny + a.tile_h - 1) / a.tile_h;
    if (a.tiles_y > 65535) return SAR_ERR_UNSUPPORTED;
    a.range_start = r.range_start;
    a.inv_dr = 1.0 / dr;
    a.dr = (float)dr;
    a.n_samples = r.n_range * r.upsample;
    a.n_range = r.n_range;
    a.u_shift = r.upsample == 8 ? 3 : r.upsample == 4 ? 2 : r.upsample == 2 ? 1 : 0;
    a.u_mask = r.upsample - 1;
    a.planar = 0;
    const double lambda = kC0 / r.fc;
    const double ph = 2.0 * r.range_start / lambda;
    a.phase0_turns = ph - std::floor(ph);
    a.kappa = 2.0 * dr / lambda;
    a.x0s = split_double(g.x0);
    a.y0s = split_double(g.y0);
    a.z0s = split_double(g.z0);
    a.dxs = split_double(g.dx);
    a.dys = split_double(g.dy);
    a.rss = split_double(r.range_start);
    a.idrs = split_double(1.0 / dr);
    a.ph0s = split_double(a.phase0_turns);
    a.kps = split_double(a.kappa);
    a.two_pi_kappa = (float)(2.0 * M_PI * a.kappa);
    // window: every pixel of a tile lies within the half-diagonal r_t of its centre, so its range lies
    // within r_t of the centre's range; wh bins on each side plus margin for the float32 offsets
    const double ex = (a.tile_w - 1) * g.dx, ey = (a.tile_h - 1) * g.dy;
    const double rt = 0.5 * std::sqrt(ex * ex + ey * ey);
    a.wh = (int)std::ceil(rt / dr) + 3;
    a.w = 2 * a.wh + 1;
    a.min_range_tiles = (float)(100.0 * rt);
    a.pulses_per_batch = pulses_per_batch;
    a.stage_bytes = stage_bytes;
    if (a.w * 16 + ((a.w + 3) & ~1) * 8 > a.stage_bytes) return SAR_ERR_UNSUPPORTED;   // pixels too coarse
    a.err = p->d_err;
    {
        const size_t entries = (size_t)a.tiles_x * a.tiles_y * r.n_pulses;
        cudaError_t et = dev_alloc(&p->d_table, entries * 3 * sizeof(float4));
        if (et != cudaSuccess) return cuda_status(et);
        a.table = p->d_table;
    }
    const int smem = (int)sar::bp_smem_bytes(a);
    cudaError_t e = sar::bp_configure(smem);
    if (e != cudaSuccess) return cuda_status(e);
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device);
    if (e != cudaSuccess) return cuda_status(e);
    p->sms = sms;
    p->bp_slots = sar::bp_ctas_per_sm(smem, a.mode) * sms;
    // partial images for the largest pulse slicing a full-aperture call can pick (at most 512 MB)
    const size_t img_bytes = (size_t)g.nx * g.ny * sizeof(float2);
    int smax = bp_pick_slices(p, r.n_pulses);
    while (smax > 1 && (size_t)smax * img_bytes > ((size_t)512 << 20)) smax--;
    p->bp_max_slices = smax;
    if (smax > 1) {
        e = dev_alloc(&p->d_partial, (size_t)smax * img_bytes);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return SAR_OK;
}

constexpr size_t kMaxTimedCalls = 4096;     // per kind (range compression, backprojection)

// The next free event pair of the plan's pool, or {null, null} when timing is off, the pool is
// full or an event cannot be created (timing is best effort; the work is launched regardless).
std::pair<cudaEvent_t, cudaEvent_t> timing_pair(sar_plan p, std::vector<std::pair<cudaEvent_t, cudaEvent_t>> &list)
{
    if (!p->timing || list.size() >= kMaxTimedCalls) return {nullptr, nullptr};
    while (p->ev_pool.size() < p->ev_used + 2) {
        cudaEvent_t e = nullptr;
        if (cudaEventCreate(&e) != cudaSuccess) return {nullptr, nullptr};
        p->ev_pool.push_back(e);
    }
    std::pair<cudaEvent_t, cudaEvent_t> pr{p->ev_pool[p->ev_used], p->ev_pool[p->ev_used + 1]};
    p->ev_used += 2;
    list.push_back(pr);
    return pr;
}

// Launch range compression with the plan's timing events around it (when timing is on).
sar_status timed_rc(sar_plan plan, const sar::RcArgs &a, const float2 *raw, float2 *rc, int64_t n_lines,
                    cudaStream_t s)
{
    const auto ev = timing_pair(plan, plan->ev_rc);
    if (ev.first && cudaEventRecord(ev.first, s) != cudaSuccess) return SAR_ERR_CUDA;
    sar_status st = cuda_status(sar::launch_rc(a, raw, rc, n_lines, s));
    if (st == SAR_OK && ev.second && cudaEventRecord(ev.second, s) != cudaSuccess) return SAR_ERR_CUDA;
    return st;
}

void free_plan(sar_plan p)
{
    if (!p) return;
    for (cudaEvent_t e : p->ev_pool) cudaEventDestroy(e);
    for (cudaEvent_t e : p->host_ev)
        if (e) cudaEventDestroy(e);
    for (cudaEvent_t e : p->img_ev)
        if (e) cudaEventDestroy(e);
    if (p->copy_stream) cudaStreamDestroy(p->copy_stream);
    if (p->aux_stream) cudaStreamDestroy(p->aux_stream);
    cudaFree(p->d_partial2);
    cudaFree(p->d_tables);
    cudaFree(p->d_partial);
    cudaFree(p->d_table);
    cudaFree(p->d_rd_tables);
    cudaFree(p->d_blue);
    cudaFree(p->d_err);
    if (p->h_err) cudaFreeHost(p->h_err);
    cudaFree(p->d_raw);
    cudaFree(p->d_pos);
    cudaFree(p->d_rc);
    cudaFree(p->d_img);
    delete p;
}

// With `concurrent`, the call keeps to its own pulses' rows of the parameter table, uses the
// given partial images and orders its writes of the image after image_wait (recording
// image_done), so that calls over disjoint pulse ranges may run on different streams at once.
sar_status do_backproject(sar_plan plan, const void *rc, const double *pos, int32_t pulse_begin,
                          int32_t pulse_count, void *image, int accumulate, cudaStream_t s, int layout,
                          bool concurrent = false, float2 *partial = nullptr, cudaEvent_t image_wait = nullptr,
                          cudaEvent_t image_done = nullptr)
{
    const size_t img_bytes = (size_t)plan->grid.nx * plan->grid.ny * sizeof(float2);
    if (pulse_count == 0) {
        if (!accumulate) return cuda_status(cudaMemsetAsync(image, 0, img_bytes, s));
        return SAR_OK;
    }
    sar::BpArgs a = plan->bp;
    a.rc = static_cast<const float2 *>(rc);
    a.pos = pos;
    a.image = static_cast<float2 *>(image);
    a.pulse_begin = pulse_begin;
    a.pulse_end = pulse_begin + pulse_count;
    a.accumulate = accumulate ? 1 : 0;
    int slices = bp_pick_slices(plan, pulse_count);
    if (slices > plan->bp_max_slices) slices = plan->bp_max_slices;
    a.slice_len = (pulse_count + slices - 1) / slices;
    a.partial = plan->d_partial;
    a.planar = (layout == SAR_RC_POLYPHASE && plan->radar.upsample > 1) ? 1 : 0;
    if (concurrent) {
        a.table += (size_t)3 * a.tiles_x * a.tiles_y * pulse_begin;
        if (partial) a.partial = partial;
    }
    plan->last_launches += slices > 1 ? 3 : 2;
    const auto ev = timing_pair(plan, plan->ev_bp);
    return cuda_status(sar::launch_bp(a, slices, plan->check_bounds, s, ev.first, ev.second, image_wait, image_done));
}

}  // namespace

extern "C" {

const char *sar_status_string(sar_status s)
{
    switch (s) {
    case SAR_OK: return "success";
    case SAR_ERR_INVALID_ARG: return "invalid argument";
    case SAR_ERR_UNSUPPORTED: return "unsupported parameters";
    case SAR_ERR_NO_MEMORY: return "out of memory";
    case SAR_ERR_CUDA: return "CUDA error";
    case SAR_ERR_TIMEOUT: return "device-side wait timed out";
    case SAR_ERR_INTERNAL: return "internal error (device bounds check)";
    }
    return "unknown status";
}

sar_status sar_plan_create(const sar_radar *radar, const sar_grid *grid, int device, sar_plan *out)
{
    if (!out) return SAR_ERR_INVALID_ARG;
    *out = nullptr;
    sar_status st = validate_radar(radar);
    if (st != SAR_OK) return st;
    if (grid && (st = validate_grid(grid)) != SAR_OK) return st;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) return SAR_ERR_CUDA;
    if (device < 0 || device >= ndev) return SAR_ERR_INVALID_ARG;
    DeviceGuard guard(device);
    if (guard.status != cudaSuccess) return SAR_ERR_CUDA;

    sar_plan p = new (std::nothrow) sar_plan_s;
    if (!p) return SAR_ERR_NO_MEMORY;
    p->device = device;
    p->radar = *radar;
    if (grid) {
        p->grid = *grid;
        p->has_grid = true;
    }
    const char *cb = std::getenv("SAR_CHECK_BOUNDS");
    p->check_bounds = cb && cb[0] == '1';
    cudaError_t e = dev_alloc(&p->d_err, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(p->d_err, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaMallocHost(&p->h_err, sizeof(int));
    if (e != cudaSuccess) {
        free_plan(p);
        return cuda_status(e);
    }
    st = setup_rc(p);
    if (st == SAR_OK && p->has_grid) st = setup_bp(p);
    if (st != SAR_OK) {
        free_plan(p);
        return st;
    }
    sar_log("plan %p: device %d, Na %d, Nr %d (%s), U %d, fc %.6g Hz, B %.6g Hz, Tp %.6g s, fs %.6g Hz, "
            "range_start %.6f m", (void *)p, device, radar->n_pulses, radar->n_range,
            p->rc.bm ? "Bluestein" : "mixed radix", radar->upsample, radar->fc, radar->bandwidth, radar->pulse_width,
            radar->fs, radar->range_start);
    if (p->has_grid)
        sar_log("plan %p: grid %d x %d at (%.3f, %.3f) m, tiles %d x %d of %d x %d pixels, window %d entries, "
                "%d resident backprojection CTAs, up to %d pulse slices", (void *)p, p->grid.nx, p->grid.ny,
                p->grid.dx, p->grid.dy, p->bp.tiles_x, p->bp.tiles_y, p->bp.tile_w, p->bp.tile_h, p->bp.w,
                p->bp_slots, p->bp_max_slices);
    *out = p;
    return SAR_OK;
}

sar_status sar_plan_destroy(sar_plan plan)
{
    if (!plan) return SAR_OK;
    DeviceGuard guard(plan->device);
    cudaDeviceSynchronize();
    free_plan(plan);
    return SAR_OK;
}

sar_status sar_workspace_size(sar_plan plan, size_t *bytes)
{
    if (!plan || !bytes) return SAR_ERR_INVALID_ARG;
    const size_t raw = (size_t)plan->radar.n_pulses * plan->radar.n_range * plan->radar.upsample * sizeof(float2);
    *bytes = (raw + 255) & ~(size_t)255;
    return SAR_OK;
}

sar_status sar_range_compress(sar_plan plan, const void *raw, void *rc, int64_t n_lines, void *stream)
{
    if (!plan || !raw || !rc || n_lines < 1) return SAR_ERR_INVALID_ARG;
    if (!aligned16(raw) || !aligned16(rc)) return SAR_ERR_INVALID_ARG;
    const int64_t in_bytes = n_lines * plan->radar.n_range * (int64_t)sizeof(float2);
    const int64_t out_bytes = in_bytes * plan->radar.upsample;
    const char *r0 = static_cast<const char *>(raw), *c0 = static_cast<const char *>(rc);
    if (r0 < c0 + out_bytes && c0 < r0 + in_bytes) return SAR_ERR_INVALID_ARG;     // overlap
    DeviceGuard guard(plan->device);
    if (guard.status != cudaSuccess) return SAR_ERR_CUDA;
    plan->last_launches = 1;
    sar::RcArgs a = plan->rc;
    a.planar = plan->rc_layout == SAR_RC_POLYPHASE ? 1 : 0;
    return timed_rc(plan, a, static_cast<const float2 *>(raw), static_cast<float2 *>(rc), n_lines,
                    static_cast<cudaStream_t>(stream));
}

sar_status sar_backproject(sar_plan plan, const void *rc, const double *pos, int32_t pulse_begin,
                           int32_t pulse_count, void *image, int accumulate, void *stream)
{
    if (!plan || !rc || !pos || !image) return SAR_ERR_INVALID_ARG;
    if (!plan->has_grid) return SAR_ERR_UNSUPPORTED;
    if (pulse_begin < 0 || pulse_count < 0 || (int64_t)pulse_begin + pulse_count > plan->radar.n_pulses)
        return SAR_ERR_INVALID_ARG;
    if (!aligned16(rc) || !aligned16(image) || (reinterpret_cast<uintptr_t>(pos) & 7u)) return SAR_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (guard.status != cudaSuccess) return SAR_ERR_CUDA;
    plan->last_launches = 0;
    return do_backproject(plan, rc, pos, pulse_begin, pulse_count, image, accumulate,
                          static_cast<cudaStream_t>(stream), plan->rc_layout);
}

sar_status sar_form_image(sar_plan plan, const void *raw, const double *pos, void *image, void *workspace,
                          size_t workspace_bytes, void *stream)
{
    if (!plan || !raw || !pos || !image || !workspace) return SAR_ERR_INVALID_ARG;
    if (!plan->has_grid) return SAR_ERR_UNSUPPORTED;
    size_t need = 0;
    sar_workspace_size(plan, &need);
    if (workspace_bytes < need) return SAR_ERR_INVALID_ARG;
    if (!aligned16(raw) || !aligned16(workspace) || !aligned16(image) || (reinterpret_cast<uintptr_t>(pos) & 7u))
        return SAR_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (guard.status != cudaSuccess) return SAR_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    plan->last_launches = 1;
    sar::RcArgs ra = plan->rc;
    ra.planar = 1;
    sar_status st = timed_rc(plan, ra, static_cast<const float2 *>(raw), static_cast<float2 *>(workspace),
                             plan->radar.n_pulses, s);
    if (st != SAR_OK) return st;
    return do_backproject(plan, workspace, pos, 0, plan->radar.n_pulses, image, 0, s, SAR_RC_POLYPHASE);
}

sar_status sar_plan_set_range_doppler(sar_plan plan, double pulse_spacing)
{
    if (!plan) return SAR_ERR_INVALID_ARG;
    const sar_radar &r = plan->radar;
    const double lambda = kC0 / r.fc;
    if (!std::isfinite(pulse_spacing) || !(pulse_spacing > 0.0)) return SAR_ERR_INVALID_ARG;
    if (r.upsample != 1 || !sar::rd_supported_pulses(r.n_pulses)) return SAR_ERR_UNSUPPORTED;
    if (lambda / (4.0 * pulse_spacing) >= 1.0) return SAR_ERR_UNSUPPORTED;
    DeviceGuard guard(plan->device);
    if (guard.status != cudaSuccess) return SAR_ERR_CUDA;
    const int na = r.n_pulses;
    // host tables in float64: azimuth twiddles, (2/lambda)(1 - D_m) split into (hi, lo), 1/D_m - 1
    std::vector<float2> tw(na), phc(na);
    std::vector<float> rcm(na);
    for (int t = 0; t < na; t++) {
        const double ang = -2.0 * M_PI * t / na;
        tw[t] = make_float2((float)std::cos(ang), (float)std::sin(ang));
        const int ms = (2 * t < na) ? t : t - na;
        const double kx = (double)ms / ((double)na * pulse_spacing);
        const double u = lambda * kx / 2.0;
        const double D = std::sqrt(1.0 - u * u);
        const double one_minus_d = u * u / (1.0 + D);             // 1 - D without cancellation
        phc[t] = split_double(2.0 / lambda * one_minus_d);
        rcm[t] = (float)(one_minus_d / D);                         // 1/D - 1
    }
    const size_t bytes = 2 * (size_t)na * sizeof(float2) + (size_t)na * sizeof(float);
    cudaError_t e = cudaDeviceSynchronize();                        // queued work may read the old tables
    if (e != cudaSuccess) return cuda_status(e);
    cudaFree(plan->d_rd_tables);
    plan->d_rd_tables = nullptr;
    plan->rd_ready = false;
    e = dev_alloc(&plan->d_rd_tables, bytes);
    char *base = static_cast<char *>(plan->d_rd_tables);
    if (e == cudaSuccess) e = cudaMemcpy(base, tw.data(), na * sizeof(float2), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(base + na * sizeof(float2), phc.data(), na * sizeof(float2), cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
        e = cudaMemcpy(base + 2 * na * sizeof(float2), rcm.data(), na * sizeof(float), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = sar::rd_configure();
    if (e != cudaSuccess) return cuda_status(e);
    sar::RdaArgs &a = plan->rd;
    a.na = na;
    a.nr = r.n_range;
    a.tw = reinterpret_cast<const float2 *>(base);
    a.phc = reinterpret_cast<const float2 *>(base + na * sizeof(float2));
    a.rcm = reinterpret_cast<const float *>(base + 2 * na * sizeof(float2));
    a.range_start = r.range_start;
    a.dr = kC0 / (2.0 * r.fs);
    a.two_over_lambda = 2.0 / lambda;
    a.inv_na = 1.0f / (float)na;
    plan->rd_ready = true;
    return SAR_OK;
}

sar_status sar_range_doppler_workspace_size(sar_plan plan, size_t *bytes)
{
    if (!plan || !bytes) return SAR_ERR_INVALID_ARG;
    if (!plan->rd_ready) return SAR_ERR_UNSUPPORTED;
    *bytes = 2 * (size_t)plan->radar.n_pulses * plan->radar.n_range * sizeof(float2);
    return SAR_OK;
}

sar_status sar_range_doppler(sar_plan plan, const void *raw, void *image, void *workspace, size_t workspace_bytes,
                             void *stream)
{
    if (!plan || !raw || !image || !workspace) return SAR_ERR_INVALID_ARG;
    if (!plan->rd_ready) return SAR_ERR_UNSUPPORTED;
    const size_t plane = (size_t)plan->radar.n_pulses * plan->radar.n_range;
    if (workspace_bytes < 2 * plane * sizeof(float2)) return SAR_ERR_INVALID_ARG;
    if (!aligned16(raw) || !aligned16(image) || !aligned16(workspace)) return SAR_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (guard.status != cudaSuccess) return SAR_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float2 *rc = static_cast<float2 *>(workspace), *work = rc + plane;
    plan->last_launches = 4;
    sar_status st = timed_rc(plan, plan->rc, static_cast<const float2 *>(raw), rc, plan->radar.n_pulses, s);
    if (st != SAR_OK) return st;
    return cuda_status(sar::launch_rd(plan->rd, rc, work, static_cast<float2 *>(image), s));
}

sar_status sar_form_image_host(sar_plan plan, const void *raw_host, const double *pos_host, void *image_host,
                               void *stream)
{
    if (!plan || !raw_host || !pos_host || !image_host) return SAR_ERR_INVALID_ARG;
    if (!plan->has_grid) return SAR_ERR_UNSUPPORTED;
    DeviceGuard guard(plan->device);
    if (guard.status != cudaSuccess) return SAR_ERR_CUDA;
    const sar_radar &r = plan->radar;
    const size_t raw_bytes = (size_t)r.n_pulses * r.n_range * sizeof(float2);
    const size_t pos_bytes = (size_t)r.n_pulses * 3 * sizeof(double);
    const size_t img_bytes = (size_t)plan->grid.nx * plan->grid.ny * sizeof(float2);
    size_t ws = 0;
    sar_workspace_size(plan, &ws);
    cudaError_t e = cudaSuccess;
    if (!plan->d_raw && e == cudaSuccess) e = dev_alloc(&plan->d_raw, raw_bytes);
    if (!plan->d_pos && e == cudaSuccess) e = dev_alloc(&plan->d_pos, pos_bytes);
    if (!plan->d_rc && e == cudaSuccess) e = dev_alloc(&plan->d_rc, ws);
    if (!plan->d_img && e == cudaSuccess) e = dev_alloc(&plan->d_img, img_bytes);
    if (e != cudaSuccess) return cuda_status(e);
    if (!plan->copy_stream && e == cudaSuccess) e = cudaStreamCreateWithFlags(&plan->copy_stream, cudaStreamNonBlocking);
    for (cudaEvent_t &ev : plan->host_ev)
        if (!ev && e == cudaSuccess) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_status(e);
    // Pulse chunks: the copy of chunk c + 1 runs on the plan's copy stream while chunk c is range
    // compressed and backprojected (accumulating into the image) on the caller's stream.  The
    // copy moves pulses about 4.5 times faster than the kernels consume them, so the chunks grow
    // (1/16, 3/16 and 3/4 of the pulses): only the small first one is not overlapped, and each
    // chunk's backprojection outlasts the next chunk's copy.  Every chunk adds a launch sequence
    // and a pulse-slice tail (measured on GB300, spotlight scene: 3.52 ms with these three chunks,
    // 3.54 ms with four (1/16, 3/16, 1/4, 1/2), 3.57 ms with five, against 3.46 ms for four chunks
    // without their copies and 3.33 ms for one).
    cudaStream_t s = static_cast<cudaStream_t>(stream), cs = plan->copy_stream;
    const int na = r.n_pulses;
    int bounds[5] = {0, na, na, na, na};
    int chunks = 1;
    if (na >= 512) {
        chunks = 3;
        bounds[1] = na / 16;
        bounds[2] = na / 4;
    }
    const size_t line_bytes = (size_t)r.n_range * sizeof(float2);
    e = cudaEventRecord(plan->host_ev[0], s);                   // earlier work on the caller's stream first
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, plan->host_ev[0], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(plan->d_pos, pos_host, pos_bytes, cudaMemcpyHostToDevice, cs);
    for (int c = 0; c < chunks && e == cudaSuccess; c++) {
        const int c0 = bounds[c], cnt = bounds[c + 1] - c0;
        e = cudaMemcpyAsync(static_cast<char *>(plan->d_raw) + c0 * line_bytes,
                            static_cast<const char *>(raw_host) + c0 * line_bytes, cnt * line_bytes,
                            cudaMemcpyHostToDevice, cs);
        if (e == cudaSuccess) e = cudaEventRecord(plan->host_ev[1 + c], cs);
    }
    if (e != cudaSuccess) return cuda_status(e);
    sar::RcArgs ra = plan->rc;
    ra.planar = 1;
    // Chunks alternate between the caller's stream and the plan's second compute stream, so that
    // one chunk's kernels fill the SMs the previous chunk's last wave leaves idle; only their
    // writes of the image are ordered (chunk c's after chunk c - 1's).  Each stream has its own
    // partial images and each chunk its own rows of the parameter table.  With kernel timing on
    // (its events sit on one stream) the chunks run in turn on the caller's stream.
    const bool overlap = chunks > 1 && !plan->timing && plan->bp_max_slices > 1;
    if (overlap) {
        if (!plan->aux_stream) e = cudaStreamCreateWithFlags(&plan->aux_stream, cudaStreamNonBlocking);
        for (cudaEvent_t &ev : plan->img_ev)
            if (!ev && e == cudaSuccess) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        if (!plan->d_partial2 && e == cudaSuccess)
            e = dev_alloc(&plan->d_partial2, (size_t)plan->bp_max_slices * img_bytes);
        // the aux stream starts after the caller's earlier work, like the copies
        if (e == cudaSuccess) e = cudaStreamWaitEvent(plan->aux_stream, plan->host_ev[0], 0);
        if (e != cudaSuccess) return cuda_status(e);
    }
    int32_t launches = 0;
    for (int c = 0; c < chunks; c++) {
        const int c0 = bounds[c], cnt = bounds[c + 1] - c0;
        const bool aux = overlap && (c & 1);
        cudaStream_t cst = aux ? plan->aux_stream : s;
        e = cudaStreamWaitEvent(cst, plan->host_ev[1 + c], 0);
        if (e != cudaSuccess) return cuda_status(e);
        float2 *rc = static_cast<float2 *>(plan->d_rc) + (size_t)c0 * r.n_range * r.upsample;
        sar_status st = timed_rc(plan, ra, static_cast<const float2 *>(plan->d_raw) + (size_t)c0 * r.n_range, rc, cnt, cst);
        if (st != SAR_OK) return st;
        plan->last_launches = 0;
        if (overlap)
            st = do_backproject(plan, plan->d_rc, static_cast<const double *>(plan->d_pos), c0, cnt, plan->d_img, c > 0,
                                cst, SAR_RC_POLYPHASE, true, aux ? plan->d_partial2 : plan->d_partial,
                                c > 0 ? plan->img_ev[c - 1] : nullptr, plan->img_ev[c]);
        else
            st = do_backproject(plan, plan->d_rc, static_cast<const double *>(plan->d_pos), c0, cnt, plan->d_img, c > 0,
                                s, SAR_RC_POLYPHASE);
        if (st != SAR_OK) return st;
        launches += 1 + plan->last_launches;
    }
    // the read-back follows the last chunk's image write
    if (overlap && ((chunks - 1) & 1)) {
        e = cudaStreamWaitEvent(s, plan->img_ev[chunks - 1], 0);
        if (e != cudaSuccess) return cuda_status(e);
    }
    plan->last_launches = launches;
    e = cudaMemcpyAsync(image_host, plan->d_img, img_bytes, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return cuda_status(e);
}

sar_status sar_plan_sync(sar_plan plan, void *stream)
{
    if (!plan) return SAR_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (guard.status != cudaSuccess) return SAR_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return SAR_ERR_CUDA;
    e = cudaMemcpy(plan->h_err, plan->d_err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return SAR_ERR_CUDA;
    const int flags = *plan->h_err;
    if (flags) {
        e = cudaMemset(plan->d_err, 0, sizeof(int));
        if (e != cudaSuccess) return SAR_ERR_CUDA;
    }
    if (flags) sar_log("plan %p: device flags 0x%x", (void *)plan, flags);
    if (flags & sar::kDevErrBounds) return SAR_ERR_INTERNAL;
    if (flags & sar::kDevErrTimeout) return SAR_ERR_TIMEOUT;
    if (flags & sar::kDevErrGeometry) return SAR_ERR_UNSUPPORTED;
    return SAR_OK;
}

int32_t sar_plan_last_launches(sar_plan plan) { return plan ? plan->last_launches : 0; }

sar_status sar_plan_set_pulse_weights(sar_plan plan, const float *weights)
{
    if (!plan) return SAR_ERR_INVALID_ARG;
    if (!plan->has_grid) return SAR_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(weights) & 3u) return SAR_ERR_INVALID_ARG;
    plan->bp.weights = weights;
    return SAR_OK;
}

namespace {

// Select variant `mode` for the plan's backprojections, or (to_default) drop it if it is the one
// selected; refuse to select a second non-default variant.
sar_status set_bp_mode(sar_plan plan, int mode, bool to_default)
{
    if (!plan) return SAR_ERR_INVALID_ARG;
    if (!plan->has_grid) return SAR_ERR_UNSUPPORTED;
    int next;
    if (to_default) next = plan->bp.mode == mode ? sar::kBpLinear : plan->bp.mode;
    else if (plan->bp.mode == sar::kBpLinear || plan->bp.mode == mode) next = mode;
    else return SAR_ERR_UNSUPPORTED;
    if (next == plan->bp.mode) return SAR_OK;
    DeviceGuard guard(plan->device);
    if (guard.status != cudaSuccess) return SAR_ERR_CUDA;
    plan->bp.mode = next;
    plan->bp_slots = sar::bp_ctas_per_sm((int)sar::bp_smem_bytes(plan->bp), next) * plan->sms;
    return SAR_OK;
}

}  // namespace

sar_status sar_plan_set_accumulation(sar_plan plan, sar_accumulation accumulation)
{
    if (accumulation != SAR_ACCUM_FP32 && accumulation != SAR_ACCUM_COMPENSATED) return SAR_ERR_INVALID_ARG;
    return set_bp_mode(plan, sar::kBpCompensated, accumulation == SAR_ACCUM_FP32);
}

sar_status sar_plan_set_stage_precision(sar_plan plan, sar_stage_precision precision)
{
    if (precision != SAR_STAGE_FP32 && precision != SAR_STAGE_FP16) return SAR_ERR_INVALID_ARG;
    return set_bp_mode(plan, sar::kBpHalfStage, precision == SAR_STAGE_FP32);
}

sar_status sar_plan_set_interpolation(sar_plan plan, sar_interpolation interpolation)
{
    if (interpolation != SAR_INTERP_LINEAR && interpolation != SAR_INTERP_SINC8) return SAR_ERR_INVALID_ARG;
    return set_bp_mode(plan, sar::kBpSinc8, interpolation == SAR_INTERP_LINEAR);
}

sar_status sar_plan_set_range_window(sar_plan plan, sar_window window, int32_t taylor_nbar, double taylor_sll_db)
{
    if (!plan) return SAR_ERR_INVALID_ARG;
    if (window != SAR_WINDOW_NONE && window != SAR_WINDOW_HAMMING && window != SAR_WINDOW_TAYLOR)
        return SAR_ERR_INVALID_ARG;
    if (window == SAR_WINDOW_TAYLOR &&
        (taylor_nbar < 2 || taylor_nbar > 64 || !(taylor_sll_db > 0.0) || !(taylor_sll_db <= 120.0)))
        return SAR_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (guard.status != cudaSuccess) return SAR_ERR_CUDA;
    std::vector<float2> H;
    build_matched_filter(plan->radar, plan->radar.n_range, H, window, taylor_nbar, taylor_sll_db);
    // work already queued on any stream may still read the old filter
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(plan->d_tables, H.data(), H.size() * sizeof(float2), cudaMemcpyHostToDevice);
    return cuda_status(e);
}

sar_status sar_plan_set_timing(sar_plan plan, int enable)
{
    if (!plan) return SAR_ERR_INVALID_ARG;
    plan->timing = enable != 0;
    return SAR_OK;
}

sar_status sar_plan_kernel_times(sar_plan plan, double *rc_ms, int32_t *rc_calls, double *bp_ms, int32_t *bp_calls)
{
    if (!plan || !rc_ms || !rc_calls || !bp_ms || !bp_calls) return SAR_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (guard.status != cudaSuccess) return SAR_ERR_CUDA;
    sar_status st = SAR_OK;
    auto sum = [&](std::vector<std::pair<cudaEvent_t, cudaEvent_t>> &list, double *ms, int32_t *n) {
        double total = 0.0;
        for (const auto &pr : list) {
            float t = 0.0f;
            cudaError_t e = cudaEventSynchronize(pr.second);
            if (e == cudaSuccess) e = cudaEventElapsedTime(&t, pr.first, pr.second);
            if (e != cudaSuccess) st = SAR_ERR_CUDA;
            total += t;
        }
        *ms = total;
        *n = (int32_t)list.size();
        list.clear();
    };
    sum(plan->ev_rc, rc_ms, rc_calls);
    sum(plan->ev_bp, bp_ms, bp_calls);
    plan->ev_used = 0;
    return st;
}

sar_status sar_plan_set_rc_layout(sar_plan plan, sar_rc_layout layout)
{
    if (!plan || (layout != SAR_RC_NATURAL && layout != SAR_RC_POLYPHASE)) return SAR_ERR_INVALID_ARG;
    plan->rc_layout = layout;
    return SAR_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// sar_form_image_noalloc: image formation whose compressed-line scratch is a
// fixed array compiled into this library instead of caller- or plan-allocated
// memory, for callers that cannot call cudaMalloc when they form an image
// (memory fixed at start-up, or owned by an allocator the library cannot use).
// The array costs every device that loads the library kNoallocScratchBytes
// until the process exits.
// ---------------------------------------------------------------------------
#include <mutex>

namespace {

constexpr size_t kNoallocScratchBytes = (size_t)32 << 20;     // 32 MiB
constexpr int kNoallocMaxDevices = 64;

// In host code this name is only a stand-in for the symbol: its device address
// comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) float2 g_noalloc_scratch[kNoallocScratchBytes / sizeof(float2)];

std::mutex g_noalloc_mutex;
float2 *g_noalloc_ptr[kNoallocMaxDevices] = {};

// Device address of the scratch array on `device`, which must be current.
sar_status noalloc_scratch(int device, float2 **out)
{
    if (device < 0 || device >= kNoallocMaxDevices) return SAR_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[device]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return SAR_ERR_CUDA;
        g_noalloc_ptr[device] = static_cast<float2 *>(p);
    }
    *out = g_noalloc_ptr[device];
    return SAR_OK;
}

}  // namespace

extern "C" sar_status sar_form_image_noalloc(sar_plan plan, const void *raw, const double *pos, void *image,
                                             void *stream)
{
    if (!plan || !raw || !pos || !image) return SAR_ERR_INVALID_ARG;
    if (!plan->has_grid) return SAR_ERR_UNSUPPORTED;
    size_t need = 0;
    sar_workspace_size(plan, &need);
    if (need > kNoallocScratchBytes) return SAR_ERR_UNSUPPORTED;
    if (!aligned16(raw) || !aligned16(image) || (reinterpret_cast<uintptr_t>(pos) & 7u)) return SAR_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (guard.status != cudaSuccess) return SAR_ERR_CUDA;
    float2 *scratch = nullptr;
    sar_status st = noalloc_scratch(plan->device, &scratch);
    if (st != SAR_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // every scratch element the backprojection reads is written by the range compression first,
    // so nothing left by an earlier call needs clearing
    plan->last_launches = 1;
    sar::RcArgs ra = plan->rc;
    ra.planar = 1;
    st = timed_rc(plan, ra, static_cast<const float2 *>(raw), scratch, plan->radar.n_pulses, s);
    if (st != SAR_OK) return st;
    return do_backproject(plan, scratch, pos, 0, plan->radar.n_pulses, image, 0, s, SAR_RC_POLYPHASE);
}
