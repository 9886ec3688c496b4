"""Seeded synthetic SAR scenes: raw pulse echoes, antenna track and pixel grid.

This module is the one input generator that both sides of every comparison
use: the fp64 CPU oracle (``oracle/``) and the CUDA library
(``domain_backprojection_gb300``).  It simulates the *forward* model only -- a
linear-FM pulse reflected by point scatterers, demodulated to baseband and
sampled -- and holds none of the arithmetic of range compression or
backprojection.  It imports neither side.

Geometry (one reading of the pages, which only fix a pixel plane z = 0 in the
backprojection kernel of "GPU-accelerated backprojection SAR imaging", section
3.3): x is along-track (azimuth), y is ground range, z is up.  The scene centre
is (0, 5000, 0) m.  The nominal track is a(t) = (v t, 0, H) with
t_n = (n - (Na - 1) / 2) / PRF.  Pixel (ix, iy) sits at
(x0 + ix dx, y0 + iy dy, z0) with the centre pixel (nx/2, ny/2) on the scene
centre.  Images are stored [ny][nx], x fastest.

Echo of a scatterer of complex amplitude a at range R from the antenna, sampled
at t_k = t0 + k / fs with t0 = 2 R_start / c0:

    e[k] = a * exp(j pi K (t_k - 2R/c0)^2) * exp(-j 4 pi fc R / c0)

for -Tp/2 <= t_k - 2R/c0 < Tp/2 (a centred up-chirp of rate K = B / Tp),
zero elsewhere.  Complex Gaussian noise of variance 10^(-SNR/10) per sample
(SNR relative to a unit scatterer) is added.  Antenna positions are
stop-and-go: one position per pulse.

Workloads (sizes from the five benchmark scenes; the pages' airborne data set
is not available, so these seeded scenes stand in for it):

  1  tiny stripmap      Na=256,   Nr=1024, U=8, 128x128 @ 0.5 m, 3 unit targets
  2  small stripmap     Na=1024,  Nr=2048, U=8, 512x512 @ 0.5 m, 16 targets
  3  spotlight          Na=4096,  Nr=4096, U=8, 1024x1024 @ 0.25 m, 64 targets
                        + one clutter scatterer per 8x8-pixel cell
  4  curved track       Na=16384, Nr=8192, U=8, 2048x2048 @ 0.2 m, 256 targets
                        + clutter, sinusoidal motion errors on all three axes
  5  range-only sweep   Na=4096 lines, Nr in {4096, 8192, 6000}, U=1
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

C0 = 299_792_458.0


@dataclasses.dataclass(frozen=True)
class Radar:
    fc: float = 10.0e9
    bandwidth: float = 150.0e6
    pulse_width: float = 2.0e-6
    fs: float = 180.0e6
    range_start: float = 0.0
    n_pulses: int = 0
    n_range: int = 0
    upsample: int = 1


@dataclasses.dataclass(frozen=True)
class Grid:
    x0: float
    y0: float
    z0: float
    dx: float
    dy: float
    nx: int
    ny: int


@dataclasses.dataclass(frozen=True)
class SceneConfig:
    name: str
    n_pulses: int
    n_range: int
    upsample: int
    prf: float
    nx: int
    ny: int
    pixel: float
    n_targets: int
    target_amp_uniform: bool
    targets_on_pixels: bool
    snr_db: float
    clutter_cell: int = 0          # one clutter scatterer per (cell x cell) pixels; 0 = none
    clutter_power: float = 0.1     # E|a|^2 of clutter scatterers (-10 dB)
    motion_amp: float = 0.0        # metres, per axis
    seed: int = 0
    velocity: float = 100.0
    altitude: float = 3000.0
    ground_range: float = 5000.0
    fixed_target_offsets: tuple = ()   # pixel offsets from the centre pixel

    @property
    def scene_centre(self):
        return (0.0, self.ground_range, 0.0)

    def centre_range(self) -> float:
        return math.hypot(self.ground_range, self.altitude)

    def radar(self) -> Radar:
        r = Radar()
        native_bin = C0 / (2.0 * r.fs)
        rs = self.centre_range() - (self.n_range / 2) * native_bin
        return dataclasses.replace(r, range_start=rs, n_pulses=self.n_pulses,
                                   n_range=self.n_range, upsample=self.upsample)

    def grid(self) -> Grid:
        return Grid(x0=-(self.nx // 2) * self.pixel,
                    y0=self.ground_range - (self.ny // 2) * self.pixel,
                    z0=0.0, dx=self.pixel, dy=self.pixel, nx=self.nx, ny=self.ny)

    @property
    def pixel_pulses(self) -> int:
        return self.n_pulses * self.nx * self.ny


def _spotlight_prf(na, v, rc, aperture_deg):
    length = 2.0 * rc * math.tan(math.radians(aperture_deg / 2.0))
    return na * v / length


SCENES = {
    1: SceneConfig("tiny-stripmap", 256, 1024, 8, 300.0, 128, 128, 0.5, 3, False, True, 20.0,
                   seed=1001, fixed_target_offsets=((0, 0), (-20, 16), (24, -28))),
    2: SceneConfig("small-stripmap", 1024, 2048, 8, 1200.0, 512, 512, 0.5, 16, True, False, 10.0,
                   seed=1002),
    3: SceneConfig("spotlight-3deg", 4096, 4096, 8,
                   _spotlight_prf(4096, 100.0, math.hypot(5000.0, 3000.0), 3.0),
                   1024, 1024, 0.25, 64, False, True, 20.0, clutter_cell=8, seed=1003),
    4: SceneConfig("curved-track", 16384, 8192, 8, 5000.0, 2048, 2048, 0.2, 256, False, True, 20.0,
                   clutter_cell=8, motion_amp=0.5, seed=1004),
}

RC_SWEEP_NR = (4096, 8192, 6000)


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + stream)
    return g


def track(cfg: SceneConfig, device="cpu") -> torch.Tensor:
    """Antenna phase-centre positions [Na][3] float64, one per pulse."""
    na = cfg.n_pulses
    n = torch.arange(na, dtype=torch.float64, device=device)
    t = (n - (na - 1) / 2.0) / cfg.prf
    pos = torch.zeros(na, 3, dtype=torch.float64, device=device)
    pos[:, 0] = cfg.velocity * t
    pos[:, 2] = cfg.altitude
    if cfg.motion_amp > 0.0:
        g = _gen(cfg.seed, 2, "cpu")
        f = torch.rand(3, generator=g, dtype=torch.float64) * 1.8 + 0.2      # 0.2..2 Hz
        ph = torch.rand(3, generator=g, dtype=torch.float64) * (2 * math.pi)
        for ax in range(3):
            pos[:, ax] += cfg.motion_amp * torch.sin(2 * math.pi * float(f[ax]) * t + float(ph[ax]))
    return pos


def targets(cfg: SceneConfig):
    """Point targets: (xyz [T][3] float64, amplitude [T] complex128, pixel index [T][2] or None)."""
    g = _gen(cfg.seed, 0, "cpu")
    grid = cfg.grid()
    cx, cy = grid.nx // 2, grid.ny // 2
    if cfg.fixed_target_offsets:
        pix = torch.tensor([[cx + ox, cy + oy] for ox, oy in cfg.fixed_target_offsets], dtype=torch.int64)
    elif cfg.targets_on_pixels:
        # distinct pixel centres in the inner 80% of the scene, at least 16 px apart
        lo_x, hi_x = int(0.1 * grid.nx), int(0.9 * grid.nx)
        lo_y, hi_y = int(0.1 * grid.ny), int(0.9 * grid.ny)
        chosen = []
        while len(chosen) < cfg.n_targets:
            ix = int(torch.randint(lo_x, hi_x, (1,), generator=g))
            iy = int(torch.randint(lo_y, hi_y, (1,), generator=g))
            if all(abs(ix - a) >= 16 or abs(iy - b) >= 16 for a, b in chosen):
                chosen.append((ix, iy))
        pix = torch.tensor(chosen, dtype=torch.int64)
    else:
        pix = None
    if pix is not None:
        xyz = torch.stack([grid.x0 + pix[:, 0].double() * grid.dx,
                           grid.y0 + pix[:, 1].double() * grid.dy,
                           torch.full((pix.shape[0],), grid.z0, dtype=torch.float64)], dim=1)
    else:
        u = torch.rand(cfg.n_targets, 2, generator=g, dtype=torch.float64) * 0.8 + 0.1
        xyz = torch.stack([grid.x0 + u[:, 0] * grid.nx * grid.dx,
                           grid.y0 + u[:, 1] * grid.ny * grid.dy,
                           torch.full((cfg.n_targets,), grid.z0, dtype=torch.float64)], dim=1)
    n = xyz.shape[0]
    if cfg.target_amp_uniform:
        amp = (torch.rand(n, generator=g, dtype=torch.float64) * 0.5 + 0.5).to(torch.complex128)
    else:
        amp = torch.ones(n, dtype=torch.complex128)
    return xyz, amp, pix


def clutter(cfg: SceneConfig):
    """Distributed clutter: one scatterer per cell, uniform within it, amplitude CN(0, clutter_power)."""
    if cfg.clutter_cell <= 0:
        return torch.zeros(0, 3, dtype=torch.float64), torch.zeros(0, dtype=torch.complex128)
    g = _gen(cfg.seed, 1, "cpu")
    grid = cfg.grid()
    cell = cfg.clutter_cell
    ncx, ncy = grid.nx // cell, grid.ny // cell
    iy, ix = torch.meshgrid(torch.arange(ncy, dtype=torch.float64),
                            torch.arange(ncx, dtype=torch.float64), indexing="ij")
    u = torch.rand(ncy, ncx, 2, generator=g, dtype=torch.float64)
    x = grid.x0 + (ix + u[..., 0]) * cell * grid.dx - 0.5 * grid.dx
    y = grid.y0 + (iy + u[..., 1]) * cell * grid.dy - 0.5 * grid.dy
    xyz = torch.stack([x.reshape(-1), y.reshape(-1), torch.full((ncx * ncy,), grid.z0, dtype=torch.float64)], 1)
    s = math.sqrt(cfg.clutter_power / 2.0)
    re = torch.randn(ncx * ncy, generator=g, dtype=torch.float64) * s
    im = torch.randn(ncx * ncy, generator=g, dtype=torch.float64) * s
    return xyz, torch.complex(re, im)


def chirp_count(radar: Radar) -> int:
    """Number of samples a pulse spans: Tp * fs, snapped to an integer when it is one."""
    x = radar.pulse_width * radar.fs
    r = round(x)
    return int(r) if abs(x - r) < 1e-6 else int(math.floor(x))


def _accumulate(acc, rows, R, amp, radar, nr):
    """Add echoes for matched (row, range, amplitude) triples; R, amp broadcast to rows' shape."""
    device = acc.device
    nc = chirp_count(radar)
    half = nc / 2.0
    d1 = C0 / (2.0 * radar.fs)                          # metres per native range bin
    carrier = 4.0 * math.pi * radar.fc / C0             # rad per metre (two-way)
    chirp_rate = math.pi * (radar.bandwidth / radar.pulse_width) / (radar.fs ** 2)  # rad per sample^2
    j = torch.arange(nc, device=device, dtype=torch.float32)
    kt = (R - radar.range_start) / d1                   # fractional sample of the echo centre (f64)
    k0 = torch.ceil(kt - half)                          # first sample inside the pulse
    frac = (k0 - kt).to(torch.float32)                  # in [-half, -half + 1)
    ph0 = torch.remainder(-carrier * R, 2.0 * math.pi).to(torch.float32)
    u = frac[..., None] + j                             # sample offset from the echo centre
    ph = ph0[..., None] + chirp_rate * u * u
    val = torch.polar(torch.ones_like(ph), ph) * amp.to(torch.complex64)[..., None]
    k = k0.to(torch.int64)[..., None] + j.to(torch.int64)
    dummy = acc.shape[0] - 1
    idx = rows[..., None] * nr + k
    idx = torch.where((k >= 0) & (k < nr), idx, torch.full_like(idx, dummy))
    acc.index_add_(0, idx.reshape(-1), torch.view_as_real(val).reshape(-1, 2))


def add_echoes(raw: torch.Tensor, pos: torch.Tensor, xyz: torch.Tensor, amp: torch.Tensor,
               radar: Radar, scat_chunk: int = 4096) -> None:
    """Add the sampled echoes of point scatterers into raw [Na][Nr] (complex64, in place).

    Geometry and carrier phase are evaluated in float64; the chirp phase of each
    sample is evaluated in float32 from an fp64 fractional offset (its error is
    below 1e-4 rad).  Accumulation uses index_add_, whose summation order is not
    fixed on CUDA: scenes generated on a GPU agree between runs to float32
    rounding only.
    """
    device = raw.device
    na, nr = raw.shape
    if xyz.shape[0] == 0:
        return
    xyz = xyz.to(device)
    amp = amp.to(device)
    nc = chirp_count(radar)
    acc = torch.zeros(na * nr + 1, 2, dtype=torch.float32, device=device)
    sc = min(scat_chunk, xyz.shape[0])
    pulse_chunk = max(1, min(na, (1 << 25) // (sc * nc)))
    for s0 in range(0, xyz.shape[0], sc):
        sx = xyz[s0:s0 + sc]
        sa = amp[s0:s0 + sc]
        for p0 in range(0, na, pulse_chunk):
            a = pos[p0:p0 + pulse_chunk].to(device)
            R = torch.linalg.vector_norm(sx[None, :, :] - a[:, None, :], dim=2)        # [P,S] f64
            rows = torch.arange(p0, p0 + a.shape[0], device=device, dtype=torch.int64)[:, None].expand_as(R)
            _accumulate(acc, rows, R, sa[None, :].expand_as(R), radar, nr)
    torch.view_as_real(raw).reshape(-1, 2).add_(acc[:-1])


def add_noise(raw: torch.Tensor, snr_db: float, seed: int) -> None:
    g = _gen(seed, 3, raw.device)
    s = math.sqrt(10.0 ** (-snr_db / 10.0) / 2.0)
    noise = torch.randn(raw.shape + (2,), generator=g, device=raw.device, dtype=torch.float32) * s
    raw += torch.view_as_complex(noise)


def make_scene(cfg_id, device="cpu", with_clutter: bool = True, with_noise: bool = True):
    """Build one of the benchmark scenes.  Returns a dict with
    raw [Na][Nr] complex64, pos [Na][3] float64, radar, grid, config, and the
    point targets (xyz, amplitude, pixel index or None)."""
    cfg = SCENES[cfg_id] if isinstance(cfg_id, int) else cfg_id
    radar = cfg.radar()
    grid = cfg.grid()
    pos = track(cfg, device)
    raw = torch.zeros(cfg.n_pulses, cfg.n_range, dtype=torch.complex64, device=device)
    txyz, tamp, tpix = targets(cfg)
    add_echoes(raw, pos, txyz, tamp, radar)
    if with_clutter and cfg.clutter_cell > 0:
        cxyz, camp = clutter(cfg)
        add_echoes(raw, pos, cxyz, camp, radar)
    if with_noise:
        add_noise(raw, cfg.snr_db, cfg.seed)
    return dict(raw=raw, pos=pos, radar=radar, grid=grid, config=cfg,
                target_xyz=txyz, target_amp=tamp, target_pix=tpix)


def make_rc_sweep(nr: int, n_lines: int = 4096, seed: int = 1005, device="cpu", snr_db: float = 20.0):
    """Range-compression-only workload: each line holds one unit chirp at a random
    delay that lies fully inside the window, with a random phase, plus noise."""
    radar = Radar(range_start=5000.0, n_pulses=n_lines, n_range=nr, upsample=1)
    g = _gen(seed + nr, 0, "cpu")
    nc = chirp_count(radar)
    d1 = C0 / (2.0 * radar.fs)
    # echo centre kt (in samples) such that the whole pulse [kt - nc/2, kt + nc/2) lies in [0, nr)
    kt = nc / 2.0 + torch.rand(n_lines, generator=g, dtype=torch.float64) * (nr - nc - 1)
    R = radar.range_start + kt * d1
    phase = torch.rand(n_lines, generator=g, dtype=torch.float64) * 2 * math.pi
    raw = torch.zeros(n_lines, nr, dtype=torch.complex64, device=device)
    carrier = 4.0 * math.pi * radar.fc / C0
    # the carrier term of the echo is undone so that each line's compressed phase is `phase`
    amp = torch.polar(torch.ones(n_lines, dtype=torch.float64), phase + carrier * R)
    acc = torch.zeros(n_lines * nr + 1, 2, dtype=torch.float32, device=device)
    rows = torch.arange(n_lines, device=device, dtype=torch.int64)
    _accumulate(acc, rows, R.to(device), amp.to(device), radar, nr)
    torch.view_as_real(raw).reshape(-1, 2).add_(acc[:-1])
    add_noise(raw, snr_db, seed + nr)
    return dict(raw=raw, radar=radar, delay_samples=kt, phase=phase)
