"""Pins for the oracle's time-domain backprojection ("GPU-accelerated
backprojection SAR imaging", sections 1.1, 2.2 and 3.3: per pixel, a sum
over pulses of the linearly interpolated compressed echo at the pixel's range
times exp(+j 4 pi R / lambda)), checked against closed forms of a point target,
invariants, and a brute-force time-domain correlation that uses no FFT and no
interpolation."""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from synth.scenes import add_echoes, chirp_count

CFG1 = synth.SCENES[1]


def single_target_scene(cfg, pix, amp=1.0 + 0j, noise=False):
    """Noise-free echoes of one scatterer on a pixel centre, from the forward model."""
    radar, grid = cfg.radar(), cfg.grid()
    pos = synth.track(cfg)
    xyz = torch.tensor([[grid.x0 + pix[0] * grid.dx, grid.y0 + pix[1] * grid.dy, grid.z0]], dtype=torch.float64)
    raw = torch.zeros(cfg.n_pulses, cfg.n_range, dtype=torch.complex64)
    add_echoes(raw, pos, xyz, torch.tensor([amp], dtype=torch.complex128), radar)
    return radar, grid, pos.numpy(), raw.numpy()


@pytest.fixture(scope="module")
def cfg1_single():
    radar, grid, pos, raw = single_target_scene(CFG1, (70, 58), amp=0.8 * np.exp(1j * 0.4))
    rc = oracle.range_compress(radar, raw)
    img = oracle.backproject(radar, grid, rc, pos)
    return radar, grid, pos, raw, rc, img


def test_point_target_peak_pixel_and_gain(cfg1_single):
    radar, grid, pos, raw, rc, img = cfg1_single
    iy, ix = np.unravel_index(np.abs(img).argmax(), img.shape)
    assert (ix, iy) == (70, 58)
    # coherent gain: Na pulses x Nchirp samples x |a|; linear interpolation at U = 8 loses < 0.2 dB
    gain_db = 20 * np.log10(np.abs(img[iy, ix]) / (CFG1.n_pulses * chirp_count(radar) * 0.8))
    assert -0.2 < gain_db <= 0.01
    # the focused pixel carries the scatterer's own phase (carrier phase fully compensated)
    assert abs(math.remainder(np.angle(img[iy, ix]) - 0.4, 2 * math.pi)) < 0.01


def _first_sidelobe_db(mag):
    pk = int(np.argmax(mag))
    db = 20 * np.log10(mag / mag[pk])
    out = []
    for side in (+1, -1):
        i = pk
        while db[i + side] < db[i]:
            i += side
        j = i
        while db[j + side] > db[j]:
            j += side
        out.append(db[j])
    return out


def _cut_grid(grid, centre, along, step, half):
    """A one-dimensional dense pixel line through `centre` (metres), along x or y."""
    n = 2 * half + 1
    if along == "x":
        return synth.Grid(x0=centre[0] - half * step, y0=centre[1], z0=grid.z0, dx=step, dy=grid.dy, nx=n, ny=1)
    return synth.Grid(x0=centre[0], y0=centre[1] - half * step, z0=grid.z0, dx=grid.dx, dy=step, nx=1, ny=n)


def test_azimuth_and_range_sidelobes(cfg1_single):
    # unweighted aperture and unweighted chirp: first sidelobes of about -13 dB (section 3.1);
    # measured on a dense line of pixels (spacing <= resolution / 16), not on the 0.5 m grid
    radar, grid, pos, raw, rc, img = cfg1_single
    centre = (grid.x0 + 70 * grid.dx, grid.y0 + 58 * grid.dy)
    az = oracle.backproject(radar, _cut_grid(grid, centre, "x", 0.05, 120), rc, pos).ravel()
    rg = oracle.backproject(radar, _cut_grid(grid, centre, "y", 0.05, 120), rc, pos).ravel()
    assert int(np.abs(az).argmax()) == 120 and int(np.abs(rg).argmax()) == 120
    for v in _first_sidelobe_db(np.abs(az)):
        assert abs(v - (-13.26)) < 0.3
    for v in _first_sidelobe_db(np.abs(rg)):
        assert abs(v - (-13.26)) < 0.5


def test_linearity():
    radar, grid = CFG1.radar(), CFG1.grid()
    pos = synth.track(CFG1).numpy()
    g = np.random.default_rng(3)
    shape = (CFG1.n_pulses, radar.n_range * radar.upsample)
    r1 = g.standard_normal(shape) + 1j * g.standard_normal(shape)
    r2 = g.standard_normal(shape) + 1j * g.standard_normal(shape)
    sub = synth.Grid(grid.x0, grid.y0, grid.z0, grid.dx, grid.dy, 16, 16)
    a, b = 0.3 - 0.2j, -1.7
    lhs = oracle.backproject(radar, sub, a * r1 + b * r2, pos)
    rhs = a * oracle.backproject(radar, sub, r1, pos) + b * oracle.backproject(radar, sub, r2, pos)
    assert np.abs(lhs - rhs).max() <= 1e-12 * np.abs(rhs).max()


@pytest.mark.parametrize("axis", [0, 1])
def test_translation_shifts_image(cfg1_single, axis):
    # moving the track by one pixel step moves the image by one pixel on the same axis: pins the
    # [ny][nx] layout, the x/y roles and the pixel-centre formula (grid.x0 + ix dx, grid.y0 + iy dy)
    radar, grid, pos, raw, rc, img = cfg1_single
    sub = synth.Grid(grid.x0 + 60 * grid.dx, grid.y0 + 50 * grid.dy, grid.z0, grid.dx, grid.dy, 20, 14)
    base = oracle.backproject(radar, sub, rc, pos)
    shifted_pos = pos.copy()
    shifted_pos[:, axis] += grid.dx if axis == 0 else grid.dy
    moved = oracle.backproject(radar, sub, rc, shifted_pos)
    if axis == 0:
        assert np.abs(moved[:, 1:] - base[:, :-1]).max() <= 1e-8 * np.abs(base).max()
    else:
        assert np.abs(moved[1:, :] - base[:-1, :]).max() <= 1e-8 * np.abs(base).max()


def test_brute_force_time_domain_correlation():
    # I(p) = sum_n sum_k s_n[k] conj(h(t_k - 2R/c0)) exp(+j 4 pi fc R / c0): the exact-delay matched
    # filter, evaluated sample by sample with no FFT and no interpolation.  The oracle (FFT matched
    # filter on integer samples, x8 upsampling, linear interpolation) must agree to about 1e-2.
    cfg = dataclasses.replace(CFG1, n_pulses=16, prf=300.0 / 16 * 2, n_range=1024, nx=16, ny=16)
    radar, grid = cfg.radar(), cfg.grid()
    pos = synth.track(cfg)
    g = torch.Generator().manual_seed(7)
    xyz = torch.stack([grid.x0 + torch.rand(3, generator=g, dtype=torch.float64) * 16 * grid.dx,
                       grid.y0 + torch.rand(3, generator=g, dtype=torch.float64) * 16 * grid.dy,
                       torch.zeros(3, dtype=torch.float64)], 1)
    amp = torch.tensor([1.0, 0.6 - 0.3j, -0.5j], dtype=torch.complex128)
    raw = torch.zeros(cfg.n_pulses, cfg.n_range, dtype=torch.complex64)
    add_echoes(raw, pos, xyz, amp, radar)
    raw = raw.numpy().astype(np.complex128)
    pos = pos.numpy()
    img = oracle.backproject(radar, grid, oracle.range_compress(radar, raw.astype(np.complex64)), pos)

    K = radar.bandwidth / radar.pulse_width
    t0 = 2 * radar.range_start / synth.C0
    tk = t0 + np.arange(cfg.n_range) / radar.fs
    ix, iy = np.meshgrid(np.arange(grid.nx), np.arange(grid.ny))
    px = grid.x0 + ix * grid.dx
    py = grid.y0 + iy * grid.dy
    bf = np.zeros((grid.ny, grid.nx), complex)
    for n in range(cfg.n_pulses):
        R = np.sqrt((px - pos[n, 0]) ** 2 + (py - pos[n, 1]) ** 2 + (grid.z0 - pos[n, 2]) ** 2)
        tau = tk[None, None, :] - 2 * R[..., None] / synth.C0
        inside = (tau >= -radar.pulse_width / 2) & (tau < radar.pulse_width / 2)
        ref = np.where(inside, np.exp(-1j * math.pi * K * tau ** 2), 0)
        bf += (ref * raw[n][None, None, :]).sum(-1) * np.exp(1j * 4 * math.pi * radar.fc * R / synth.C0)
    rel = np.linalg.norm(img - bf) / np.linalg.norm(bf)
    assert rel < 1e-2


def test_pulse_split_with_accumulate_equals_full(cfg1_single):
    radar, grid, pos, raw, rc, img = cfg1_single
    part = oracle.backproject(radar, grid, rc, pos, pulse_begin=0, pulse_count=100)
    oracle.backproject(radar, grid, rc, pos, pulse_begin=100, pulse_count=CFG1.n_pulses - 100, out=part,
                       accumulate=True)
    assert np.abs(part - img).max() <= 1e-12 * np.abs(img).max()


def test_pixel_subset_matches_full_image(cfg1_single):
    radar, grid, pos, raw, rc, img = cfg1_single
    pix = np.array([0, 5, 127, 128 * 58 + 70, 128 * 128 - 1], dtype=np.int64)
    sub = oracle.backproject(radar, grid, rc, pos, pixels=pix)
    assert np.array_equal(sub, img.ravel()[pix])


def test_out_of_window_samples_contribute_zero(cfg1_single):
    # pixels whose range lies outside the compressed window for every pulse image to exactly zero
    radar, grid, pos, raw, rc, img = cfg1_single
    far = synth.Grid(grid.x0, grid.y0 + 2000.0, grid.z0, grid.dx, grid.dy, 4, 4)
    assert np.all(oracle.backproject(radar, far, rc, pos) == 0)
    near = synth.Grid(grid.x0, grid.y0 - 3000.0, grid.z0, grid.dx, grid.dy, 4, 4)
    assert np.all(oracle.backproject(radar, near, rc, pos) == 0)
