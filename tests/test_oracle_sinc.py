"""Pins for the oracle's 8-tap sinc interpolation ("GPU-accelerated backprojection
SAR imaging", section 2.2: nearest, linear or sinc interpolation of the compressed
line, sinc being the accurate one).  Reading: h(d) = sinc(d) (1 + cos(pi d / 4)) / 2
on |d| < 4, taps k = -3 .. 4 around floor(q), weights normalised to unit sum.
Checked against the sinc's zeros, exact reproduction at sample positions and of a
constant, the exact values of band-limited tones (an independent closed form), the
point-target gain and the brute-force exact-delay correlation."""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from synth.scenes import add_echoes, chirp_count

SINC, LIN = oracle.INTERP_SINC8, oracle.INTERP_LINEAR


def test_kernel_zeros_symmetry_and_support():
    assert oracle.sinc8_kernel(0.0) == 1.0
    for d in (1, 2, 3, 4, 5, 7.5):
        assert abs(oracle.sinc8_kernel(d)) < 1e-15 and abs(oracle.sinc8_kernel(-d)) < 1e-15
    for d in (0.1, 0.5, 1.3, 2.7, 3.9):
        assert oracle.sinc8_kernel(d) == oracle.sinc8_kernel(-d)
    assert 0.0 < oracle.sinc8_kernel(0.5) < 1.0
    assert oracle.sinc8_kernel(1.5) < 0.0 < oracle.sinc8_kernel(2.5)      # sinc's alternating lobes


def test_samples_and_constants_reproduced():
    rng = np.random.default_rng(3)
    line = rng.standard_normal(64) + 1j * rng.standard_normal(64)
    q = np.arange(4, 60, dtype=float)
    assert np.abs(oracle.interp_line(line, q, SINC) - line[4:60]).max() < 1e-14
    const = np.full(64, 0.7 - 0.2j)
    q = np.linspace(4.0, 58.0, 217)
    assert np.abs(oracle.interp_line(const, q, SINC) - const[0]).max() < 1e-14


@pytest.mark.parametrize("nu,bound", [(0.052, 3e-3), (0.1, 7e-3), (0.208, 5e-3)])
def test_band_limited_tone(nu, bound):
    # nu = 0.052 cycles per sample is the chirp band edge of x8 upsampled lines, 0.208 of x2 lines
    x = np.arange(128)
    line = np.exp(2j * math.pi * nu * x)
    q = np.linspace(40.0, 80.0, 401)
    exact = np.exp(2j * math.pi * nu * q)
    err_sinc = np.abs(oracle.interp_line(line, q, SINC) - exact).max()
    err_lin = np.abs(oracle.interp_line(line, q, LIN) - exact).max()
    assert err_sinc < bound
    assert err_sinc < err_lin / 4


def test_outside_line_is_zero():
    line = np.ones(16, complex)
    # near the start, taps before sample 0 read zero, so a constant line no longer interpolates to
    # the constant; far outside, every tap reads zero
    assert abs(oracle.interp_line(line, np.array([0.5]), SINC)[0] - 1.0) > 1e-3
    assert abs(oracle.interp_line(line, np.array([8.5]), SINC)[0] - 1.0) < 1e-14
    assert oracle.interp_line(line, np.array([40.0]), SINC)[0] == 0.0


def _scene(cfg, pix, amp):
    radar, grid = cfg.radar(), cfg.grid()
    pos = synth.track(cfg)
    xyz = torch.tensor([[grid.x0 + pix[0] * grid.dx, grid.y0 + pix[1] * grid.dy, grid.z0]], dtype=torch.float64)
    raw = torch.zeros(cfg.n_pulses, cfg.n_range, dtype=torch.complex64)
    add_echoes(raw, pos, xyz, torch.tensor([amp], dtype=torch.complex128), radar)
    return radar, grid, pos.numpy(), raw.numpy()


def test_point_target_gain_with_sinc():
    cfg = dataclasses.replace(synth.SCENES[1], nx=32, ny=32)
    radar, grid, pos, raw = _scene(cfg, (16, 12), 0.8 * np.exp(1j * 0.4))
    rc = oracle.range_compress(radar, raw)
    img = oracle.backproject(radar, grid, rc, pos, interp=SINC)
    iy, ix = np.unravel_index(np.abs(img).argmax(), img.shape)
    assert (ix, iy) == (16, 12)
    gain_db = 20 * np.log10(np.abs(img[iy, ix]) / (cfg.n_pulses * chirp_count(radar) * 0.8))
    assert -0.05 < gain_db <= 0.01
    assert abs(math.remainder(np.angle(img[iy, ix]) - 0.4, 2 * math.pi)) < 0.01


@pytest.mark.parametrize("upsample", [8, 2])
def test_brute_force_correlation_closer_than_linear(upsample):
    # the exact-delay time-domain correlation (no FFT, no interpolation) as in the linear pin; sinc
    # interpolation of the same compressed lines must land closer to it than linear interpolation,
    # and at x2 upsampling far closer
    cfg = dataclasses.replace(synth.SCENES[1], n_pulses=16, prf=300.0 / 16 * 2, n_range=1024, nx=16, ny=16,
                              upsample=upsample)
    radar, grid = cfg.radar(), cfg.grid()
    pos = synth.track(cfg)
    g = torch.Generator().manual_seed(7)
    xyz = torch.stack([grid.x0 + torch.rand(3, generator=g, dtype=torch.float64) * 16 * grid.dx,
                       grid.y0 + torch.rand(3, generator=g, dtype=torch.float64) * 16 * grid.dy,
                       torch.zeros(3, dtype=torch.float64)], 1)
    amp = torch.tensor([1.0, 0.6 - 0.3j, -0.5j], dtype=torch.complex128)
    raw = torch.zeros(cfg.n_pulses, cfg.n_range, dtype=torch.complex64)
    add_echoes(raw, pos, xyz, amp, radar)
    raw = raw.numpy()
    pos = pos.numpy()
    rc = oracle.range_compress(radar, raw)
    img_s = oracle.backproject(radar, grid, rc, pos, interp=SINC)
    img_l = oracle.backproject(radar, grid, rc, pos, interp=LIN)
    K = radar.bandwidth / radar.pulse_width
    tk = 2 * radar.range_start / synth.C0 + np.arange(cfg.n_range) / radar.fs
    ix, iy = np.meshgrid(np.arange(grid.nx), np.arange(grid.ny))
    px, py = grid.x0 + ix * grid.dx, grid.y0 + iy * grid.dy
    bf = np.zeros((grid.ny, grid.nx), complex)
    raw = raw.astype(np.complex128)
    for n in range(cfg.n_pulses):
        R = np.sqrt((px - pos[n, 0]) ** 2 + (py - pos[n, 1]) ** 2 + (grid.z0 - pos[n, 2]) ** 2)
        tau = tk[None, None, :] - 2 * R[..., None] / synth.C0
        inside = (tau >= -radar.pulse_width / 2) & (tau < radar.pulse_width / 2)
        ref = np.where(inside, np.exp(-1j * math.pi * K * tau ** 2), 0)
        bf += (ref * raw[n][None, None, :]).sum(-1) * np.exp(1j * 4 * math.pi * radar.fc * R / synth.C0)
    rel_s = np.linalg.norm(img_s - bf) / np.linalg.norm(bf)
    rel_l = np.linalg.norm(img_l - bf) / np.linalg.norm(bf)
    assert rel_s < (rel_l if upsample == 8 else rel_l / 5)
    assert rel_s < 1e-2
