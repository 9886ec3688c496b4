"""Pins for the oracle's range-Doppler image formation ("Fused FFT -> filter -> IFFT
for SAR on Apple Silicon", sections 2.1 and 5.1: range compression, azimuth DFT,
range cell migration correction by sinc interpolation, azimuth matched filter,
azimuth IDFT).  Checked against closed forms that do not come from the oracle's
own formula: the stationary-phase gain and phase of a focused point target, the
loss without migration correction, Parseval's theorem for the phase-only filter,
the -13.26 dB azimuth sidelobe of a uniform aperture, linearity, and the
independent time-domain backprojection of the same compressed lines."""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from synth.scenes import add_echoes, chirp_count


def _target(na, prf, n_t, di, amp=0.8 * np.exp(1j * 0.4)):
    """One scatterer on range bin n_range/2 + di at the along-track position of pulse n_t."""
    cfg = dataclasses.replace(synth.SCENES[2], n_pulses=na, prf=prf, upsample=1)
    radar, pos = cfg.radar(), synth.track(cfg)
    dr = synth.C0 / (2 * radar.fs)
    i_t = cfg.n_range // 2 + di
    R0 = radar.range_start + i_t * dr
    xyz = torch.tensor([[float(pos[n_t, 0]), math.sqrt(R0 ** 2 - cfg.altitude ** 2), 0.0]], dtype=torch.float64)
    raw = torch.zeros(na, cfg.n_range, dtype=torch.complex64)
    add_echoes(raw, pos, xyz, torch.tensor([amp], dtype=torch.complex128), radar)
    rc = oracle.range_compress(radar, raw.numpy())
    du = cfg.velocity / cfg.prf
    return dict(cfg=cfg, radar=radar, pos=pos.numpy(), rc=rc, du=du, i_t=i_t, n_t=n_t, R0=R0, amp=amp)


SHORT = dict(na=512, prf=600.0, n_t=300, di=3)            # 85 m aperture, 0.19 bins of migration
LONG = dict(na=1024, prf=100.0 / 0.28, n_t=500, di=-7)     # 287 m aperture, 2.1 bins of migration


def _closed_form_peak(t):
    # phase-only azimuth filter: the focused peak is Nchirp |a| sqrt(M), with M = 2 L^2 / (lambda R0)
    # the number of Doppler bins the target's azimuth chirp occupies (Parseval), and its phase is
    # arg(a) - pi/4 (stationary phase of the azimuth chirp)
    lam = synth.C0 / t["radar"].fc
    L = t["cfg"].n_pulses * t["du"]
    return chirp_count(t["radar"]) * abs(t["amp"]) * math.sqrt(2 * L * L / (lam * t["R0"]))


@pytest.mark.parametrize("case", [SHORT, LONG])
def test_point_target_focus_gain_and_phase(case):
    t = _target(**case)
    img = oracle.range_doppler(t["radar"], t["rc"], t["du"])
    i, n = np.unravel_index(np.abs(img).argmax(), img.shape)
    assert (i, n) == (t["i_t"], t["n_t"])
    gain_db = 20 * np.log10(abs(img[i, n]) / _closed_form_peak(t))
    assert -0.3 < gain_db < 0.1
    assert abs(math.remainder(np.angle(img[i, n]) - (np.angle(t["amp"]) - math.pi / 4), 2 * math.pi)) < 0.01


def test_migration_correction_is_needed():
    t = _target(**LONG)
    img = oracle.range_doppler(t["radar"], t["rc"], t["du"], rcmc=False)
    i, n = np.unravel_index(np.abs(img).argmax(), img.shape)
    assert 20 * np.log10(abs(img[i, n]) / _closed_form_peak(t)) < -3.0


def test_parseval_without_migration_correction():
    # the azimuth DFT, the unit-magnitude filter and the scaled IDFT preserve energy per range bin
    rng = np.random.default_rng(5)
    radar = synth.Radar(range_start=5000.0, n_pulses=256, n_range=64, upsample=1)
    rc = rng.standard_normal((256, 64)) + 1j * rng.standard_normal((256, 64))
    img = oracle.range_doppler(radar, rc, 0.3, rcmc=False)
    e_in = (np.abs(rc) ** 2).sum(0)
    e_out = (np.abs(img) ** 2).sum(1)
    assert np.abs(e_out / e_in - 1).max() < 1e-12


def test_azimuth_sidelobes():
    t = _target(**SHORT)
    img = oracle.range_doppler(t["radar"], t["rc"], t["du"])
    mag = np.abs(img[t["i_t"]])
    pk = int(mag.argmax())
    db = 20 * np.log10(mag / mag[pk])
    for side in (+1, -1):
        j = pk
        while db[j + side] < db[j]:
            j += side
        k = j
        while db[k + side] > db[k]:
            k += side
        assert abs(db[k] + 13.26) < 0.5


def test_linearity():
    rng = np.random.default_rng(6)
    radar = synth.Radar(range_start=5000.0, n_pulses=128, n_range=96, upsample=1)
    a = rng.standard_normal((128, 96)) + 1j * rng.standard_normal((128, 96))
    b = rng.standard_normal((128, 96)) + 1j * rng.standard_normal((128, 96))
    al, be = 0.7 - 0.2j, -1.3 + 0.4j
    lhs = oracle.range_doppler(radar, al * a + be * b, 0.25)
    rhs = al * oracle.range_doppler(radar, a, 0.25) + be * oracle.range_doppler(radar, b, 0.25)
    assert np.abs(lhs - rhs).max() <= 1e-12 * np.abs(rhs).max()


def test_agrees_with_backprojection_around_a_target():
    # time-domain backprojection of the same lines, evaluated at the ground points of the
    # range-Doppler cells (x of pulse n, slant range of bin i on z = 0): the same peak cell and the
    # same normalised response within the difference of the two filters' spectral weighting
    t = _target(**LONG)
    img = oracle.range_doppler(t["radar"], t["rc"], t["du"])
    radar, pos, cfg = t["radar"], t["pos"], t["cfg"]
    dr = synth.C0 / (2 * radar.fs)
    h = 8
    cells = [(i, n) for i in range(t["i_t"] - h, t["i_t"] + h + 1) for n in range(t["n_t"] - h, t["n_t"] + h + 1)]
    bp = np.zeros(len(cells), complex)
    for k, (i, n) in enumerate(cells):
        y = math.sqrt((radar.range_start + i * dr) ** 2 - cfg.altitude ** 2)
        g = synth.Grid(x0=float(pos[n, 0]), y0=y, z0=0.0, dx=1.0, dy=1.0, nx=1, ny=1)
        bp[k] = oracle.backproject(radar, g, t["rc"], pos).ravel()[0]
    rd = np.array([img[i, n] for i, n in cells])
    bpm, rdm = np.abs(bp) / np.abs(bp).max(), np.abs(rd) / np.abs(rd).max()
    assert np.argmax(bpm) == np.argmax(rdm)
    assert np.linalg.norm(bpm - rdm) / np.linalg.norm(bpm) < 0.25


def test_pulse_spacing_below_quarter_wavelength_rejected():
    radar = synth.Radar(range_start=5000.0, n_pulses=16, n_range=16, upsample=1)
    with pytest.raises(ValueError):
        oracle.range_doppler(radar, np.zeros((16, 16), complex), 0.007)
