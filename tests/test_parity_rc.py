"""GPU range compression (sar_range_compress through the C ABI) against the
fp64 oracle, element by element, within relative L2 2e-4."""
import dataclasses

import numpy as np
import pytest
import torch

import domain_backprojection_gb300 as sar
import oracle
import synth
from helpers import ORACLE_THREADS, RC_TOL, rel_l2

pytestmark = pytest.mark.gpu


def _short_pulse_radar(n, U, n_lines):
    # a 12-sample pulse so that short lines still hold it
    return synth.Radar(bandwidth=150e6, pulse_width=12 / 180e6, fs=180e6, range_start=5000.0, n_pulses=n_lines,
                       n_range=n, upsample=U)


def _noise(lines, n, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.complex(torch.randn(lines, n, generator=g), torch.randn(lines, n, generator=g))


def _run(radar, raw_cpu):
    plan = sar.sar_plan_create(radar, None, 0)
    raw = raw_cpu.cuda()
    rc = sar.sar_range_compress(plan, raw)
    sar.sar_plan_sync(plan)
    assert sar.sar_plan_last_launches(plan) == 1
    return rc.cpu().numpy()


@pytest.mark.parametrize("n,U,lines", [
    (16, 1, 3), (16, 8, 2), (30, 2, 5), (240, 4, 7), (1000, 1, 9), (1000, 8, 3), (1536, 2, 4),
    (1024, 1, 1), (1024, 8, 37), (2048, 8, 64), (4096, 1, 100), (4096, 1, 7), (4096, 1, 1), (4096, 8, 16),
    (6000, 1, 50), (6000, 8, 5), (8192, 1, 33), (8192, 1, 2), (8192, 8, 9), (8192, 4, 3), (4050, 2, 3),
    # Bluestein lengths: 2 * 3^3 * 19, the prime 1009, odd 3 * 5^3, 2 * 23 * 89, odd 3^2 5 7 13;
    # beyond 4096 (M = 16384): the prime 5003, the odd 4097 = 17 * 241, 2 * 3^2 * 5 * 7 * 13, and 8191
    (1026, 1, 5), (1026, 8, 3), (1009, 2, 4), (375, 1, 3), (375, 4, 2), (4094, 4, 2), (4095, 1, 2),
    (5003, 1, 3), (5003, 8, 2), (4097, 2, 2), (8190, 1, 3), (8190, 8, 2), (8191, 4, 2),
])
def test_rc_random_lines(n, U, lines):
    radar = _short_pulse_radar(n, U, lines) if n < 400 else synth.Radar(range_start=5000.0, n_pulses=lines,
                                                                       n_range=n, upsample=U)
    raw = _noise(lines, n, n * 10 + U)
    got = _run(radar, raw)
    ref = oracle.range_compress(radar, raw.numpy(), threads=ORACLE_THREADS)
    assert got.shape == ref.shape
    for i in range(lines):
        assert rel_l2(got[i], ref[i]) <= RC_TOL, f"line {i}"


@pytest.mark.parametrize("nr", tuple(synth.RC_SWEEP_NR) + (4094, 8190))
def test_rc_sweep_full_size(nr):
    # the range-compression-only workload at its full size (4096 lines), sampled lines checked; also
    # at two Bluestein lengths (convolution lengths 8192 and 16384) in the same launch shape
    scene = synth.make_rc_sweep(nr, n_lines=4096, device="cuda")
    radar = scene["radar"]
    plan = sar.sar_plan_create(radar, None, 0)
    rc = sar.sar_range_compress(plan, scene["raw"])
    sar.sar_plan_sync(plan)
    sample = np.arange(0, 4096, 61)
    raw = scene["raw"][sample].cpu().numpy()
    ref = oracle.range_compress(radar, raw, threads=ORACLE_THREADS)
    got = rc[sample].cpu().numpy()
    assert rel_l2(got, ref) <= RC_TOL
    # each line's compressed chirp peaks at its delay with the line's phase
    kt = scene["delay_samples"][sample].numpy()
    pk = np.abs(got).argmax(axis=1)
    assert np.all(np.abs(pk - kt) <= 0.5 + 1e-9)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_rc_scene_configs_sampled(scene_cache, cfg):
    c = synth.SCENES[cfg]
    scene = scene_cache(cfg)
    plan = sar.sar_plan_create(scene["radar"], None, 0)
    rc = sar.sar_range_compress(plan, scene["raw"])
    sar.sar_plan_sync(plan)
    sample = np.linspace(0, c.n_pulses - 1, 12).astype(int)
    ref = oracle.range_compress(scene["radar"], scene["raw"][sample].cpu().numpy(), threads=ORACLE_THREADS)
    assert rel_l2(rc[sample].cpu().numpy(), ref) <= RC_TOL


@pytest.mark.parametrize("n", [4096, 8192])
def test_rc_subset_at_odd_offset(n):
    # a batch that starts at an odd line hands every line to another CTA (persistent CTAs for
    # 8192-point lines): the lines agree with the full batch's to fp32 rounding
    radar = synth.Radar(range_start=5000.0, n_pulses=16, n_range=n, upsample=1)
    plan = sar.sar_plan_create(radar, None, 0)
    raw = _noise(16, n, 11).cuda()
    full = sar.sar_range_compress(plan, raw)
    part = sar.sar_range_compress(plan, raw[5:12].contiguous())
    sar.sar_plan_sync(plan)
    a, b = full[5:12], part
    assert (torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(a)).item() <= 1e-6


def test_rc_subset_of_lines_and_bad_arguments():
    radar = synth.Radar(range_start=5000.0, n_pulses=64, n_range=2048, upsample=8)
    plan = sar.sar_plan_create(radar, None, 0)
    raw = _noise(64, 2048, 3).cuda()
    full = sar.sar_range_compress(plan, raw)
    part = sar.sar_range_compress(plan, raw[10:17].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(full[10:17], part)
    L = sar.lib()
    import ctypes
    # n_lines < 1, misaligned, overlapping input/output
    assert L.sar_range_compress(plan.handle, ctypes.c_void_p(raw.data_ptr()), ctypes.c_void_p(full.data_ptr()), 0,
                                None) == 1
    assert L.sar_range_compress(plan.handle, ctypes.c_void_p(raw.data_ptr() + 8), ctypes.c_void_p(full.data_ptr()),
                                1, None) == 1
    assert L.sar_range_compress(plan.handle, ctypes.c_void_p(full.data_ptr()), ctypes.c_void_p(full.data_ptr()), 1,
                                None) == 1


@pytest.mark.parametrize("n,U", [(4096, 8), (2048, 4), (8192, 2), (6000, 8), (1000, 2), (512, 8)])
def test_rc_polyphase_layout(n, U):
    # plane u of a polyphase line holds the natural samples U m + u
    radar = synth.Radar(range_start=5000.0, n_pulses=5, n_range=n, upsample=U)
    raw = _noise(5, n, 17 * n + U)
    plan = sar.sar_plan_create(radar, None, 0)
    nat = sar.sar_range_compress(plan, raw.cuda())
    sar.sar_plan_set_rc_layout(plan, sar.SAR_RC_POLYPHASE)
    pla = sar.sar_range_compress(plan, raw.cuda())
    sar.sar_plan_sync(plan)
    pla = pla.cpu().numpy().reshape(5, U, n)
    nat = nat.cpu().numpy().reshape(5, n, U).transpose(0, 2, 1)
    assert np.array_equal(pla, nat)
    ref = oracle.range_compress(radar, raw.numpy(), threads=ORACLE_THREADS).reshape(5, n, U).transpose(0, 2, 1)
    assert rel_l2(pla, ref) <= RC_TOL


@pytest.mark.parametrize("window,nbar,sll", [(sar.SAR_WINDOW_HAMMING, 4, 35.0), (sar.SAR_WINDOW_TAYLOR, 4, 35.0),
                                             (sar.SAR_WINDOW_TAYLOR, 6, 40.0)])
@pytest.mark.parametrize("n,U,lines", [(4096, 8, 6), (6000, 1, 20), (1000, 2, 5), (1024, 4, 8)])
def test_rc_range_window(window, nbar, sll, n, U, lines):
    # the weighted matched filter ("GPU-accelerated backprojection SAR imaging", section 3.1)
    radar = synth.Radar(range_start=5000.0, n_pulses=lines, n_range=n, upsample=U)
    raw = _noise(lines, n, n + 7 * U + window)
    plan = sar.sar_plan_create(radar, None, 0)
    sar.sar_plan_set_range_window(plan, window, nbar, sll)
    got = sar.sar_range_compress(plan, raw.cuda()).cpu().numpy()
    ref = oracle.range_compress(radar, raw.numpy(), threads=ORACLE_THREADS, window=window, nbar=nbar, sll_db=sll)
    for i in range(lines):
        assert rel_l2(got[i], ref[i]) <= RC_TOL, f"line {i}"
    # back to the unweighted filter
    sar.sar_plan_set_range_window(plan, sar.SAR_WINDOW_NONE, 0, 0.0)
    got0 = sar.sar_range_compress(plan, raw.cuda()).cpu().numpy()
    assert rel_l2(got0[0], oracle.range_compress(radar, raw[:1].numpy())[0]) <= RC_TOL


def test_range_window_bad_arguments():
    radar = synth.Radar(range_start=5000.0, n_pulses=1, n_range=1024, upsample=1)
    plan = sar.sar_plan_create(radar, None, 0)
    L = sar.lib()
    assert L.sar_plan_set_range_window(plan.handle, 3, 4, 35.0) == 1
    assert L.sar_plan_set_range_window(plan.handle, sar.SAR_WINDOW_TAYLOR, 1, 35.0) == 1
    assert L.sar_plan_set_range_window(plan.handle, sar.SAR_WINDOW_TAYLOR, 4, 0.0) == 1
    assert L.sar_plan_set_range_window(plan.handle, sar.SAR_WINDOW_TAYLOR, 4, float("nan")) == 1
    assert L.sar_plan_set_range_window(plan.handle, sar.SAR_WINDOW_HAMMING, 0, 0.0) == 0


def test_image_from_bluestein_length_lines():
    # a whole image whose lines (1026 samples) go through the Bluestein kernel: range compression
    # (U = 8, natural and polyphase layouts) and backprojection against the oracle
    import dataclasses
    from helpers import IMG_TOL
    cfg = dataclasses.replace(synth.SCENES[1], n_pulses=96, prf=300.0 * 96 / 256, n_range=1026, nx=45, ny=70,
                              fixed_target_offsets=((0, 0), (-9, 11), (13, -20)))
    s = synth.make_scene(cfg, device="cuda")
    plan = sar.sar_plan_create(s["radar"], s["grid"], 0)
    img = sar.sar_form_image(plan, s["raw"], s["pos"])
    rc = sar.sar_range_compress(plan, s["raw"])
    sar.sar_plan_sync(plan)
    ref_rc = oracle.range_compress(s["radar"], s["raw"].cpu().numpy(), threads=ORACLE_THREADS)
    assert rel_l2(rc.cpu().numpy(), ref_rc) <= RC_TOL
    ref = oracle.backproject(s["radar"], s["grid"], ref_rc, s["pos"].cpu().numpy(), threads=ORACLE_THREADS)
    assert rel_l2(img.cpu().numpy(), ref) <= IMG_TOL
