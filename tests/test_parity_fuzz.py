"""Seeded random configurations through the C ABI against the fp64 oracle: line lengths on every
range-compression path (powers of two, mixed radix, Bluestein with an odd length), every
upsampling factor, pixel spacings that pick each tile shape (128 x 16, 64 x 32, 32 x 64), grids
off the track and ragged against their tiles, both compressed-line layouts, pulse sub-ranges and
the near geometry that keeps the series' quartic term.  Each case checks the compressed lines
against the oracle's (relative L2 <= 2e-4) and the image backprojected from those lines against
the oracle's image of the same lines (<= 1e-3)."""
import dataclasses

import numpy as np
import pytest
import torch

import domain_backprojection_gb300 as sar
import oracle
import synth
from helpers import IMG_TOL, ORACLE_THREADS, RC_TOL, rel_l2

pytestmark = pytest.mark.gpu

# per case: line length, upsampling, pixel spacing (m), near geometry
CASES = [(1024, 8, 0.5, False), (1000, 4, 0.75, False), (1009, 2, 1.0, False), (512, 1, 0.25, False),
         (2048, 8, 0.75, True), (1024, 2, 0.5, True), (750, 8, 1.0, False), (2048, 4, 0.25, False)]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_random_configuration(case):
    n_range, upsample, pixel, near = CASES[case]
    rng = np.random.default_rng(7000 + case)
    na = int(rng.choice([24, 40, 64]))
    nx, ny = int(rng.integers(1, 72)), int(rng.integers(1, 72))
    altitude, ground = (2000.0, 2800.0) if near else (3000.0, 5000.0)
    cfg = dataclasses.replace(synth.SCENES[1], n_pulses=na, n_range=n_range, upsample=upsample,
                              prf=300.0 * na / 256, nx=nx, ny=ny, pixel=pixel, altitude=altitude,
                              ground_range=ground, fixed_target_offsets=((0, 0),), seed=9000 + case)
    s = synth.make_scene(cfg, device="cuda")
    radar, g = s["radar"], s["grid"]
    # the grid moved along track (squint) and across (within the swath), off its pixel lattice
    x_shift = float(rng.uniform(-150.0, 150.0)) + (900.0 if near else 0.0)
    y_shift = float(rng.uniform(-20.0, 20.0))
    grid = dataclasses.replace(g, x0=g.x0 + x_shift + 0.37 * pixel, y0=g.y0 + y_shift + 0.21 * pixel)
    plan = sar.sar_plan_create(radar, grid, 0)
    layout = int(rng.integers(0, 2)) if upsample > 1 else sar.SAR_RC_NATURAL
    sar.sar_plan_set_rc_layout(plan, layout)
    rc = sar.sar_range_compress(plan, s["raw"])
    p0 = int(rng.integers(0, na // 3))
    cnt = int(rng.integers(1, na - p0 + 1))
    img = sar.sar_backproject(plan, rc, s["pos"], p0, cnt)
    sar.sar_plan_sync(plan)
    # the lines in natural order, whichever layout the plan keeps
    got_rc = rc.cpu().numpy()
    if layout == sar.SAR_RC_POLYPHASE:
        got_rc = got_rc.reshape(na, upsample, n_range).transpose(0, 2, 1).reshape(na, upsample * n_range)
    ref_rc = oracle.range_compress(radar, s["raw"].cpu().numpy(), threads=ORACLE_THREADS)
    assert rel_l2(got_rc, ref_rc) <= RC_TOL
    ref = oracle.backproject(radar, grid, got_rc.astype(np.complex64), s["pos"].cpu().numpy(), p0, cnt,
                             threads=ORACLE_THREADS)
    assert np.linalg.norm(ref) > 0.0
    err = rel_l2(img.cpu().numpy(), ref)
    print(f"case {case}: Nr {n_range} U {upsample} pixel {pixel} m, {nx} x {ny}, pulses {p0}+{cnt} of {na}: "
          f"image rel L2 {err:.2e}")
    assert err <= IMG_TOL


# per case: line length, upsampling, pixel spacing (m), along-track grid offset (m), pixel-kernel variant
MODE_CASES = [(4095, 8, 0.5, 0.0, "sinc8"), (5003, 2, 0.5, 300.0, "linear"), (8192, 8, 0.25, -200.0, "compensated"),
              (6000, 4, 0.5, 1200.0, "fp16_stage"), (4096, 1, 0.2, 0.0, "sinc8"), (2000, 8, 0.3, -1500.0, "linear"),
              (1536, 2, 0.75, 600.0, "compensated"), (3000, 8, 0.4, -800.0, "fp16_stage")]
_MODE_SET = {
    "linear": (lambda p: None, oracle.INTERP_LINEAR),
    "compensated": (lambda p: sar.sar_plan_set_accumulation(p, sar.SAR_ACCUM_COMPENSATED), oracle.INTERP_LINEAR),
    "fp16_stage": (lambda p: sar.sar_plan_set_stage_precision(p, sar.SAR_STAGE_FP16), oracle.INTERP_LINEAR),
    "sinc8": (lambda p: sar.sar_plan_set_interpolation(p, sar.SAR_INTERP_SINC8), oracle.INTERP_SINC8),
}


@pytest.mark.parametrize("case", range(len(MODE_CASES)))
def test_random_configuration_variants(case):
    # the pixel-kernel variants and the longer line paths (Bluestein up to 4096 and above it, the
    # staged 8192-point kernel, 6000 points) on squinted grids, through sar_form_image (polyphase
    # planes), against the oracle's compressed lines and its image of those lines with the
    # variant's interpolation
    n_range, upsample, pixel, x_off, mode = MODE_CASES[case]
    rng = np.random.default_rng(8000 + case)
    na = int(rng.choice([16, 24, 32]))
    nx, ny = int(rng.integers(1, 60)), int(rng.integers(1, 60))
    cfg = dataclasses.replace(synth.SCENES[1], n_pulses=na, n_range=n_range, upsample=upsample,
                              prf=300.0 * na / 256, nx=nx, ny=ny, pixel=pixel,
                              fixed_target_offsets=((0, 0),), seed=9500 + case)
    s = synth.make_scene(cfg, device="cuda")
    radar, g = s["radar"], s["grid"]
    grid = dataclasses.replace(g, x0=g.x0 + x_off + 0.29 * pixel, y0=g.y0 + float(rng.uniform(-10.0, 10.0)))
    plan = sar.sar_plan_create(radar, grid, 0)
    _MODE_SET[mode][0](plan)
    img = sar.sar_form_image(plan, s["raw"], s["pos"])
    sar.sar_plan_sync(plan)
    # the same plan's compressed lines, in natural order, for the image reference
    sar.sar_plan_set_rc_layout(plan, sar.SAR_RC_NATURAL)
    rc = sar.sar_range_compress(plan, s["raw"])
    sar.sar_plan_sync(plan)
    got_rc = rc.cpu().numpy()
    ref_rc = oracle.range_compress(radar, s["raw"].cpu().numpy(), threads=ORACLE_THREADS)
    assert rel_l2(got_rc, ref_rc) <= RC_TOL
    ref = oracle.backproject(radar, grid, got_rc.astype(np.complex64), s["pos"].cpu().numpy(),
                             threads=ORACLE_THREADS, interp=_MODE_SET[mode][1])
    assert np.linalg.norm(ref) > 0.0
    err = rel_l2(img.cpu().numpy(), ref)
    print(f"variant case {case}: Nr {n_range} U {upsample} pixel {pixel} m, {nx} x {ny}, x offset {x_off} m, "
          f"{mode}: image rel L2 {err:.2e}")
    assert err <= IMG_TOL


# per case: pulses, line length, upsampling, range window, pulse weights
HOST_CASES = [(512, 1024, 8, "hamming", True), (640, 600, 4, "taylor", False), (768, 512, 2, "none", True),
              (544, 1000, 8, "taylor", True)]


@pytest.mark.parametrize("case", range(len(HOST_CASES)))
def test_random_configuration_host_path(case):
    # sar_form_image_host (pulses copied in chunks that overlap the kernels, from pinned host
    # buffers) with a weighted matched filter and random pulse weights, against the oracle's
    # weighted compression of the same echoes and its image of those lines scaled by the weights
    na, n_range, upsample, window, weighted = HOST_CASES[case]
    rng = np.random.default_rng(8500 + case)
    nx, ny = int(rng.integers(8, 48)), int(rng.integers(8, 48))
    cfg = dataclasses.replace(synth.SCENES[1], n_pulses=na, n_range=n_range, upsample=upsample,
                              prf=300.0 * na / 256, nx=nx, ny=ny, fixed_target_offsets=((0, 0), (3, -2)),
                              seed=9700 + case)
    s = synth.make_scene(cfg, device="cuda")
    radar, grid = s["radar"], s["grid"]
    plan = sar.sar_plan_create(radar, grid, 0)
    win = {"none": (sar.SAR_WINDOW_NONE, oracle.WINDOW_NONE), "hamming": (sar.SAR_WINDOW_HAMMING, oracle.WINDOW_HAMMING),
           "taylor": (sar.SAR_WINDOW_TAYLOR, oracle.WINDOW_TAYLOR)}[window]
    sar.sar_plan_set_range_window(plan, win[0])
    w = None
    if weighted:
        w = torch.tensor(rng.uniform(0.5, 1.5, na), dtype=torch.float32, device="cuda")
        sar.sar_plan_set_pulse_weights(plan, w)
    img = sar.sar_form_image_host(plan, s["raw"].cpu().pin_memory(), s["pos"].cpu().pin_memory())
    sar.sar_plan_sync(plan)
    rc = oracle.range_compress(radar, s["raw"].cpu().numpy(), threads=ORACLE_THREADS, window=win[1])
    if weighted:
        rc = rc * w.cpu().numpy()[:, None]
    ref = oracle.backproject(radar, grid, rc, s["pos"].cpu().numpy(), threads=ORACLE_THREADS)
    err = rel_l2(img.numpy(), ref)
    print(f"host case {case}: {na} pulses, Nr {n_range} U {upsample}, {window} window, weights {weighted}, "
          f"{nx} x {ny}: image rel L2 {err:.2e}")
    assert err <= IMG_TOL


# per case: pulses (a power of two), line length, PRF (Hz)
RD_CASES = [(512, 1024, 200.0), (1024, 600, 900.0), (2048, 512, 2500.0), (512, 4096, 350.0)]


@pytest.mark.parametrize("case", range(len(RD_CASES)))
def test_random_configuration_range_doppler(case):
    # range-Doppler image formation at random pulse counts, line lengths (one a mixed radix) and pulse
    # spacings (so that the range migration and its step between neighbouring range bins vary),
    # against the oracle's range-Doppler image of the same echoes
    na, n_range, prf = RD_CASES[case]
    cfg = dataclasses.replace(synth.SCENES[1], n_pulses=na, n_range=n_range, upsample=1, prf=prf,
                              nx=64, ny=64, fixed_target_offsets=((0, 0), (10, -6)), seed=9800 + case)
    s = synth.make_scene(cfg, device="cuda")
    radar, du = s["radar"], cfg.velocity / cfg.prf
    plan = sar.sar_plan_create(radar, None, 0)
    sar.sar_plan_set_range_doppler(plan, du)
    img = sar.sar_range_doppler(plan, s["raw"])
    sar.sar_plan_sync(plan)
    rc = oracle.range_compress(radar, s["raw"].cpu().numpy(), threads=ORACLE_THREADS)
    ref = oracle.range_doppler(radar, rc, du, threads=ORACLE_THREADS)
    err = rel_l2(img.cpu().numpy(), ref)
    print(f"range-Doppler case {case}: {na} pulses, Nr {n_range}, pulse spacing {du:.3f} m: image rel L2 {err:.2e}")
    assert err <= IMG_TOL


# per case: line length, upsampling, pixel spacing (m), which end of the window, pixel-kernel variant
EDGE_CASES = [(1024, 8, 0.5, "near", "sinc8"), (1000, 2, 0.25, "far", "linear"), (512, 4, 0.75, "near", "fp16_stage"),
              (2048, 1, 0.3, "far", "sinc8")]


@pytest.mark.parametrize("case", range(len(EDGE_CASES)))
def test_random_configuration_window_edges(case):
    # grids straddling the near or far end of the compressed window: every row's gather runs past
    # the line and must read zeros there (the sinc rows three samples before and four after), in
    # each variant
    n_range, upsample, pixel, end, mode = EDGE_CASES[case]
    rng = np.random.default_rng(8700 + case)
    na = int(rng.choice([16, 32]))
    nx, ny = int(rng.integers(4, 40)), int(rng.integers(20, 60))
    cfg = dataclasses.replace(synth.SCENES[1], n_pulses=na, n_range=n_range, upsample=upsample,
                              prf=300.0 * na / 256, nx=nx, ny=ny, pixel=pixel, seed=9900 + case)
    s = synth.make_scene(cfg, device="cuda")
    radar, g = s["radar"], s["grid"]
    edge = radar.range_start + (0.0 if end == "near" else n_range * synth.C0 / (2 * radar.fs))
    y_edge = float(np.sqrt(edge ** 2 - cfg.altitude ** 2))
    grid = dataclasses.replace(g, y0=y_edge - (ny // 2) * pixel + float(rng.uniform(-1.0, 1.0)))
    plan = sar.sar_plan_create(radar, grid, 0)
    _MODE_SET[mode][0](plan)
    rc = sar.sar_range_compress(plan, s["raw"])
    img = sar.sar_backproject(plan, rc, s["pos"])
    sar.sar_plan_sync(plan)
    ref = oracle.backproject(radar, grid, rc.cpu().numpy(), s["pos"].cpu().numpy(), threads=ORACLE_THREADS,
                             interp=_MODE_SET[mode][1])
    err = np.linalg.norm(img.cpu().numpy() - ref) / max(np.linalg.norm(ref), 1e-3)
    print(f"edge case {case}: Nr {n_range} U {upsample} pixel {pixel} m, {end} end, {mode}: image rel L2 {err:.2e}")
    assert err <= IMG_TOL


# per case: line length, chirp duration (s), upsampling, pulses, grid (nx, ny)
SHORT_CASES = [(64, 0.1e-6, 8, 512, (3, 200)), (100, 0.2e-6, 4, 256, (200, 1)), (250, 0.5e-6, 2, 1024, (9, 9)),
               (16, 0.05e-6, 1, 64, (40, 40))]


@pytest.mark.parametrize("case", range(len(SHORT_CASES)))
def test_random_configuration_short_lines(case):
    # short lines of short chirps (the shared-memory mixed-radix kernel at 16..250 samples), extreme
    # grid aspects and many pulses on few pixels (the most pulse slices), against the oracle
    from synth.scenes import add_echoes, targets, track
    n_range, tp, upsample, na, (nx, ny) = SHORT_CASES[case]
    cfg = dataclasses.replace(synth.SCENES[1], n_pulses=na, n_range=n_range, upsample=upsample,
                              prf=300.0 * na / 256, nx=nx, ny=ny, fixed_target_offsets=((0, 0),), seed=9950 + case)
    radar = dataclasses.replace(cfg.radar(), pulse_width=tp)
    grid = cfg.grid()
    pos = track(cfg, "cuda")
    raw = torch.zeros(na, n_range, dtype=torch.complex64, device="cuda")
    xyz, amp, _ = targets(cfg)
    add_echoes(raw, pos, xyz, amp, radar)
    g = torch.Generator(device="cuda").manual_seed(123 + case)
    raw += 0.05 * torch.complex(torch.randn(na, n_range, generator=g, device="cuda"),
                                torch.randn(na, n_range, generator=g, device="cuda"))
    plan = sar.sar_plan_create(radar, grid, 0)
    img = sar.sar_form_image(plan, raw, pos)
    sar.sar_plan_sync(plan)
    rc = oracle.range_compress(radar, raw.cpu().numpy(), threads=ORACLE_THREADS)
    ref = oracle.backproject(radar, grid, rc, pos.cpu().numpy(), threads=ORACLE_THREADS)
    assert np.linalg.norm(ref) > 0.0
    err = rel_l2(img.cpu().numpy(), ref)
    print(f"short case {case}: Nr {n_range} ({round(tp * radar.fs)}-sample chirp) U {upsample}, {na} pulses, "
          f"{nx} x {ny}: image rel L2 {err:.2e}")
    assert err <= IMG_TOL
