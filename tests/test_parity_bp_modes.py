"""The backprojection variants (sar_plan_set_accumulation, sar_plan_set_stage_precision,
sar_plan_set_interpolation) through the C ABI against the fp64 oracle: the same
bar as the default kernel (relative L2 <= 1e-3, identical peak pixels, peaks
within 0.05 dB).  Compensated sums and float16 staging compute the oracle's
linear-interpolation image; the 8-tap sinc variant the oracle's sinc image."""
import dataclasses

import numpy as np
import pytest
import torch

import domain_backprojection_gb300 as sar
import oracle
import synth
from helpers import IMG_TOL, ORACLE_THREADS, check_peaks, oracle_image_pixels, rel_l2, target_pixels, window_pixels

pytestmark = pytest.mark.gpu

MODES = {
    "compensated": (lambda p: sar.sar_plan_set_accumulation(p, sar.SAR_ACCUM_COMPENSATED), oracle.INTERP_LINEAR),
    "fp16_stage": (lambda p: sar.sar_plan_set_stage_precision(p, sar.SAR_STAGE_FP16), oracle.INTERP_LINEAR),
    "sinc8": (lambda p: sar.sar_plan_set_interpolation(p, sar.SAR_INTERP_SINC8), oracle.INTERP_SINC8),
}


def _plan(s, mode, grid=None):
    plan = sar.sar_plan_create(s["radar"], grid or s["grid"], 0)
    MODES[mode][0](plan)
    return plan


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("cfg", [1, 2])
def test_mode_full_image(scene_cache, mode, cfg):
    s = scene_cache(cfg)
    plan = _plan(s, mode)
    img = sar.sar_form_image(plan, s["raw"], s["pos"])
    sar.sar_plan_sync(plan)
    rc = oracle.range_compress(s["radar"], s["raw"].cpu().numpy(), threads=ORACLE_THREADS)
    ref = oracle.backproject(s["radar"], s["grid"], rc, s["pos"].cpu().numpy(), threads=ORACLE_THREADS,
                             interp=MODES[mode][1])
    got = img.cpu().numpy()
    assert rel_l2(got, ref) <= IMG_TOL
    check_peaks(got, ref, s["grid"], target_pixels(s), 6)


@pytest.mark.parametrize("mode", list(MODES))
def test_mode_spotlight_sampled(scene_cache, mode):
    s = scene_cache(3)
    grid = s["grid"]
    plan = _plan(s, mode)
    img = sar.sar_form_image(plan, s["raw"], s["pos"])
    sar.sar_plan_sync(plan)
    got = img.cpu().numpy()
    rand = np.random.default_rng(33).choice(grid.nx * grid.ny, 2048, replace=False)
    tp = target_pixels(s)
    pix = np.unique(np.concatenate([rand, window_pixels(grid, tp, 6)]))
    ref = oracle_image_pixels(s["radar"], grid, s["raw"].cpu().numpy(), s["pos"].cpu().numpy(), pix,
                              interp=MODES[mode][1])
    assert rel_l2(got.ravel()[pix], ref) <= IMG_TOL
    full_ref = np.zeros(grid.nx * grid.ny, complex)
    full_ref[pix] = ref
    check_peaks(got, full_ref.reshape(grid.ny, grid.nx), grid, tp, 6)


def test_compensated_sums_no_worse_on_the_long_aperture(scene_cache):
    # 16384 pulses: the compensated variant's error against the oracle is at most the plain one's
    s = scene_cache(4)
    grid = s["grid"]
    rand = np.random.default_rng(44).choice(grid.nx * grid.ny, 1024, replace=False)
    ref = oracle_image_pixels(s["radar"], grid, s["raw"].cpu().numpy(), s["pos"].cpu().numpy(), rand)
    errs = {}
    for comp in (False, True):
        plan = sar.sar_plan_create(s["radar"], grid, 0)
        if comp:
            sar.sar_plan_set_accumulation(plan, sar.SAR_ACCUM_COMPENSATED)
        img = sar.sar_form_image(plan, s["raw"], s["pos"])
        sar.sar_plan_sync(plan)
        errs[comp] = rel_l2(img.cpu().numpy().ravel()[rand], ref)
        del plan, img
    assert errs[True] <= IMG_TOL
    assert errs[True] <= errs[False] * 1.02, errs


@pytest.mark.parametrize("mode", list(MODES))
def test_mode_pulse_weights_blocks_and_bounds(mode, monkeypatch):
    # pulse weights, two pulse blocks accumulated, and the bounds-checked build (no flag raised)
    monkeypatch.setenv("SAR_CHECK_BOUNDS", "1")
    cfg = dataclasses.replace(synth.SCENES[1], n_pulses=96, prf=300.0 * 96 / 256, nx=45, ny=70,
                              fixed_target_offsets=((0, 0), (-9, 11), (13, -20)))
    s = synth.make_scene(cfg, device="cuda")
    plan = _plan(s, mode)
    w = torch.hamming_window(96, periodic=False, dtype=torch.float32, device="cuda")
    sar.sar_plan_set_pulse_weights(plan, w)
    rc = sar.sar_range_compress(plan, s["raw"])
    img = sar.sar_backproject(plan, rc, s["pos"], 0, 40)
    sar.sar_backproject(plan, rc, s["pos"], 40, 56, image=img, accumulate=True)
    sar.sar_plan_sync(plan)
    rc_w = (rc * w[:, None]).cpu().numpy()
    ref = oracle.backproject(s["radar"], s["grid"], rc_w, s["pos"].cpu().numpy(), interp=MODES[mode][1])
    assert rel_l2(img.cpu().numpy(), ref) <= IMG_TOL


def test_sinc_at_low_upsampling(scene_cache):
    # sinc interpolation of x2 lines: compared with the oracle's sinc image of the same lines
    cfg = dataclasses.replace(synth.SCENES[2], upsample=2)
    s = synth.make_scene(cfg, device="cuda")
    plan = _plan(s, "sinc8")
    img = sar.sar_form_image(plan, s["raw"], s["pos"])
    sar.sar_plan_sync(plan)
    rc = oracle.range_compress(s["radar"], s["raw"].cpu().numpy(), threads=ORACLE_THREADS)
    ref = oracle.backproject(s["radar"], s["grid"], rc, s["pos"].cpu().numpy(), threads=ORACLE_THREADS,
                             interp=oracle.INTERP_SINC8)
    assert rel_l2(img.cpu().numpy(), ref) <= IMG_TOL


def test_option_setters():
    s = synth.make_scene(dataclasses.replace(synth.SCENES[1], n_pulses=16, nx=8, ny=8), device="cuda")
    plan = sar.sar_plan_create(s["radar"], s["grid"], 0)
    sar.sar_plan_set_interpolation(plan, sar.SAR_INTERP_SINC8)
    with pytest.raises(sar.SarError) as e:                       # a second non-default option
        sar.sar_plan_set_accumulation(plan, sar.SAR_ACCUM_COMPENSATED)
    assert e.value.status == 2
    with pytest.raises(sar.SarError) as e:
        sar.sar_plan_set_stage_precision(plan, sar.SAR_STAGE_FP16)
    assert e.value.status == 2
    sar.sar_plan_set_accumulation(plan, sar.SAR_ACCUM_FP32)       # resetting another option: no change
    sar.sar_plan_set_interpolation(plan, sar.SAR_INTERP_LINEAR)
    sar.sar_plan_set_accumulation(plan, sar.SAR_ACCUM_COMPENSATED)
    for setter in (sar.sar_plan_set_accumulation, sar.sar_plan_set_stage_precision, sar.sar_plan_set_interpolation):
        with pytest.raises(sar.SarError) as e:
            setter(plan, 7)
        assert e.value.status == 1
    rc_only = sar.sar_plan_create(s["radar"], None, 0)
    with pytest.raises(sar.SarError) as e:
        sar.sar_plan_set_interpolation(rc_only, sar.SAR_INTERP_SINC8)
    assert e.value.status == 2
