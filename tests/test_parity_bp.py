"""GPU backprojection and end-to-end image formation (through the C ABI)
against the fp64 oracle: relative L2 <= 1e-3 over the whole image (over
sampled pixels and every target's window on the large curved-track scene),
identical point-target peak pixels, peak magnitudes within 0.05 dB and
per-target peak-to-background ratios within 0.05 dB."""
import ctypes
import dataclasses
import os

import numpy as np
import pytest
import torch

import domain_backprojection_gb300 as sar
import oracle
import synth
from helpers import (IMG_TOL, ORACLE_THREADS, SNR_HALF, check_peaks, check_snr, oracle_image_pixels, rel_l2,
                     target_pixels, window_pixels)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def scenes(scene_cache):
    return scene_cache


def _oracle_rc(scene):
    return oracle.range_compress(scene["radar"], scene["raw"].cpu().numpy(), threads=ORACLE_THREADS)


@pytest.mark.parametrize("cfg", [1, 2])
def test_form_image_full(scenes, cfg):
    s = scenes(cfg)
    plan = sar.sar_plan_create(s["radar"], s["grid"], 0)
    img = sar.sar_form_image(plan, s["raw"], s["pos"])
    sar.sar_plan_sync(plan)
    assert 2 <= sar.sar_plan_last_launches(plan) <= 4   # range compression, tile parameters, pixel loop (+ slice sum)
    rc = _oracle_rc(s)
    ref = oracle.backproject(s["radar"], s["grid"], rc, s["pos"].cpu().numpy(), threads=ORACLE_THREADS)
    got = img.cpu().numpy()
    assert rel_l2(got, ref) <= IMG_TOL
    check_peaks(got, ref, s["grid"], target_pixels(s), 6)
    check_snr(got, ref, s["grid"], target_pixels(s))
    # backprojection alone from the oracle's own compressed lines (rounded to complex64)
    img2 = sar.sar_backproject(plan, torch.from_numpy(rc.astype(np.complex64)).cuda(), s["pos"])
    sar.sar_plan_sync(plan)
    ref2 = oracle.backproject(s["radar"], s["grid"], rc.astype(np.complex64), s["pos"].cpu().numpy(),
                              threads=ORACLE_THREADS)
    assert rel_l2(img2.cpu().numpy(), ref2) <= IMG_TOL


def test_form_image_spotlight_whole(scenes):
    # the spotlight scene (4096 pulses, 1024 x 1024 pixels): every pixel against the oracle
    s = scenes(3)
    grid = s["grid"]
    plan = sar.sar_plan_create(s["radar"], grid, 0)
    img = sar.sar_form_image(plan, s["raw"], s["pos"])
    sar.sar_plan_sync(plan)
    got = img.cpu().numpy()
    pix = np.arange(grid.nx * grid.ny, dtype=np.int64)
    ref = oracle_image_pixels(s["radar"], grid, s["raw"].cpu().numpy(), s["pos"].cpu().numpy(), pix)
    ref = ref.reshape(grid.ny, grid.nx)
    assert rel_l2(got, ref) <= IMG_TOL
    tp = target_pixels(s)
    check_peaks(got, ref, grid, tp, 6)
    check_snr(got, ref, grid, tp)


def test_form_image_curved_track_sampled(scenes):
    # the large curved-track scene (16384 pulses, 2048 x 2048 pixels): 1024 random pixels and the
    # whole window around every target
    s = scenes(4)
    grid = s["grid"]
    plan = sar.sar_plan_create(s["radar"], grid, 0)
    img = sar.sar_form_image(plan, s["raw"], s["pos"])
    sar.sar_plan_sync(plan)
    got = img.cpu().numpy()
    rng = np.random.default_rng(4)
    rand = rng.choice(grid.nx * grid.ny, 1024, replace=False)
    tp = target_pixels(s)
    win = window_pixels(grid, tp, SNR_HALF)
    pix = np.unique(np.concatenate([rand, win]))
    ref = oracle_image_pixels(s["radar"], grid, s["raw"].cpu().numpy(), s["pos"].cpu().numpy(), pix)
    assert rel_l2(got.ravel()[pix], ref) <= IMG_TOL
    in_rand = np.isin(pix, rand)
    assert rel_l2(got.ravel()[pix[in_rand]], ref[in_rand]) <= IMG_TOL
    full_ref = np.zeros(grid.nx * grid.ny, complex)
    full_ref[pix] = ref
    full_ref = full_ref.reshape(grid.ny, grid.nx)
    check_peaks(got, full_ref, grid, tp, 6)
    check_snr(got, full_ref, grid, tp)


def _small_case(nx=45, ny=70, na=96):
    cfg = dataclasses.replace(synth.SCENES[1], n_pulses=na, prf=300.0 * na / 256, nx=nx, ny=ny,
                              fixed_target_offsets=((0, 0), (-9, 11), (13, -20)))
    return synth.make_scene(cfg, device="cuda")


def test_ragged_grid_and_pulse_blocks():
    s = _small_case()
    plan = sar.sar_plan_create(s["radar"], s["grid"], 0)
    rc = sar.sar_range_compress(plan, s["raw"])
    full = sar.sar_backproject(plan, rc, s["pos"])
    part = sar.sar_backproject(plan, rc, s["pos"], 0, 40)
    sar.sar_backproject(plan, rc, s["pos"], 40, 56, image=part, accumulate=True)
    sar.sar_plan_sync(plan)
    ref = oracle.backproject(s["radar"], s["grid"], rc.cpu().numpy(), s["pos"].cpu().numpy(), threads=ORACLE_THREADS)
    assert rel_l2(full.cpu().numpy(), ref) <= IMG_TOL
    assert rel_l2(part.cpu().numpy(), ref) <= IMG_TOL
    # a single pulse, and an empty pulse range (overwrite -> zeros; accumulate -> unchanged)
    one = sar.sar_backproject(plan, rc, s["pos"], 17, 1)
    ref1 = oracle.backproject(s["radar"], s["grid"], rc.cpu().numpy(), s["pos"].cpu().numpy(), 17, 1)
    assert rel_l2(one.cpu().numpy(), ref1) <= IMG_TOL
    z = sar.sar_backproject(plan, rc, s["pos"], 5, 0)
    keep = full.clone()
    sar.sar_backproject(plan, rc, s["pos"], 5, 0, image=keep, accumulate=True)
    torch.cuda.synchronize()
    assert torch.count_nonzero(z) == 0 and torch.equal(keep, full)


@pytest.mark.parametrize("nx,ny", [(1, 1), (33, 1), (1, 65), (32, 32), (64, 96)])
def test_grid_shapes(nx, ny):
    s = _small_case(nx, ny, na=40)
    plan = sar.sar_plan_create(s["radar"], s["grid"], 0)
    rc = sar.sar_range_compress(plan, s["raw"])
    img = sar.sar_backproject(plan, rc, s["pos"])
    sar.sar_plan_sync(plan)
    ref = oracle.backproject(s["radar"], s["grid"], rc.cpu().numpy(), s["pos"].cpu().numpy())
    assert rel_l2(img.cpu().numpy(), ref) <= IMG_TOL


@pytest.mark.parametrize("x_centre", [175.0, 1500.0])
def test_squinted_grid(x_centre, monkeypatch):
    # a grid off to the side of the track (squint up to ~15 degrees at x = 1500 m): the range
    # gradient along azimuth is large, so neighbouring pixels of a warp read entries several bins
    # apart and tile windows widen; both grids stay inside the compressed window
    s = _small_case(48, 40, na=64)
    g = s["grid"]
    grid = dataclasses.replace(g, x0=x_centre - 0.5 * g.nx * g.dx)
    plan = sar.sar_plan_create(s["radar"], grid, 0)
    rc = sar.sar_range_compress(plan, s["raw"])
    img = sar.sar_backproject(plan, rc, s["pos"])
    sar.sar_plan_sync(plan)
    ref = oracle.backproject(s["radar"], grid, rc.cpu().numpy(), s["pos"].cpu().numpy())
    assert np.linalg.norm(ref) > 0.0
    assert rel_l2(img.cpu().numpy(), ref) <= IMG_TOL
    # the bounds-checked build finds every staged index inside its window on both paths
    monkeypatch.setenv("SAR_CHECK_BOUNDS", "1")
    checked = sar.sar_plan_create(s["radar"], grid, 0)
    img_c = sar.sar_backproject(checked, rc, s["pos"])
    sar.sar_plan_sync(checked)
    assert rel_l2(img_c.cpu().numpy(), img.cpu().numpy()) <= 1e-6


def test_near_squinted_grid_needs_the_quartic_term(monkeypatch):
    # 3.4 km slant range (the expansion's limit for these 128 x 16 tiles of 0.5 m pixels is 3.2 km)
    # and a grid 1 km along track, 16 degrees of squint: the series' quartic term moves the phase
    # by up to ~1e-4 rad at tile corners, so the pixel kernel must keep it (the scenes at 5.8 km
    # stay below 1e-6 rad and leave it out); checked against the oracle with and without bounds
    # checks
    na = 64
    cfg = dataclasses.replace(synth.SCENES[1], n_pulses=na, prf=300.0 * na / 256, nx=48, ny=40,
                              altitude=2000.0, ground_range=2800.0, fixed_target_offsets=((0, 0),))
    s = synth.make_scene(cfg, device="cuda")
    g = s["grid"]
    grid = dataclasses.replace(g, x0=1000.0 - 0.5 * g.nx * g.dx)
    plan = sar.sar_plan_create(s["radar"], grid, 0)
    rc = sar.sar_range_compress(plan, s["raw"])
    img = sar.sar_backproject(plan, rc, s["pos"])
    sar.sar_plan_sync(plan)
    ref = oracle.backproject(s["radar"], grid, rc.cpu().numpy(), s["pos"].cpu().numpy())
    assert np.linalg.norm(ref) > 0.0
    assert rel_l2(img.cpu().numpy(), ref) <= IMG_TOL
    monkeypatch.setenv("SAR_CHECK_BOUNDS", "1")
    checked = sar.sar_plan_create(s["radar"], grid, 0)
    img_c = sar.sar_backproject(checked, rc, s["pos"])
    sar.sar_plan_sync(checked)
    assert rel_l2(img_c.cpu().numpy(), ref) <= IMG_TOL


def test_window_edges_read_zero_outside_the_line():
    # a grid straddling the near and far ends of the compressed window: samples outside [0, U Nr) are zero
    s = _small_case(40, 40, na=32)
    r = s["radar"]
    dr = synth.C0 / (2 * r.fs)
    for edge in (r.range_start, r.range_start + r.n_range * dr):
        g = s["grid"]
        y_edge = float(np.sqrt(max(edge ** 2 - 3000.0 ** 2, 1.0)))
        grid = dataclasses.replace(g, y0=y_edge - 20 * g.dy)
        plan = sar.sar_plan_create(r, grid, 0)
        rc = sar.sar_range_compress(plan, s["raw"])
        img = sar.sar_backproject(plan, rc, s["pos"])
        sar.sar_plan_sync(plan)
        ref = oracle.backproject(r, grid, rc.cpu().numpy(), s["pos"].cpu().numpy())
        assert np.linalg.norm(img.cpu().numpy() - ref) <= IMG_TOL * max(np.linalg.norm(ref), 1e-3)


def test_bounds_checked_build_reports_nothing(monkeypatch):
    monkeypatch.setenv("SAR_CHECK_BOUNDS", "1")
    s = synth.make_scene(1, device="cuda")
    plan = sar.sar_plan_create(s["radar"], s["grid"], 0)
    img = sar.sar_form_image(plan, s["raw"], s["pos"])
    sar.sar_plan_sync(plan)        # raises SAR_ERR_INTERNAL if any staged index left its window
    rc = _oracle_rc(s)
    ref = oracle.backproject(s["radar"], s["grid"], rc, s["pos"].cpu().numpy(), threads=ORACLE_THREADS)
    assert rel_l2(img.cpu().numpy(), ref) <= IMG_TOL


def test_near_field_geometry_is_reported():
    # an antenna 50 m above the grid is inside the range expansion's validity limit: the plan's
    # device flag surfaces as SAR_ERR_UNSUPPORTED at sync, and the next sync is clean again
    s = _small_case(32, 32, na=8)
    pos = s["pos"].clone()
    pos[:, 2] = 50.0
    pos[:, 1] = s["grid"].y0
    plan = sar.sar_plan_create(s["radar"], s["grid"], 0)
    rc = sar.sar_range_compress(plan, s["raw"])
    sar.sar_backproject(plan, rc, pos)
    with pytest.raises(sar.SarError) as e:
        sar.sar_plan_sync(plan)
    assert e.value.status == 2
    sar.sar_plan_sync(plan)


def test_argument_errors():
    s = _small_case(32, 32, na=8)
    plan = sar.sar_plan_create(s["radar"], s["grid"], 0)
    rc = sar.sar_range_compress(plan, s["raw"])
    img = torch.empty(32, 32, dtype=torch.complex64, device="cuda")
    L = sar.lib()
    P = ctypes.c_void_p
    args = lambda b, c: (plan.handle, P(rc.data_ptr()), P(s["pos"].data_ptr()), b, c, P(img.data_ptr()), 0, None)
    assert L.sar_backproject(*args(-1, 1)) == 1
    assert L.sar_backproject(*args(0, 9)) == 1
    assert L.sar_backproject(*args(8, 1)) == 1
    assert L.sar_backproject(*args(0, -1)) == 1
    ws = torch.empty(sar.sar_workspace_size(plan) - 256, dtype=torch.uint8, device="cuda")
    assert L.sar_form_image(plan.handle, P(s["raw"].data_ptr()), P(s["pos"].data_ptr()), P(img.data_ptr()),
                            P(ws.data_ptr()), ws.numel(), None) == 1
    rc_only = sar.sar_plan_create(s["radar"], None, 0)
    assert L.sar_backproject(rc_only.handle, P(rc.data_ptr()), P(s["pos"].data_ptr()), 0, 1, P(img.data_ptr()), 0,
                             None) == 2


def test_form_image_host_matches_device_path():
    s = synth.make_scene(1, device="cuda")
    plan = sar.sar_plan_create(s["radar"], s["grid"], 0)
    dev = sar.sar_form_image(plan, s["raw"], s["pos"])
    raw_h = s["raw"].cpu().pin_memory()
    pos_h = s["pos"].cpu().pin_memory()
    host = sar.sar_form_image_host(plan, raw_h, pos_h)
    torch.cuda.synchronize()
    assert torch.equal(host, dev.cpu())


def test_form_image_host_chunks_match_device_path(scenes):
    # 1024 pulses go in 3 chunks whose copies overlap the kernels; the image equals the
    # device path's up to the float32 order of the chunk sums
    s = scenes(2)
    plan = sar.sar_plan_create(s["radar"], s["grid"], 0)
    dev = sar.sar_form_image(plan, s["raw"], s["pos"])
    host = sar.sar_form_image_host(plan, s["raw"].cpu().pin_memory(), s["pos"].cpu().pin_memory())
    assert sar.sar_plan_last_launches(plan) >= 3 * 3     # per chunk: compression, parameters, pixels (+ slice sum)
    sar.sar_plan_sync(plan)
    assert rel_l2(host.numpy(), dev.cpu().numpy()) <= 1e-5



def test_form_image_host_on_a_caller_stream(scenes):
    # chunks alternate between the caller's stream and the plan's own: on a side stream, two calls
    # in a row with new inputs (twice the echoes: an exactly doubled image, every step being linear
    # and the scaling a power of two) reuse no stale chunk, and with kernel timing on (all chunks on
    # the caller's stream, in turn) the image is bit-identical
    s = scenes(2)
    plan = sar.sar_plan_create(s["radar"], s["grid"], 0)
    raw_h = s["raw"].cpu().pin_memory()
    raw2_h = (s["raw"] * 2).cpu().pin_memory()
    pos_h = s["pos"].cpu().pin_memory()
    side = torch.cuda.Stream()
    one = sar.sar_form_image_host(plan, raw_h, pos_h, stream=side).clone()
    two = sar.sar_form_image_host(plan, raw2_h, pos_h, stream=side).clone()
    assert torch.equal(two, one * 2)
    dev = sar.sar_form_image(plan, s["raw"], s["pos"])
    assert rel_l2(one.numpy(), dev.cpu().numpy()) <= 1e-5
    sar.sar_plan_set_timing(plan, True)
    timed = sar.sar_form_image_host(plan, raw_h, pos_h, stream=side).clone()
    sar.sar_plan_set_timing(plan, False)
    assert torch.equal(timed, one)
    sar.sar_plan_sync(plan)

def test_polyphase_layout_backprojection_matches_natural():
    # the same compressed lines in either layout give the same image
    s = _small_case(70, 45, na=64)
    plan = sar.sar_plan_create(s["radar"], s["grid"], 0)
    nat = sar.sar_range_compress(plan, s["raw"])
    img_nat = sar.sar_backproject(plan, nat, s["pos"])
    sar.sar_plan_set_rc_layout(plan, sar.SAR_RC_POLYPHASE)
    pla = sar.sar_range_compress(plan, s["raw"])
    img_pla = sar.sar_backproject(plan, pla, s["pos"])
    sar.sar_plan_sync(plan)
    U, n = s["radar"].upsample, s["radar"].n_range
    assert torch.equal(pla.reshape(-1, U, n), nat.reshape(-1, n, U).transpose(1, 2))
    assert torch.equal(img_nat, img_pla)
    ref = oracle.backproject(s["radar"], s["grid"], nat.cpu().numpy(), s["pos"].cpu().numpy())
    assert rel_l2(img_pla.cpu().numpy(), ref) <= IMG_TOL
    L = sar.lib()
    assert L.sar_plan_set_rc_layout(plan.handle, 7) == 1


def test_kernel_timing_records_each_call_and_leaves_results_unchanged():
    s = synth.make_scene(1, device="cuda")
    plan = sar.sar_plan_create(s["radar"], s["grid"], 0)
    want = sar.sar_form_image(plan, s["raw"], s["pos"])
    sar.sar_plan_set_timing(plan, True)
    got = [sar.sar_form_image(plan, s["raw"], s["pos"]) for _ in range(3)]
    rc = sar.sar_range_compress(plan, s["raw"])
    t = sar.sar_plan_kernel_times(plan)
    assert t["rc_calls"] == 4 and t["bp_calls"] == 3
    assert t["rc_ms"] > 0.0 and t["bp_ms"] > 0.0
    assert all(torch.equal(g, want) for g in got)
    assert rc.shape[0] == s["raw"].shape[0]
    # read clears the record; timing off records nothing
    sar.sar_plan_set_timing(plan, False)
    sar.sar_form_image(plan, s["raw"], s["pos"])
    t = sar.sar_plan_kernel_times(plan)
    assert t == {"rc_ms": 0.0, "rc_calls": 0, "bp_ms": 0.0, "bp_calls": 0}


@pytest.mark.parametrize("cfg", [1, 3])
def test_form_image_captures_into_a_cuda_graph(scene_cache, cfg):
    # sar_form_image enqueues its launches with no allocation or synchronisation, so a caller can
    # capture it into a CUDA graph and replay it on new echoes copied into the captured buffers
    # (the tiny scene, one pulse slice; the spotlight scene, eight slices and their sum)
    s = scene_cache(cfg)
    plan = sar.sar_plan_create(s["radar"], s["grid"], 0)
    raw = s["raw"].clone()
    pos = s["pos"].clone()
    ws = torch.empty(sar.sar_workspace_size(plan), dtype=torch.uint8, device="cuda")
    img = torch.empty(s["grid"].ny, s["grid"].nx, dtype=torch.complex64, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        sar.sar_form_image(plan, raw, pos, image=img, workspace=ws)      # warm-up outside capture
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sar.sar_form_image(plan, raw, pos, image=img, workspace=ws)
    other = {"raw": torch.roll(s["raw"], 7, dims=0) * (0.5 - 0.25j), "pos": s["pos"] + 0.01}
    for scene in (s, other):
        raw.copy_(scene["raw"])
        pos.copy_(scene["pos"])
        g.replay()
        want = sar.sar_form_image(plan, scene["raw"], scene["pos"])
        torch.cuda.synchronize()
        assert torch.equal(img, want)
    sar.sar_plan_sync(plan)


def test_form_image_with_range_weighting():
    # Hamming-weighted range compression through sar_form_image against the oracle's weighted image
    s = synth.make_scene(1, device="cuda")
    plan = sar.sar_plan_create(s["radar"], s["grid"], 0)
    sar.sar_plan_set_range_window(plan, sar.SAR_WINDOW_HAMMING)
    img = sar.sar_form_image(plan, s["raw"], s["pos"])
    sar.sar_plan_sync(plan)
    rc = oracle.range_compress(s["radar"], s["raw"].cpu().numpy(), threads=ORACLE_THREADS,
                               window=oracle.WINDOW_HAMMING)
    ref = oracle.backproject(s["radar"], s["grid"], rc, s["pos"].cpu().numpy(), threads=ORACLE_THREADS)
    assert rel_l2(img.cpu().numpy(), ref) <= IMG_TOL
    centres = target_pixels(s)
    check_peaks(img.cpu().numpy(), ref, s["grid"], centres, 6)


def test_pulse_weights():
    # a Hamming taper over the aperture: the image is the oracle's backprojection of the compressed
    # lines each scaled by its weight; unit weights give the unweighted image bit for bit
    s = _small_case(48, 40, na=96)
    na = s["radar"].n_pulses
    plan = sar.sar_plan_create(s["radar"], s["grid"], 0)
    rc = sar.sar_range_compress(plan, s["raw"])
    plain = sar.sar_backproject(plan, rc, s["pos"])
    w = torch.tensor(np.hamming(na), dtype=torch.float32, device="cuda")
    sar.sar_plan_set_pulse_weights(plan, w)
    weighted = sar.sar_backproject(plan, rc, s["pos"])
    part = sar.sar_backproject(plan, rc, s["pos"], 0, 50)
    sar.sar_backproject(plan, rc, s["pos"], 50, na - 50, image=part, accumulate=True)
    sar.sar_plan_set_pulse_weights(plan, torch.ones(na, dtype=torch.float32, device="cuda"))
    ones = sar.sar_backproject(plan, rc, s["pos"])
    sar.sar_plan_set_pulse_weights(plan, None)
    again = sar.sar_backproject(plan, rc, s["pos"])
    sar.sar_plan_sync(plan)
    rcw = rc.cpu().numpy() * w.cpu().numpy()[:, None]
    ref = oracle.backproject(s["radar"], s["grid"], rcw, s["pos"].cpu().numpy())
    assert rel_l2(weighted.cpu().numpy(), ref) <= IMG_TOL
    assert rel_l2(part.cpu().numpy(), ref) <= IMG_TOL
    assert torch.equal(ones, plain) and torch.equal(again, plain)
    with pytest.raises(ValueError):
        sar.sar_plan_set_pulse_weights(plan, torch.ones(na + 1, dtype=torch.float32, device="cuda"))


def test_tile_shape_follows_the_range_bound():
    # the plan picks the longest azimuth tile whose half-diagonal h stays within
    # clamp(R_start / 150, 20 m, 32 m): 128 x 16 pixels at 0.5 m (h = 32 m) for the small scene's
    # 4978 m window start, 64 x 32 (h = 17.6 m) when the window starts at 1500 m; with 1 m pixels no
    # shape stays within 32 m, and of the two with the smallest h (35 m) the longer in azimuth,
    # 64 x 32, keeps the range offsets short
    import os
    import re
    import subprocess
    import sys
    code = ("import dataclasses, synth, domain_backprojection_gb300 as sar; c = synth.SCENES[2]; "
            "sar.sar_plan_create(c.radar(), c.grid(), 0); "
            "sar.sar_plan_create(dataclasses.replace(c.radar(), range_start=1500.0), c.grid(), 0); "
            "sar.sar_plan_create(c.radar(), dataclasses.replace(c.grid(), dx=1.0, dy=1.0), 0)")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=dict(os.environ, SAR_LOG="1"),
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    shapes = re.findall(r"tiles \d+ x \d+ of (\d+) x (\d+) pixels", r.stderr)
    assert shapes == [("128", "16"), ("64", "32"), ("64", "32")], r.stderr
