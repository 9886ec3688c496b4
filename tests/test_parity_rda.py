"""GPU range-Doppler image formation (sar_range_doppler, through the C ABI) against
the fp64 oracle's range-Doppler image of the same raw echoes: relative L2 <= 1e-3
over the whole image, identical point-target peak cells and peak magnitudes within
0.05 dB; a focused point target's phase equals arg(a) - pi/4; argument errors."""
import ctypes
import dataclasses
import math
import types

import numpy as np
import pytest
import torch

import domain_backprojection_gb300 as sar
import oracle
import synth
from helpers import IMG_TOL, ORACLE_THREADS, check_peaks, rel_l2
from synth.scenes import add_echoes

pytestmark = pytest.mark.gpu


def _u1(scene):
    """The scene's radar at native range sampling and its along-track pulse spacing."""
    cfg = scene["config"]
    return dataclasses.replace(scene["radar"], upsample=1), cfg.velocity / cfg.prf


def _rd_cells(scene, radar, du):
    """(column, row) of every point target in range-Doppler coordinates, rounded."""
    pos = scene["pos"].cpu().numpy()
    alt = scene["config"].altitude
    dr = synth.C0 / (2 * radar.fs)
    out = []
    for x, y, z in scene["target_xyz"].numpy():
        r0 = math.sqrt(y * y + (alt - z) ** 2)
        out.append((int(round((x - pos[0, 0]) / du)), int(round((r0 - radar.range_start) / dr))))
    return out


def _oracle_rd(scene, radar, du):
    rc = oracle.range_compress(radar, scene["raw"].cpu().numpy(), threads=ORACLE_THREADS)
    return oracle.range_doppler(radar, rc, du, threads=ORACLE_THREADS)


@pytest.mark.parametrize("cfg", [2, 3])
def test_range_doppler_matches_oracle(scene_cache, cfg):
    s = scene_cache(cfg)
    radar, du = _u1(s)
    plan = sar.sar_plan_create(radar, None, 0)
    sar.sar_plan_set_range_doppler(plan, du)
    img = sar.sar_range_doppler(plan, s["raw"])
    sar.sar_plan_sync(plan)
    assert sar.sar_plan_last_launches(plan) == 4
    got = img.cpu().numpy()
    ref = _oracle_rd(s, radar, du)
    assert got.shape == ref.shape == (radar.n_range, radar.n_pulses)
    assert rel_l2(got, ref) <= IMG_TOL
    cells = [c for c in _rd_cells(s, radar, du) if 8 <= c[0] < radar.n_pulses - 8 and 8 <= c[1] < radar.n_range - 8]
    assert cells
    check_peaks(got, ref, types.SimpleNamespace(nx=radar.n_pulses, ny=radar.n_range), cells, 4)


def test_point_target_phase_and_position():
    cfg = dataclasses.replace(synth.SCENES[2], n_pulses=1024, prf=100.0 / 0.28, upsample=1)
    radar, pos = cfg.radar(), synth.track(cfg)
    du, dr = cfg.velocity / cfg.prf, synth.C0 / (2 * radar.fs)
    i_t, n_t = cfg.n_range // 2 - 7, 500
    R0 = radar.range_start + i_t * dr
    a = 0.8 * np.exp(1j * 0.4)
    raw = torch.zeros(cfg.n_pulses, cfg.n_range, dtype=torch.complex64)
    xyz = torch.tensor([[float(pos[n_t, 0]), math.sqrt(R0 ** 2 - cfg.altitude ** 2), 0.0]], dtype=torch.float64)
    add_echoes(raw, pos, xyz, torch.tensor([a], dtype=torch.complex128), radar)
    plan = sar.sar_plan_create(radar, None, 0)
    sar.sar_plan_set_range_doppler(plan, du)
    img = sar.sar_range_doppler(plan, raw.cuda()).cpu().numpy()
    i, n = np.unravel_index(np.abs(img).argmax(), img.shape)
    assert (i, n) == (i_t, n_t)
    assert abs(math.remainder(np.angle(img[i, n]) - (0.4 - math.pi / 4), 2 * math.pi)) < 0.01


def test_non_power_of_two_range_and_smallest_aperture():
    cfg = dataclasses.replace(synth.SCENES[2], n_pulses=512, prf=600.0, n_range=1000, upsample=1)
    radar, pos = cfg.radar(), synth.track(cfg)
    g = torch.Generator().manual_seed(9)
    raw = torch.complex(torch.randn(512, 1000, generator=g), torch.randn(512, 1000, generator=g)) * 0.1
    xyz = torch.tensor([[float(pos[200, 0]), 5000.0, 0.0], [float(pos[340, 0]) + 0.03, 5004.1, 0.0]],
                       dtype=torch.float64)
    add_echoes(raw, pos, xyz, torch.tensor([1.0, 0.5j], dtype=torch.complex128), radar)
    du = cfg.velocity / cfg.prf
    plan = sar.sar_plan_create(radar, None, 0)
    sar.sar_plan_set_range_doppler(plan, du)
    got = sar.sar_range_doppler(plan, raw.cuda()).cpu().numpy()
    rc = oracle.range_compress(radar, raw.numpy(), threads=ORACLE_THREADS)
    ref = oracle.range_doppler(radar, rc, du, threads=ORACLE_THREADS)
    assert rel_l2(got, ref) <= IMG_TOL


@pytest.mark.parametrize("na,nr", [(2048, 512), (8192, 768)])
def test_other_aperture_lengths(na, nr):
    # the 2048- and 8192-point azimuth transforms (one CTA per range bin of N/16 threads)
    cfg = dataclasses.replace(synth.SCENES[2], n_pulses=na, prf=1200.0 * na / 1024, n_range=nr, upsample=1)
    radar, pos = cfg.radar(), synth.track(cfg)
    g = torch.Generator().manual_seed(na)
    raw = torch.complex(torch.randn(na, nr, generator=g), torch.randn(na, nr, generator=g)) * 0.05
    xyz = torch.tensor([[float(pos[na // 3, 0]), 5000.0, 0.0], [float(pos[na // 2, 0]) + 0.01, 4998.7, 0.0]],
                       dtype=torch.float64)
    add_echoes(raw, pos, xyz, torch.tensor([1.0, 0.7 - 0.2j], dtype=torch.complex128), radar)
    du = cfg.velocity / cfg.prf
    plan = sar.sar_plan_create(radar, None, 0)
    sar.sar_plan_set_range_doppler(plan, du)
    got = sar.sar_range_doppler(plan, raw.cuda()).cpu().numpy()
    rc = oracle.range_compress(radar, raw.numpy(), threads=ORACLE_THREADS)
    ref = oracle.range_doppler(radar, rc, du, threads=ORACLE_THREADS)
    assert rel_l2(got, ref) <= IMG_TOL


def test_range_doppler_captures_into_a_cuda_graph():
    # sar_range_doppler enqueues its launches with no allocation or synchronisation once the plan's
    # tables exist: capture it once, replay it on new echoes copied into the captured buffer
    cfg = dataclasses.replace(synth.SCENES[2], n_pulses=512, prf=600.0, n_range=1024, upsample=1)
    radar = cfg.radar()
    plan = sar.sar_plan_create(radar, None, 0)
    sar.sar_plan_set_range_doppler(plan, cfg.velocity / cfg.prf)
    raw = torch.zeros(512, 1024, dtype=torch.complex64, device="cuda")
    ws = torch.empty(sar.sar_range_doppler_workspace_size(plan), dtype=torch.uint8, device="cuda")
    img = torch.empty(1024, 512, dtype=torch.complex64, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        sar.sar_range_doppler(plan, raw, img, ws)                    # warm-up outside capture
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sar.sar_range_doppler(plan, raw, img, ws)
    for seed in (1, 2):
        gen = torch.Generator().manual_seed(seed)
        new = torch.complex(torch.randn(512, 1024, generator=gen), torch.randn(512, 1024, generator=gen)).cuda()
        raw.copy_(new)
        g.replay()
        want = sar.sar_range_doppler(plan, new)
        torch.cuda.synchronize()
        assert torch.equal(img, want)
    sar.sar_plan_sync(plan)


def test_range_doppler_arguments():
    radar = dataclasses.replace(synth.SCENES[2].radar(), upsample=1)
    plan = sar.sar_plan_create(radar, None, 0)
    L = sar.lib()
    n = ctypes.c_size_t()
    assert L.sar_range_doppler_workspace_size(plan.handle, ctypes.byref(n)) == 2      # before the tables
    raw = torch.zeros(radar.n_pulses, radar.n_range, dtype=torch.complex64, device="cuda")
    img = torch.empty(radar.n_range, radar.n_pulses, dtype=torch.complex64, device="cuda")
    ws = torch.empty(2 * raw.numel() * 8, dtype=torch.uint8, device="cuda")
    P = ctypes.c_void_p
    assert L.sar_range_doppler(plan.handle, P(raw.data_ptr()), P(img.data_ptr()), P(ws.data_ptr()), ws.numel(),
                               None) == 2
    assert L.sar_plan_set_range_doppler(plan.handle, -1.0) == 1
    assert L.sar_plan_set_range_doppler(plan.handle, math.nan) == 1
    assert L.sar_plan_set_range_doppler(plan.handle, 0.005) == 2       # lambda / (4 du) >= 1
    sar.sar_plan_set_range_doppler(plan, 0.0833)
    assert L.sar_range_doppler_workspace_size(plan.handle, ctypes.byref(n)) == 0 and n.value == ws.numel()
    assert L.sar_range_doppler(plan.handle, P(raw.data_ptr()), P(img.data_ptr()), P(ws.data_ptr()), ws.numel() - 1,
                               None) == 1
    assert L.sar_range_doppler(plan.handle, P(raw.data_ptr() + 8), P(img.data_ptr()), P(ws.data_ptr()), ws.numel(),
                               None) == 1
    up8 = sar.sar_plan_create(dataclasses.replace(radar, upsample=8), None, 0)
    assert L.sar_plan_set_range_doppler(up8.handle, 0.0833) == 2
    odd = sar.sar_plan_create(dataclasses.replace(radar, n_pulses=300), None, 0)
    assert L.sar_plan_set_range_doppler(odd.handle, 0.0833) == 2
