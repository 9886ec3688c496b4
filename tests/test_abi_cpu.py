"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every entry point include/sar.h declares, and rejects invalid
arguments before touching a device."""
import ctypes
import dataclasses
import math
import subprocess

import pytest
import torch

import domain_backprojection_gb300 as sar
import synth
from domain_backprojection_gb300 import _binding as B

RADAR = synth.SCENES[1].radar()
GRID = synth.SCENES[1].grid()


def _create(radar=RADAR, grid=GRID, device=0, out=True):
    L = sar.lib()
    r = B._to_radar(radar) if radar is not None else None
    g = B._to_grid(grid) if grid is not None else None
    h = ctypes.c_void_p()
    return L.sar_plan_create(ctypes.byref(r) if r is not None else None, ctypes.byref(g) if g is not None else None,
                             device, ctypes.byref(h) if out else None)


def test_library_exports_every_declared_symbol():
    names = sar.declared_symbols()
    assert len(names) >= 10
    out = subprocess.run(["nm", "-D", "--defined-only", sar.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    L = sar.lib()
    for n in names:
        assert hasattr(L, n)


def test_status_strings():
    for code in range(7):
        s = sar.sar_status_string(code)
        assert isinstance(s, str) and s
    assert sar.sar_status_string(99) == "unknown status"


def test_null_handles():
    L = sar.lib()
    assert L.sar_plan_destroy(None) == 0
    n = ctypes.c_size_t()
    assert L.sar_workspace_size(None, ctypes.byref(n)) == 1
    assert L.sar_range_compress(None, None, None, 1, None) == 1
    assert L.sar_backproject(None, None, None, 0, 1, None, 0, None) == 1
    assert L.sar_form_image(None, None, None, None, None, 0, None) == 1
    assert L.sar_form_image_host(None, None, None, None, None) == 1
    assert L.sar_plan_sync(None, None) == 1
    assert L.sar_plan_last_launches(None) == 0
    assert L.sar_plan_set_timing(None, 1) == 1
    assert L.sar_plan_set_range_window(None, 1, 4, 35.0) == 1
    assert L.sar_plan_set_pulse_weights(None, None) == 1
    assert L.sar_plan_set_accumulation(None, 1) == 1
    assert L.sar_plan_set_stage_precision(None, 1) == 1
    assert L.sar_plan_set_interpolation(None, 1) == 1
    assert L.sar_plan_set_range_doppler(None, 0.1) == 1
    assert L.sar_range_doppler_workspace_size(None, ctypes.byref(n)) == 1
    assert L.sar_range_doppler(None, None, None, None, 0, None) == 1
    d, i = ctypes.c_double(), ctypes.c_int32()
    assert L.sar_plan_kernel_times(None, ctypes.byref(d), ctypes.byref(i), ctypes.byref(d), ctypes.byref(i)) == 1


@pytest.mark.parametrize("change,expect", [
    (dict(fs=-1.0), 1), (dict(fc=math.nan), 1), (dict(range_start=math.inf), 1), (dict(bandwidth=0.0), 1),
    (dict(n_pulses=0), 1), (dict(upsample=0), 1),
    (dict(n_range=8193), 2),        # odd, beyond the Bluestein limit (8192)
    (dict(n_range=8194), 2),        # 2 * 17 * 241: beyond the Bluestein limit
    (dict(n_range=10000), 2),       # 2^4 5^4, but beyond the on-chip line
    (dict(n_range=16384), 2),       # beyond the on-chip line
    (dict(n_range=15), 2),          # below 16
    (dict(upsample=3), 2), (dict(upsample=16), 2),
    (dict(n_range=256), 2),         # the 360-sample pulse does not fit the line
])
def test_invalid_radar_rejected_before_any_device_call(change, expect):
    assert _create(dataclasses.replace(RADAR, **change)) == expect


def test_invalid_grid_and_outputs():
    assert _create(out=False) == 1
    assert _create(radar=None) == 1
    assert _create(grid=dataclasses.replace(GRID, nx=0)) == 1
    assert _create(grid=dataclasses.replace(GRID, dy=-0.5)) == 1
    assert _create(grid=dataclasses.replace(GRID, x0=math.nan)) == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
@pytest.mark.parametrize("n_range", [1026, 375, 1009, 4096, 6000])
def test_bluestein_and_direct_lengths_pass_validation(n_range):
    # 2 * 3^3 * 19, odd 3 * 5^3 and the prime 1009 go through Bluestein transforms; validation
    # accepts them, so plan creation gets as far as the device (and fails there without a GPU)
    assert _create(dataclasses.replace(RADAR, n_range=n_range)) == 4


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_plan_without_gpu_reports_cuda_error():
    assert _create() == 4
    with pytest.raises(sar.SarError) as e:
        sar.sar_plan_create(RADAR, GRID)
    assert e.value.status == 4
