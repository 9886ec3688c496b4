"""Failure detection without a GPU fault: a bounded device-side wait that runs out
(the plan's SAR_WAIT_LIMIT_NS knob set to 0 makes the staged kernels test their
line copy once instead of waiting), reported as SAR_ERR_TIMEOUT by
sar_plan_sync with the context still usable; and device allocations that fail
(the SAR_INJECT_ALLOC_FAILURE hook), reported as SAR_ERR_NO_MEMORY with
nothing leaked or left half-built."""
import dataclasses

import numpy as np
import pytest
import torch

import domain_backprojection_gb300 as sar
import oracle
import synth
from helpers import ORACLE_THREADS, RC_TOL, rel_l2

pytestmark = pytest.mark.gpu

SAR_ERR_NO_MEMORY, SAR_ERR_TIMEOUT = 3, 5


def _lines(n, lines, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.complex(torch.randn(lines, n, generator=g), torch.randn(lines, n, generator=g))


def test_wait_that_runs_out_reports_timeout_and_context_survives(monkeypatch):
    # 8192-sample lines with upsampling are staged by bulk copy; with the limit at 0 every CTA finds
    # its first copy still in flight, sets the timeout flag, lets the copy land and returns
    radar = synth.Radar(range_start=5000.0, n_pulses=64, n_range=8192, upsample=2)
    raw = _lines(8192, 64, 1)
    monkeypatch.setenv("SAR_WAIT_LIMIT_NS", "0")
    plan = sar.sar_plan_create(radar, None, 0)
    monkeypatch.delenv("SAR_WAIT_LIMIT_NS")
    sar.sar_range_compress(plan, raw.cuda())
    with pytest.raises(sar.SarError) as e:
        sar.sar_plan_sync(plan)
    assert e.value.status == SAR_ERR_TIMEOUT
    sar.sar_plan_sync(plan)                          # the flag was read and cleared
    # the same device keeps working: a plan with the default limit compresses the lines correctly
    good = sar.sar_plan_create(radar, None, 0)
    rc = sar.sar_range_compress(good, raw.cuda())
    sar.sar_plan_sync(good)
    ref = oracle.range_compress(radar, raw.numpy(), threads=ORACLE_THREADS)
    assert rel_l2(rc.cpu().numpy(), ref) <= RC_TOL


def test_injected_allocation_failures(monkeypatch):
    cfg = dataclasses.replace(synth.SCENES[1], n_pulses=32, nx=16, ny=16)
    radar, grid = cfg.radar(), cfg.grid()
    monkeypatch.setenv("SAR_INJECT_ALLOC_FAILURE", "1")
    with pytest.raises(sar.SarError) as e:                     # the plan's first allocation
        sar.sar_plan_create(radar, grid, 0)
    assert e.value.status == SAR_ERR_NO_MEMORY
    monkeypatch.delenv("SAR_INJECT_ALLOC_FAILURE")
    plan = sar.sar_plan_create(radar, grid, 0)
    s = synth.make_scene(cfg, device="cuda")
    monkeypatch.setenv("SAR_INJECT_ALLOC_FAILURE", "1")
    img = torch.empty(grid.ny, grid.nx, dtype=torch.complex64).pin_memory()
    with pytest.raises(sar.SarError) as e:                     # the host path's lazy buffers
        sar.sar_form_image_host(plan, s["raw"].cpu().pin_memory(), s["pos"].cpu().pin_memory(), img)
    assert e.value.status == SAR_ERR_NO_MEMORY
    monkeypatch.delenv("SAR_INJECT_ALLOC_FAILURE")
    rd_plan = sar.sar_plan_create(dataclasses.replace(synth.SCENES[2].radar(), upsample=1, n_pulses=512), None, 0)
    monkeypatch.setenv("SAR_INJECT_ALLOC_FAILURE", "1")
    with pytest.raises(sar.SarError) as e:                     # the range-Doppler tables
        sar.sar_plan_set_range_doppler(rd_plan, 0.1)
    assert e.value.status == SAR_ERR_NO_MEMORY
    monkeypatch.delenv("SAR_INJECT_ALLOC_FAILURE")
    # after the failures the plan still forms an image (its buffers are allocated on the next call)
    out = sar.sar_form_image_host(plan, s["raw"].cpu().pin_memory(), s["pos"].cpu().pin_memory(), img)
    ref = sar.sar_form_image(plan, s["raw"], s["pos"])
    sar.sar_plan_sync(plan)
    assert np.abs(out.numpy() - ref.cpu().numpy()).max() <= 1e-5 * np.abs(ref.cpu().numpy()).max()
    sar.sar_plan_set_range_doppler(rd_plan, 0.1)


def test_log_trace_on_request():
    # SAR_LOG=1: plan parameters and kernel choices go to stderr (a fresh process: the switch is read
    # once); without it the library prints nothing
    import os
    import subprocess
    import sys
    code = ("import synth, domain_backprojection_gb300 as sar; c = synth.SCENES[1]; "
            "p = sar.sar_plan_create(c.radar(), c.grid(), 0)")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, SAR_LOG="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert "[sar] plan" in r.stderr and "tiles" in r.stderr
    env.pop("SAR_LOG")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "[sar]" not in r.stderr
