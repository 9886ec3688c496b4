"""sar_form_image_noalloc: the image-formation entry point that allocates no
device memory, for callers that cannot call cudaMalloc when they form an image
(device memory fixed at start-up, or owned by an allocator the library cannot
use).  Its compressed-line scratch is a 32 MiB array inside the library.

Checked through the C ABI against sar_form_image (same kernels, caller-provided
workspace) on two calls in a row with different inputs, so that anything the
first call leaves in the shared scratch array would show in the second.  Kept in
a file that pytest collects last."""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

import domain_backprojection_gb300 as sar
import synth
from helpers import IMG_TOL, rel_l2

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p


def _entry():
    fn = sar.lib().sar_form_image_noalloc
    fn.argtypes = [P, P, P, P, P]
    fn.restype = ctypes.c_int
    return fn


def test_noalloc_matches_form_image_on_two_calls_in_a_row():
    noalloc = _entry()
    base = synth.make_scene(1, device="cuda")            # 256 x 8192 compressed samples = 16 MiB of scratch
    other = synth.make_scene(dataclasses.replace(synth.SCENES[1], seed=77,
                                                 fixed_target_offsets=((5, -7), (30, 12))), device="cuda")
    plan = sar.sar_plan_create(base["radar"], base["grid"], 0)
    stream = torch.cuda.current_stream()
    for scene in (base, other):
        want = sar.sar_form_image(plan, scene["raw"], scene["pos"])
        got = torch.full_like(want, float("nan"))
        st = noalloc(plan.handle, P(scene["raw"].data_ptr()), P(scene["pos"].data_ptr()), P(got.data_ptr()),
                     P(stream.cuda_stream))
        assert st == 0, sar.sar_status_string(st)
        sar.sar_plan_sync(plan)
        assert 2 <= sar.sar_plan_last_launches(plan) <= 4
        w, g = want.cpu().numpy(), got.cpu().numpy()
        assert np.all(np.isfinite(g))
        assert rel_l2(g, w) <= IMG_TOL


def test_noalloc_records_both_kernel_timings():
    """With kernel timing on, one call records one range-compression and one backprojection pair,
    like sar_form_image."""
    noalloc = _entry()
    scene = synth.make_scene(1, device="cuda")
    plan = sar.sar_plan_create(scene["radar"], scene["grid"], 0)
    sar.sar_plan_set_timing(plan, True)
    got = torch.empty(scene["grid"].ny, scene["grid"].nx, dtype=torch.complex64, device="cuda")
    st = noalloc(plan.handle, P(scene["raw"].data_ptr()), P(scene["pos"].data_ptr()), P(got.data_ptr()),
                 P(torch.cuda.current_stream().cuda_stream))
    assert st == 0, sar.sar_status_string(st)
    sar.sar_plan_sync(plan)
    times = sar.sar_plan_kernel_times(plan)
    assert times["rc_calls"] == 1 and times["bp_calls"] == 1, times
    assert times["rc_ms"] > 0 and times["bp_ms"] > 0, times


def test_noalloc_rejects_plans_beyond_its_scratch():
    noalloc = _entry()
    s = synth.make_scene(1, device="cuda")
    big = dataclasses.replace(s["radar"], n_pulses=1024, n_range=1024)    # 1024 x 8192 x 8 B = 64 MiB
    plan = sar.sar_plan_create(big, s["grid"], 0)
    raw = torch.zeros(1024, 1024, dtype=torch.complex64, device="cuda")
    pos = torch.zeros(1024, 3, dtype=torch.float64, device="cuda")
    img = torch.zeros(s["grid"].ny, s["grid"].nx, dtype=torch.complex64, device="cuda")
    assert noalloc(plan.handle, P(raw.data_ptr()), P(pos.data_ptr()), P(img.data_ptr()), None) == 2
    assert noalloc(None, P(raw.data_ptr()), P(pos.data_ptr()), P(img.data_ptr()), None) == 1
