"""Benchmark: SAR image formation (fused range compression + time-domain
backprojection) on the spotlight scene sized like the pages' example
(Na = 4096 pulses, Nr = 4096 samples, x8 range upsampling, 1024 x 1024 image
at 0.25 m, 64 point targets + clutter).

One step = range-compress every pulse, then backproject every pulse into the
image, through the C ABI (sar_range_compress + sar_backproject, the two
halves of sar_form_image), with inputs resident in HBM.  Four input sets
rotate between steps (536 MB of raw echoes, more than the 129 MB L2).  Prints
one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (the oracle is the reference arm: the pages ship
no code).  Under torchrun every rank forms its own image (independent
problems, weak scaling, no collective on the data path).
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "backprojection Gpix-pulse/s + range lines/s; % FP32 and % HBM roofline"
UNIT = "Gpix-pulse/s"
SCENE_ID = 3
FLOPS_PER_PIXEL_PULSE = 30          # range 9, index 4, interpolation 6, phase 3, complex MAC 8
PAGES_BP_GPIX_PULSE_S = 4096 * 1024 * 1024 / 0.8 / 1e9   # RTX 3080, BP only, same workload (context)


def rank_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x, world, device=None):
    """The largest of one float per rank over all ranks (the value itself for a single rank)."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, seconds):
    """Units per second of the whole job: every rank processes units_per_rank in `seconds` (the slowest
    rank's time), so the job processes world * units_per_rank in that time (weak scaling)."""
    return world * units_per_rank / seconds


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "sm_max_mhz": 2070.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


KERNEL_SOURCES = {
    # the pixel kernel's launch shape (tile shape, pulse slices) is chosen in sar_api.cu
    "bp_kernel": ["bp_kernel.cu", "sar_internal.cuh", "sar_api.cu"],
    "rc_reg_kernel": ["rc_kernel.cu", "fft_reg.cuh", "sar_internal.cuh"],
    "rc_fused_kernel": ["rc_kernel.cu", "fft_reg.cuh", "sar_internal.cuh"],
    "rc_mixed6000_kernel": ["rc_kernel.cu", "fft_reg.cuh", "sar_internal.cuh"],
    "rc_reg32_kernel": ["rc_kernel.cu", "fft_reg.cuh", "sar_internal.cuh"],
    "rc_blue32_kernel": ["rc_kernel.cu", "fft_reg.cuh", "sar_internal.cuh"],
}


def source_digest(kernel):
    """sha256 over the source files a kernel is compiled from (concatenated in a fixed order)."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "domain_backprojection_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def kernel_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's sources are unchanged since."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("source_sha256") == source_digest(kernel):
            return rec.get("dram_bytes_per_launch")
    except (OSError, ValueError, KeyError):
        pass
    return None


def time_image_step(sar, scene, dev, steps, warmup, world, n_sets):
    """The image-formation step on one scene (range compression of every pulse into polyphase
    planes, then backprojection of every pulse), timed over `steps` steps with CUDA events on the
    launching stream, the library's own events around its two main kernels, and nvidia-smi clocks
    sampled during the timed region.  n_sets input sets rotate between steps."""
    import torch

    radar, grid = scene["radar"], scene["grid"]
    na = radar.n_pulses
    plan = sar.sar_plan_create(radar, grid, dev.index)
    # compressed lines in polyphase planes, as sar_form_image keeps its workspace
    sar.sar_plan_set_rc_layout(plan, sar.SAR_RC_POLYPHASE)
    raws = [scene["raw"]] + [scene["raw"].clone() for _ in range(n_sets - 1)]
    poss = [scene["pos"]] + [scene["pos"].clone() for _ in range(n_sets - 1)]
    rc = torch.empty(na, radar.n_range * radar.upsample, dtype=torch.complex64, device=dev)
    img = torch.empty(grid.ny, grid.nx, dtype=torch.complex64, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        sar.sar_range_compress(plan, raws[i % n_sets], rc, stream=stream)
        sar.sar_backproject(plan, rc, poss[i % n_sets], 0, na, img, stream=stream)

    for i in range(warmup):
        step(i)
    sar.sar_plan_sync(plan, stream)
    # the library records CUDA events on `stream` around the two main kernels of every timed step
    sar.sar_plan_set_timing(plan, True)
    sar.sar_plan_kernel_times(plan)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    launches = 0
    with ClockSampler(dev.index) as clocks:
        t0.record(stream)
        for i in range(steps):
            step(i)
            launches += 1 + sar.sar_plan_last_launches(plan)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
    sar.sar_plan_sync(plan, stream)
    ms_total = t0.elapsed_time(t1)
    kt = sar.sar_plan_kernel_times(plan)
    sar.sar_plan_set_timing(plan, False)
    assert kt["rc_calls"] == steps and kt["bp_calls"] == steps, kt
    ms_total = max_over_ranks(ms_total, world, dev)

    # end to end through the host-buffer entry point: H2D of raw + positions, both kernels, D2H of the image
    raw_h = scene["raw"].cpu().pin_memory()
    pos_h = scene["pos"].cpu().pin_memory()
    img_h = torch.empty(grid.ny, grid.nx, dtype=torch.complex64, pin_memory=True)
    for _ in range(2):
        sar.sar_form_image_host(plan, raw_h, pos_h, img_h)
    e2e_steps = max(3, min(steps, 10))
    torch.cuda.synchronize(dev)
    w0 = time.perf_counter()
    for _ in range(e2e_steps):
        sar.sar_form_image_host(plan, raw_h, pos_h, img_h)
    e2e_s = (time.perf_counter() - w0) / e2e_steps
    e2e_s = max_over_ranks(e2e_s, world, dev)
    res = {"ms_step": ms_total / steps, "rc_ms": kt["rc_ms"] / kt["rc_calls"], "bp_ms": kt["bp_ms"] / kt["bp_calls"],
           "launches": launches, "clocks": clocks.summary(), "e2e_s": e2e_s,
           "h2d": raw_h.numel() * 8 + pos_h.numel() * 8, "d2h": img_h.numel() * 8}
    del plan, raws, poss, rc, img, raw_h, pos_h, img_h
    torch.cuda.empty_cache()
    return res


def headline_record(t, scene, cid, args, world, dev, peaks, peak_src, fp32_sm_mhz=None):
    """The bench line's keys for one scene from its step timing `t` (time_image_step)."""
    import torch
    import synth

    cfg = synth.SCENES[cid]
    radar, grid = scene["radar"], scene["grid"]
    props = torch.cuda.get_device_properties(dev)
    clk = t["clocks"]
    sm_mhz = clk["sm_mhz"] if clk else (fp32_sm_mhz or float(peaks.get("clocks_under_load", {}).get("sm_mhz_median", 1455.0)))
    fp32_peak = props.multi_processor_count * 128 * 2 * sm_mhz * 1e6 / 1e12      # TFLOP/s at the sampled clock
    fp32_peak_max = props.multi_processor_count * 128 * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12
    pp = cfg.pixel_pulses
    bp_tflops = FLOPS_PER_PIXEL_PULSE * pp / (t["bp_ms"] * 1e-3) / 1e12
    n_range, U = radar.n_range, radar.upsample
    rc_bytes = cfg.n_pulses * 8 * n_range * (1 + U)
    rc_gbs = rc_bytes / (t["rc_ms"] * 1e-3) / 1e9
    rc_name = rc_kernel_name(n_range, U)
    value = whole_job_rate(pp, world, t["ms_step"] * 1e-3) / 1e9
    content = {3: "64 targets + 16384 clutter scatterers", 4: "curved track (0.5 m sinusoidal errors), 256 targets + "
               "65536 clutter scatterers"}.get(cid, "")
    l2 = ("4 rotating input sets (536 MB raw) > 129 MB L2; 1.07 GB compressed lines per step" if cid == 3 else
          "inputs 1.07 GB raw > 129 MB L2; 8.6 GB compressed lines per step")
    return {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t["ms_step"], 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": round(value / PAGES_BP_GPIX_PULSE_S, 2), "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{cfg.name}: Na={cfg.n_pulses} Nr={n_range} U={U} image {grid.nx}x{grid.ny}"
                               f" @ {grid.dx} m, {content}",
                   "pixel_pulses_per_step": pp, "range_lines_per_step": cfg.n_pulses, "l2": l2,
                   "step": "sar_range_compress + sar_backproject with polyphase-plane compressed lines "
                           "(the kernels sar_form_image runs)"},
        "rc_lines_per_s": round(whole_job_rate(cfg.n_pulses, world, t["rc_ms"] * 1e-3), 1),
        "bp_gpix_pulse_per_s": round(whole_job_rate(pp, world, t["bp_ms"] * 1e-3) / 1e9, 3),
        "kernel_ms": {rc_name: round(t["rc_ms"], 4), "bp_kernel": round(t["bp_ms"], 4)},
        "roofline": {"kernel": "bp_kernel", "bound": "alu", "achieved": round(bp_tflops, 3),
                     "peak": round(fp32_peak, 3), "unit": "TFLOP/s", "frac": round(bp_tflops / fp32_peak, 4),
                     "traffic": kernel_traffic("bp_kernel") if cid == SCENE_ID else None,
                     "peak_basis": f"{props.multi_processor_count} SMs x 128 FP32 lanes x 2 x {sm_mhz:.0f} MHz "
                                   f"(median SM clock sampled during the timed region)",
                     "frac_of_max_clock_peak": round(bp_tflops / fp32_peak_max, 4),
                     "flops_per_pixel_pulse": FLOPS_PER_PIXEL_PULSE},
        "roofline_rc": {"kernel": rc_name, "bound": "hbm", "achieved": round(rc_gbs, 1),
                        "peak": peaks.get("hbm_gbs"), "unit": "GB/s",
                        "frac": round(rc_gbs / float(peaks.get("hbm_gbs", 6800.0)), 4),
                        "traffic": kernel_traffic(rc_name.split("<")[0]) if cid == SCENE_ID else None,
                        "peak_source": peak_src, "algorithmic_bytes_per_line": 8 * n_range * (1 + U),
                        "context_tflops": round(rc_flops_per_line(n_range, U) * cfg.n_pulses / (t["rc_ms"] * 1e-3) / 1e12, 3)},
        "clocks": clk,
        "e2e": {"value": round(whole_job_rate(pp, world, t["e2e_s"]) / 1e9, 3), "unit": UNIT,
                "h2d_bytes_per_step": t["h2d"], "d2h_bytes_per_step": t["d2h"], "api": "sar_form_image_host"},
        "gpu_launches": t["launches"],
    }


def write_traffic_record(csv_path, kernel, launch, workload, command):
    """profiles/<kernel>_traffic.json from an ncu --csv log of one launch of `kernel` with
    dram__bytes_read.sum and dram__bytes_write.sum, tied to the sha256 of the kernel's sources."""
    import csv
    rows = [r for r in csv.reader(open(csv_path)) if r and not r[0].startswith("==")]
    hdr = rows[0]
    ki, mn, mv, mu = (hdr.index(k) for k in ("Kernel Name", "Metric Name", "Metric Value", "Metric Unit"))
    vals = {}
    for r in rows[1:]:
        if kernel in r[ki]:
            scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}.get(r[mu], 1)
            vals[r[mn]] = int(round(float(r[mv].replace(",", "")) * scale))
    rd, wr = vals["dram__bytes_read.sum"], vals["dram__bytes_write.sum"]
    rec = {"kernel": kernel, "launch": launch, "workload": workload, "dram_bytes_read": rd,
           "dram_bytes_write": wr, "dram_bytes_per_launch": rd + wr, "command": command,
           "source_sha256": source_digest(kernel), "source_files": KERNEL_SOURCES[kernel]}
    with open(os.path.join(ROOT, "profiles", f"{kernel}_traffic.json"), "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    return rec


def run_ours(args, rank, world, local_rank):
    import torch
    import domain_backprojection_gb300 as sar
    import synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks, peak_src = measured_peaks()
    scene = synth.make_scene(SCENE_ID, device=dev)
    t = time_image_step(sar, scene, dev, args.steps, args.warmup, world, n_sets=4)
    out = headline_record(t, scene, SCENE_ID, args, world, dev, peaks, peak_src)
    if rank != 0:
        return None
    clk = out["clocks"]
    props = torch.cuda.get_device_properties(dev)
    fp32_peak = out["roofline"]["peak"]
    if not args.no_rda:
        out["range_doppler"] = rda_bench(scene, dev, peaks, reps=max(5, min(args.steps, 20)))
    if not args.no_bp_variants:
        out["bp_variants"] = bp_variants(scene, dev, reps=max(5, min(args.steps, 20)))
    if not args.no_cpu_baseline:
        # the oracle, as it stands, on every host core: the whole step (range compression of every
        # pulse, backprojection of every pixel); and on one core, on a stated sample
        out["cpu_baseline"] = oracle_baseline(scene, SCENE_ID)
        out["cpu_baseline_1thread"] = oracle_baseline(scene, SCENE_ID, threads=1, full=args.cpu_full)
    del scene
    torch.cuda.empty_cache()
    if not args.no_rc_sweep:
        out["rc_sweep"] = rc_sweep(dev, peaks, reps=max(10, min(args.steps, 50)), cpu=not args.no_cpu_baseline,
                                   cpu_full=args.cpu_full)
    if not args.no_scenes:
        out["scenes"] = other_scenes(dev, peaks, fp32_peak, reps=max(5, min(args.steps, 20)),
                                     cpu=not args.no_cpu_baseline, cpu_full=args.cpu_full)
    if not args.no_large:
        # the largest configuration, in the same form as the headline record
        big = synth.make_scene(4, device=dev)
        tb = time_image_step(sar, big, dev, max(3, min(args.steps, 20)), max(3, min(args.warmup, 5)), 1, n_sets=1)
        rec = headline_record(tb, big, 4, args, 1, dev, peaks, peak_src, fp32_sm_mhz=clk["sm_mhz"] if clk else None)
        rec["steps"], rec["warmup"] = max(3, min(args.steps, 20)), max(3, min(args.warmup, 5))
        if not args.no_cpu_baseline:
            rec["cpu_baseline"] = oracle_baseline(big, 4)
            rec["cpu_baseline_1thread"] = oracle_baseline(big, 4, threads=1, full=args.cpu_full)
        out["large_scene"] = rec
        del big
        torch.cuda.empty_cache()
    return out


def rc_flops_per_line(nr, upsample=1):
    """Conventional flop count of one compressed line, reported as context beside the HBM roofline:
    5 N log2 N per N-point transform for the forward transform and the U inverse ones, plus 6 N for
    the matched-filter product."""
    return 5.0 * nr * math.log2(nr) * (1 + upsample) + 6.0 * nr


def rc_kernel_name(nr, upsample=1):
    """The range-compression kernel the library launches for Nr-sample lines: the register-resident
    radix-16 kernel for powers of two from 512 to 8192 (the 32-element kernel for 8192 without
    upsampling), the register-resident radix-10/6 kernel for 6000, the shared-memory mixed-radix one for other even 2^a 3^b 5^c lengths, Bluestein otherwise
    (register-resident without upsampling, in shared memory with it)."""
    if nr == 8192 and upsample == 1:
        return "rc_reg32_kernel"
    if nr >= 512 and nr <= 8192 and nr & (nr - 1) == 0:
        return f"rc_reg_kernel<{nr}>"
    if nr == 6000:
        return "rc_mixed6000_kernel"
    m = nr
    for p in (2, 3, 5):
        while m % p == 0:
            m //= p
    if m == 1 and nr % 2 == 0:
        return "rc_fused_kernel"
    bm = 512
    while bm < 2 * nr - 1:
        bm *= 2
    if bm == 16384:
        return "rc_blue32_kernel"
    return f"rc_blue_reg_kernel<{bm}>" if upsample == 1 else "rc_bluestein_kernel"


def profile_case(case="spotlight"):
    import torch
    import domain_backprojection_gb300 as sar
    import synth

    if case.startswith("sweep"):
        # sweepNR: 4096 lines of NR samples, U = 1; sweepNRuU: 2048 lines with upsampling by U into
        # polyphase planes (the large scene's line kernel on a case small enough for a full capture)
        spec = case[len("sweep"):]
        nr, U = (int(spec.split("u")[0]), int(spec.split("u")[1])) if "u" in spec else (int(spec), 1)
        lines = 4096 if U == 1 else 2048
        sc = synth.make_rc_sweep(nr, n_lines=lines, device="cuda")
        import dataclasses
        radar = dataclasses.replace(sc["radar"], upsample=U)
        plan = sar.sar_plan_create(radar, None, 0)
        if U > 1:
            sar.sar_plan_set_rc_layout(plan, sar.SAR_RC_POLYPHASE)
        out = torch.empty(lines, nr * U, dtype=torch.complex64, device="cuda")
        for _ in range(3):
            sar.sar_range_compress(plan, sc["raw"], out)
        sar.sar_plan_sync(plan)
        print(json.dumps({"profile_case": "ok", "workload": f"range-only sweep, {lines} lines of {nr} samples, U={U}"}))
        return
    if case == "rda":
        import dataclasses
        scene = synth.make_scene(SCENE_ID, device="cuda")
        cfg = scene["config"]
        plan = sar.sar_plan_create(dataclasses.replace(scene["radar"], upsample=1), None, 0)
        sar.sar_plan_set_range_doppler(plan, cfg.velocity / cfg.prf)
        for _ in range(2):
            img = sar.sar_range_doppler(plan, scene["raw"])
        sar.sar_plan_sync(plan)
        print(json.dumps({"profile_case": "ok", "workload": "range-Doppler, 4096 x 4096, spotlight scene raw echoes"}))
        return
    scene_ids = {"spotlight": SCENE_ID, "scene1": 1, "scene2": 2, "scene4": 4}
    if case not in scene_ids:
        raise SystemExit(f"unknown profile case {case!r}")
    scene = synth.make_scene(scene_ids[case], device="cuda")
    radar = scene["radar"]
    plan = sar.sar_plan_create(radar, scene["grid"], 0)
    sar.sar_plan_set_rc_layout(plan, sar.SAR_RC_POLYPHASE)
    rc = torch.empty(radar.n_pulses, radar.n_range * radar.upsample, dtype=torch.complex64, device="cuda")
    for _ in range(2):
        sar.sar_range_compress(plan, scene["raw"], rc)
        sar.sar_backproject(plan, rc, scene["pos"])
    sar.sar_plan_sync(plan)
    g = scene["grid"]
    print(json.dumps({"profile_case": "ok", "workload": f"{case}: Na={radar.n_pulses} Nr={radar.n_range} "
                                                        f"U={radar.upsample}, {g.nx}x{g.ny} image"}))


def bp_variants(scene, dev, reps=10):
    """The backprojection variants on the same spotlight scene (polyphase-plane lines, same step as the
    headline): pixel-kernel time and rate for compensated sums, float16 staging and 8-tap sinc
    interpolation; and the step (range compression + backprojection) with x2 instead of x8 upsampled
    lines and sinc interpolation."""
    import dataclasses
    import torch
    import domain_backprojection_gb300 as sar

    radar, grid = scene["radar"], scene["grid"]
    pp = radar.n_pulses * grid.nx * grid.ny
    setters = {
        "compensated": lambda p: sar.sar_plan_set_accumulation(p, sar.SAR_ACCUM_COMPENSATED),
        "fp16_stage": lambda p: sar.sar_plan_set_stage_precision(p, sar.SAR_STAGE_FP16),
        "sinc8": lambda p: sar.sar_plan_set_interpolation(p, sar.SAR_INTERP_SINC8),
        "sinc8_u2": lambda p: sar.sar_plan_set_interpolation(p, sar.SAR_INTERP_SINC8),
    }
    res = {}
    for name, setter in setters.items():
        r = dataclasses.replace(radar, upsample=2) if name.endswith("_u2") else radar
        plan = sar.sar_plan_create(r, grid, dev.index)
        sar.sar_plan_set_rc_layout(plan, sar.SAR_RC_POLYPHASE)
        setter(plan)
        rc = sar.sar_range_compress(plan, scene["raw"])
        img = sar.sar_backproject(plan, rc, scene["pos"])
        sar.sar_plan_sync(plan)
        sar.sar_plan_set_timing(plan, True)
        sar.sar_plan_kernel_times(plan)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            sar.sar_range_compress(plan, scene["raw"], rc)
            sar.sar_backproject(plan, rc, scene["pos"], image=img)
        e1.record()
        torch.cuda.synchronize(dev)
        sar.sar_plan_sync(plan)
        kt = sar.sar_plan_kernel_times(plan)
        bp_ms = kt["bp_ms"] / kt["bp_calls"]
        step_ms = e0.elapsed_time(e1) / reps
        res[name] = {"upsample": r.upsample, "bp_kernel_ms": round(bp_ms, 4),
                     "bp_gpix_pulse_per_s": round(pp / (bp_ms * 1e-3) / 1e9, 1),
                     "rc_kernel_ms": round(kt["rc_ms"] / kt["rc_calls"], 4), "step_ms": round(step_ms, 4),
                     "step_gpix_pulse_per_s": round(pp / (step_ms * 1e-3) / 1e9, 1)}
        del plan, rc, img
    return res


def rda_bench(scene, dev, peaks, reps=10):
    """Range-Doppler image formation (sar_range_doppler) of the same scene's raw echoes at native range
    sampling: Na = 4096 pulses x Nr = 4096 range bins -> a 4096 x 4096 image.  Time per image, and the
    algorithmic DRAM bytes (8 passes over the 134 MB complex plane: compression, transpose, azimuth
    transform, migration correction + filter + inverse transform, each one read and one write) over it."""
    import dataclasses
    import torch
    import domain_backprojection_gb300 as sar

    cfg = scene["config"]
    radar = dataclasses.replace(scene["radar"], upsample=1)
    plan = sar.sar_plan_create(radar, None, dev.index)
    sar.sar_plan_set_range_doppler(plan, cfg.velocity / cfg.prf)
    img = sar.sar_range_doppler(plan, scene["raw"])
    ws = torch.empty(sar.sar_range_doppler_workspace_size(plan), dtype=torch.uint8, device=dev)
    raws = [scene["raw"]] + [scene["raw"].clone() for _ in range(3)]
    for i in range(3):
        sar.sar_range_doppler(plan, raws[i % 4], img, ws)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(reps):
        sar.sar_range_doppler(plan, raws[i % 4], img, ws)
    e1.record()
    torch.cuda.synchronize(dev)
    sar.sar_plan_sync(plan)
    ms = e0.elapsed_time(e1) / reps
    plane = radar.n_pulses * radar.n_range * 8
    gbs = 8 * plane / (ms * 1e-3) / 1e9
    del plan, img, ws, raws
    return {"workload": f"range-Doppler: Na={radar.n_pulses} x Nr={radar.n_range} (spotlight scene raw echoes, "
                        f"straight track, U=1) -> {radar.n_range}x{radar.n_pulses} image",
            "ms": round(ms, 4), "images_per_s": round(1e3 / ms, 1),
            "range_lines_per_s": round(radar.n_pulses / (ms * 1e-3), 1),
            "algorithmic_gbs": round(gbs, 1), "frac_hbm": round(gbs / float(peaks.get("hbm_gbs", 6800.0)), 4),
            "launches": 4, "pages_context": "Apple M1, 4096x4096 range-Doppler: 370 ms (other hardware)"}


def other_scenes(dev, peaks, fp32_peak, reps=20, cpu=True, cpu_full=False):
    """The tiny (256 x 1024, 128^2) and small (1024 x 2048, 512^2) scenes, each formed as the headline
    step forms its image (range compression into polyphase planes, then backprojection).  Per scene:
    step time, pixel-pulse and line rates, the backprojection kernel's fraction of the FP32 peak, the
    range compression's fraction of the measured HBM bandwidth, the same step replayed from a CUDA
    graph, and the oracle timed on the whole scene.  Both scenes' inputs fit in L2, so their rates
    are L2-warm.  (The large curved-track
    scene has a record of its own, in the headline's form.)"""
    import torch
    import domain_backprojection_gb300 as sar
    import synth

    res = {}
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    for cid in (1, 2):
        cfg = synth.SCENES[cid]
        scene = synth.make_scene(cid, device=dev)
        radar, grid = scene["radar"], scene["grid"]
        plan = sar.sar_plan_create(radar, grid, dev.index)
        sar.sar_plan_set_rc_layout(plan, sar.SAR_RC_POLYPHASE)
        rc = torch.empty(cfg.n_pulses, radar.n_range * radar.upsample, dtype=torch.complex64, device=dev)
        img = torch.empty(grid.ny, grid.nx, dtype=torch.complex64, device=dev)
        for _ in range(3):
            sar.sar_range_compress(plan, scene["raw"], rc)
            sar.sar_backproject(plan, rc, scene["pos"], image=img)
        sar.sar_plan_sync(plan)
        sar.sar_plan_set_timing(plan, True)
        sar.sar_plan_kernel_times(plan)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            sar.sar_range_compress(plan, scene["raw"], rc)
            sar.sar_backproject(plan, rc, scene["pos"], image=img)
        e1.record()
        torch.cuda.synchronize(dev)
        sar.sar_plan_sync(plan)
        kt = sar.sar_plan_kernel_times(plan)
        sar.sar_plan_set_timing(plan, False)
        step_ms = e0.elapsed_time(e1) / reps
        bp_ms = kt["bp_ms"] / kt["bp_calls"]
        rc_ms = kt["rc_ms"] / kt["rc_calls"]
        # the same step captured once in a CUDA graph and replayed: the launches without their
        # host-side gaps (these scenes are small enough for the gaps to show)
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                sar.sar_range_compress(plan, scene["raw"], rc, stream=cap)
                sar.sar_backproject(plan, rc, scene["pos"], image=img, stream=cap)
        torch.cuda.current_stream(dev).wait_stream(cap)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize(dev)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record()
        for _ in range(reps):
            graph.replay()
        g1.record()
        torch.cuda.synchronize(dev)
        sar.sar_plan_sync(plan)
        graph_ms = g0.elapsed_time(g1) / reps
        del graph
        pp = cfg.pixel_pulses
        rc_gbs = cfg.n_pulses * 8 * radar.n_range * (1 + radar.upsample) / (rc_ms * 1e-3) / 1e9
        bp_tflops = FLOPS_PER_PIXEL_PULSE * pp / (bp_ms * 1e-3) / 1e12
        res[str(cid)] = {
            "workload": f"{cfg.name}: Na={cfg.n_pulses} Nr={radar.n_range} U={radar.upsample} image "
                        f"{grid.nx}x{grid.ny} @ {grid.dx} m",
            "pixel_pulses": pp, "step_ms": round(step_ms, 4),
            "step_gpix_pulse_per_s": round(pp / (step_ms * 1e-3) / 1e9, 1),
            "step_ms_graph": round(graph_ms, 4),
            "step_graph_gpix_pulse_per_s": round(pp / (graph_ms * 1e-3) / 1e9, 1),
            "bp_kernel_ms": round(bp_ms, 4), "bp_gpix_pulse_per_s": round(pp / (bp_ms * 1e-3) / 1e9, 1),
            "bp_frac_fp32": round(bp_tflops / fp32_peak, 4),
            "rc_kernel": rc_kernel_name(radar.n_range, radar.upsample), "rc_kernel_ms": round(rc_ms, 4),
            "rc_lines_per_s": round(cfg.n_pulses / (rc_ms * 1e-3), 1), "rc_frac_hbm": round(rc_gbs / hbm, 4),
            "launches_per_step": 1 + sar.sar_plan_last_launches(plan), "l2": "inputs fit in L2"}
        if cpu:
            res[str(cid)]["cpu_baseline"] = oracle_baseline(scene, cid)
            res[str(cid)]["cpu_baseline_1thread"] = oracle_baseline(scene, cid, threads=1, full=cpu_full)
        del plan, rc, img, scene
        torch.cuda.empty_cache()
    return res


def rc_sweep(dev, peaks, reps=20, n_sets=4, cpu=True, cpu_full=False):
    """Range compression alone on the range-only workload: 4096 lines of Nr in {4096, 8192, 6000}
    samples, U = 1, four rotating input sets; lines/s, the fraction of the measured HBM bandwidth, and
    the oracle's range compression of all 4096 lines (every host core; one core on a sample)."""
    import torch
    import domain_backprojection_gb300 as sar
    import synth

    res = {}
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    # the range-only lengths, then two lengths with a prime factor that take the Bluestein kernels
    # (2 x 23 x 89: M = 8192; 2 x 3^2 x 5 x 7 x 13: M = 16384)
    for nr in tuple(synth.RC_SWEEP_NR) + (4094, 8190):
        scene = synth.make_rc_sweep(nr, n_lines=4096, device=dev)
        plan = sar.sar_plan_create(scene["radar"], None, dev.index)
        raws = [scene["raw"]] + [scene["raw"].clone() for _ in range(n_sets - 1)]
        outs = [torch.empty_like(r) for r in raws]
        for i in range(3):
            sar.sar_range_compress(plan, raws[i % n_sets], outs[i % n_sets])
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(reps):
            sar.sar_range_compress(plan, raws[i % n_sets], outs[i % n_sets])
        e1.record()
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / reps
        gbs = 4096 * 16 * nr / (ms * 1e-3) / 1e9
        res[str(nr)] = {"kernel": rc_kernel_name(nr), "ms": round(ms, 4), "lines_per_s": round(4096 / (ms * 1e-3), 1),
                        "gbs": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4)}
        if cpu and nr in synth.RC_SWEEP_NR:
            res[str(nr)]["cpu_baseline"] = oracle_rc_baseline(scene)
            res[str(nr)]["cpu_baseline_1thread"] = oracle_rc_baseline(scene, threads=1, full=cpu_full)
        del plan, raws, outs, scene
    return res


def cpu_model():
    """The host CPU's model name (lscpu), for the oracle timing records."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine() or "unknown"


def _threads(threads):
    return threads or os.cpu_count()


def oracle_time(radar, grid, raw, pos, threads, lines, pixels=None, chunk=1024):
    """Seconds the oracle takes to range-compress the first `lines` pulses and, with a grid, to
    backproject them into the listed flat pixel indices (every pixel when None), chunk by chunk so
    that its float64 lines stay within a few GB of host memory.  Copies from the device are not
    timed.  Returns (rc_s, bp_s)."""
    import numpy as np
    import oracle

    oracle.lib()
    rc_s = bp_s = 0.0
    out = None
    if grid is not None:
        out = np.zeros(grid.nx * grid.ny if pixels is None else pixels.size, dtype=np.complex128)
    for n0 in range(0, lines, chunk):
        n1 = min(lines, n0 + chunk)
        r = raw[n0:n1].cpu().numpy()
        t = time.perf_counter()
        rc = oracle.range_compress(radar, r, threads=threads)
        rc_s += time.perf_counter() - t
        if grid is not None:
            p = pos[n0:n1].cpu().numpy()
            t = time.perf_counter()
            oracle.backproject(radar, grid, rc, p, pixels=pixels, out=out, accumulate=True, threads=threads)
            bp_s += time.perf_counter() - t
        del rc
    return rc_s, bp_s


def central_pixels(grid, side):
    """Flat indices of the central side x side pixels of the grid."""
    import numpy as np
    side = min(side, grid.nx, grid.ny)
    y0, x0 = (grid.ny - side) // 2, (grid.nx - side) // 2
    yy, xx = np.mgrid[y0:y0 + side, x0:x0 + side]
    return (yy * grid.nx + xx).ravel().astype(np.int64)


def oracle_baseline(scene, cid, threads=None, full=False):
    """The fp64 oracle, as it stands, timed on the host cores on one imaging scene.  With every core
    (threads None): the whole step of the tiny, small and spotlight scenes (range compression of
    every pulse, backprojection of every pixel); on the large curved-track scene the range
    compression of every pulse and the backprojection of the central 256 x 256 pixels over every
    pulse, extrapolated to the 2048 x 2048 image (x64).  With one thread: the tiny and small scenes
    whole; the spotlight and large scenes on the first 256 pulses and the central 256 x 256 (128 x
    128) pixels, scaled to the whole step (or, with `full`, as with every core)."""
    radar, grid = scene["radar"], scene["grid"]
    na = radar.n_pulses
    n = _threads(threads)
    lines, side = na, None
    if cid == 4:
        side = 256
    if threads == 1 and not full:
        if cid == 3:
            lines, side = 256, 256
        elif cid == 4:
            lines, side = 256, 128
    pix = None if side is None else central_pixels(grid, side)
    rc_s, bp_s = oracle_time(radar, grid, scene["raw"], scene["pos"], n, lines, pix)
    npix = grid.nx * grid.ny if pix is None else pix.size
    full_s = (rc_s + bp_s * (grid.nx * grid.ny) / npix) * na / lines
    pp = na * grid.nx * grid.ny
    measured = lines == na and npix == grid.nx * grid.ny
    sample = (f"whole step: range compression of {na} pulses ({rc_s:.2f} s) and backprojection of the "
              f"{grid.nx}x{grid.ny} image ({bp_s:.2f} s)" if measured else
              f"range compression of {lines} of {na} pulses ({rc_s:.2f} s) and their backprojection into the "
              f"central {int(round(npix ** 0.5))}x{int(round(npix ** 0.5))} pixels ({bp_s:.2f} s), scaled to "
              f"{na} pulses and the {grid.nx}x{grid.ny} image")
    return {"value": round(pp / full_s / 1e9, 5), "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": sample + f"; fp64, {n} thread{'s' if n > 1 else ''}", "cpu": cpu_model(),
            "rc_s": float(f"{rc_s:.4g}"), "bp_s": float(f"{bp_s:.4g}"), "full_step_s": float(f"{full_s:.4g}"),
            "extrapolated": not measured}


def oracle_rc_baseline(scene, threads=None, full=False):
    """The oracle's range compression of the range-only workload's 4096 lines on the host cores
    (every core), or of its first 512 lines scaled to 4096 on one core (all 4096 with `full`)."""
    radar = scene["radar"]
    na = scene["raw"].shape[0]
    n = _threads(threads)
    lines = na if (threads is None or full) else min(512, na)
    rc_s, _ = oracle_time(radar, None, scene["raw"], None, n, lines)
    full_s = rc_s * na / lines
    return {"value": round(na / full_s, 1), "unit": "lines/s", "cores": n, "kind": "oracle",
            "sample": (f"range compression of {lines} of {na} lines of {radar.n_range} samples ({rc_s:.2f} s)"
                       + ("" if lines == na else f", scaled to {na}") + f"; fp64, {n} thread{'s' if n > 1 else ''}"),
            "cpu": cpu_model(), "full_s": round(full_s, 3), "extrapolated": lines != na}


def reference_sample(scene, threads, budget_s):
    """One step of the reference arm: the oracle on the first pulses of the spotlight scene, their
    range compression and backprojection of a central pixel patch that grows until it takes about
    half the budget, scaled to every pulse and every pixel."""
    radar, grid = scene["radar"], scene["grid"]
    na = radar.n_pulses
    lines = min(512, na)
    side = 16
    while True:
        pix = central_pixels(grid, side)
        rc_s, bp_s = oracle_time(radar, grid, scene["raw"], scene["pos"], threads, lines, pix)
        if bp_s > 0.5 * budget_s or side >= min(grid.nx, grid.ny):
            break
        side *= 2
    full_s = (rc_s + bp_s * grid.nx * grid.ny / pix.size) * na / lines
    pp = na * grid.nx * grid.ny
    return {"value": round(pp / full_s / 1e9, 5), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{lines} of {na} pulses: their range compression ({rc_s:.2f} s) and backprojection of a "
                      f"{side}x{side} pixel patch ({bp_s:.2f} s), scaled to {na} pulses and the "
                      f"{grid.nx}x{grid.ny} image; fp64, {threads} threads",
            "cpu": cpu_model(), "est_full_step_s": round(full_s, 2)}


def run_reference(args, rank, world, local_rank):
    import synth
    import torch

    if rank != 0:
        return None
    scene = synth.make_scene(SCENE_ID, device="cuda" if torch.cuda.is_available() else "cpu")
    per_step = max(1.0, min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup)))
    threads = os.cpu_count()
    for _ in range(args.warmup):
        reference_sample(scene, threads, per_step)
    runs = [reference_sample(scene, threads, per_step) for _ in range(args.steps)]
    vals = [r["value"] for r in runs]
    cb = dict(runs[-1])
    v = statistics.median(vals)
    cfg = synth.SCENES[SCENE_ID]
    ms = cfg.pixel_pulses / (v * 1e9) * 1e3
    cb["value"] = round(v, 5)
    return {"impl": "reference", "metric": METRIC, "value": round(v, 5), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"spotlight-3deg: Na={cfg.n_pulses} Nr={cfg.n_range} U={cfg.upsample} image "
                                   f"{cfg.nx}x{cfg.ny} @ {cfg.pixel} m (bounded sample per step, scaled)"},
            "cpu_baseline": cb,
            "e2e": {"value": round(v, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rc-sweep", action="store_true")
    ap.add_argument("--no-bp-variants", action="store_true")
    ap.add_argument("--no-rda", action="store_true")
    ap.add_argument("--no-scenes", action="store_true")
    ap.add_argument("--no-large", action="store_true", help="skip the large curved-track scene's record")
    ap.add_argument("--cpu-full", action="store_true",
                    help="time the oracle on one core over the whole spotlight step, all of the large scene's pulses "
                         "and all 4096 sweep lines too (several minutes), instead of the stated samples")
    ap.add_argument("--profile-case", nargs="?", const="spotlight", default=None,
                    help="run a short untimed case for profiler captures and exit: 'spotlight' (default) forms two "
                         "images of the spotlight scene (RC then BP, polyphase planes), 'scene1', 'scene2' and 'scene4' "
                         "the same on the tiny, small and large curved-track scenes; 'sweepNR' (e.g. NR = 4096, 8192, "
                         "6000, 4094) range-compresses the 4096 lines of the range-only workload three times; 'rda' forms "
                         "two range-Doppler images of the spotlight scene's raw echoes")
    ap.add_argument("--write-traffic", nargs=5, metavar=("CSV", "KERNEL", "LAUNCH", "WORKLOAD", "COMMAND"),
                    help="write profiles/KERNEL_traffic.json from an ncu --csv log of one launch (DRAM bytes read "
                         "and written) and exit")
    args = ap.parse_args()
    rank, world, local_rank = rank_env()
    if args.write_traffic:
        print(json.dumps(write_traffic_record(*args.write_traffic)))
        return
    if args.profile_case:
        profile_case(args.profile_case)
        return
    if world > 1 and args.impl == "ours":
        import torch
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out = (run_reference if args.impl == "reference" else run_ours)(args, rank, world, local_rank)
    if out is not None:
        print(json.dumps(out), flush=True)
    if world > 1 and args.impl == "ours":
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
