"""bench.py's host-side bookkeeping, on CPU: the kernel it names for each line length, the
traffic records it reports (only while the kernel's sources are unchanged), and the clock
summary of an nvidia-smi sample stream."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("nr,u,name", [
    (512, 8, "rc_reg_kernel<512>"), (4096, 8, "rc_reg_kernel<4096>"), (8192, 1, "rc_reg32_kernel"), (8192, 8, "rc_reg_kernel<8192>"),
    (6000, 1, "rc_mixed6000_kernel"), (3000, 1, "rc_fused_kernel"), (1200, 8, "rc_fused_kernel"),
    (4094, 1, "rc_blue_reg_kernel<8192>"), (1009, 1, "rc_blue_reg_kernel<2048>"), (257, 1, "rc_blue_reg_kernel<1024>"),
    (100, 1, "rc_fused_kernel"), (17, 1, "rc_blue_reg_kernel<512>"), (4095, 4, "rc_bluestein_kernel"),
    (5003, 1, "rc_blue32_kernel"), (8190, 8, "rc_blue32_kernel"),
])
def test_rc_kernel_name(nr, u, name):
    # powers of two 512..8192 -> register kernel (8192 without upsampling: the 32-element one);
    # 6000 -> its own kernel; other even 2^a 3^b 5^c ->
    # the mixed-radix shared-memory kernel; anything else -> Bluestein with M >= 2 Nr - 1 (at least 512)
    assert bench.rc_kernel_name(nr, u) == name


def test_traffic_record_follows_the_sources(tmp_path, monkeypatch):
    # every committed record names its kernel, carries read + write = per-launch bytes, and is
    # reported only while the sha256 of the kernel's sources matches
    for kernel in ("bp_kernel", "rc_reg_kernel", "rc_mixed6000_kernel", "rc_reg32_kernel"):
        with open(os.path.join(ROOT, "profiles", f"{kernel}_traffic.json")) as f:
            rec = json.load(f)
        assert rec["kernel"] == kernel
        assert rec["dram_bytes_read"] + rec["dram_bytes_write"] == rec["dram_bytes_per_launch"]
        assert rec["source_files"] == bench.KERNEL_SOURCES[kernel]
    # a copy of the tree with one changed byte in a source file: the record no longer applies
    csrc = tmp_path / "domain_backprojection_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = os.path.join(ROOT, "domain_backprojection_gb300", "csrc")
    for name in bench.KERNEL_SOURCES["bp_kernel"]:
        with open(os.path.join(src, name), "rb") as f:
            (csrc / name).write_bytes(f.read())
    rec = {"kernel": "bp_kernel", "dram_bytes_per_launch": 123, "source_files": bench.KERNEL_SOURCES["bp_kernel"]}
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec["source_sha256"] = bench.source_digest("bp_kernel")
    (tmp_path / "profiles" / "bp_kernel_traffic.json").write_text(json.dumps(rec))
    assert bench.kernel_traffic("bp_kernel") == 123
    (csrc / "bp_kernel.cu").write_bytes((csrc / "bp_kernel.cu").read_bytes() + b"\n")
    assert bench.kernel_traffic("bp_kernel") is None
    assert bench.kernel_traffic("rc_fused_kernel") is None          # no record at all


def test_whole_job_rate_is_weak_scaling():
    assert bench.whole_job_rate(1000.0, 1, 2.0) == 500.0
    assert bench.whole_job_rate(1000.0, 4, 2.0) == 2000.0
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_clock_summary_reads_reasons():
    # the sampler's summary: median SM clock under load and the throttle reasons seen active
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.lines = [                       # --format=csv,noheader,nounits
        "0, 2070, 2070, 900.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.00, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1200.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbled line",
    ]
    out = s.summary()
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0 and out["samples"] == 3
    assert out["reasons"] == ["sw_power_cap"]


def test_rc_context_flops():
    # 5 N log2 N per transform, (1 + U) transforms, plus the 6 N flops of the filter product
    assert bench.rc_flops_per_line(4096, 8) == 5 * 4096 * 12 * 9 + 6 * 4096
    assert bench.rc_flops_per_line(1024, 1) == 5 * 1024 * 10 * 2 + 6 * 1024


def test_oracle_timing_records_on_a_small_case():
    # the CPU-baseline records: whole-step timing when nothing is sampled, scaled sampling otherwise,
    # and the range-only record in lines/s; every record names its cores, CPU model and sample
    import dataclasses
    import synth
    cfg = dataclasses.replace(synth.SCENES[1], n_pulses=32, nx=16, ny=16)
    scene = synth.make_scene(cfg, device="cpu")
    whole = bench.oracle_baseline(scene, 1, threads=1)
    assert whole["kind"] == "oracle" and whole["cores"] == 1 and not whole["extrapolated"]
    assert whole["value"] > 0 and whole["full_step_s"] > 0 and whole["cpu"]
    assert whole["sample"].startswith("whole step")
    pp = 32 * 16 * 16
    assert abs(whole["value"] - pp / (whole["rc_s"] + whole["bp_s"]) / 1e9) <= 0.02 * whole["value"] + 1e-5
    # a sampled record (the spotlight rule: first 256 pulses, central 256^2 pixels) extrapolates
    big = dataclasses.replace(synth.SCENES[1], n_pulses=300, nx=300, ny=300)
    s2 = synth.make_scene(big, device="cpu")
    samp = bench.oracle_baseline(s2, 3, threads=1)
    assert samp["extrapolated"] and "256 of 300" in samp["sample"] and "256x256" in samp["sample"]
    sweep = synth.make_rc_sweep(1024, n_lines=64, device="cpu")
    rc = bench.oracle_rc_baseline(sweep, threads=1)
    assert rc["unit"] == "lines/s" and rc["value"] > 0 and not rc["extrapolated"]
    rc1 = bench.oracle_rc_baseline(synth.make_rc_sweep(1024, n_lines=1024, device="cpu"), threads=1)
    assert rc1["extrapolated"] and "512 of 1024" in rc1["sample"]
    assert bench.central_pixels(cfg.grid(), 4).tolist() == [6 * 16 + 6 + i + 16 * j for j in range(4) for i in range(4)]
