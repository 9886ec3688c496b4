"""Checks against numbers the pages print (tests/golden/page_facts.json) and the oracle's
regression fixture (tests/golden/oracle_point_patch.json, written by make_golden.py)."""
import json
import os

import numpy as np

import synth

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _facts():
    with open(os.path.join(GOLD, "page_facts.json")) as f:
        return json.load(f)


def test_pixel_pulse_counts_match_printed_examples():
    # the cost model O(Na Nx Ny) and its two worked examples
    for ex in _facts()["pixel_pulse_examples"]:
        assert abs(ex["n_pulses"] * ex["nx"] * ex["ny"] / ex["printed"] - 1) < 0.02
    # the benchmark scenes sized like the pages' examples
    assert synth.SCENES[3].pixel_pulses == 4096 * 1024 * 1024
    assert synth.SCENES[4].pixel_pulses == 16384 * 2048 * 2048


def test_sinc_first_sidelobe_is_near_printed_value():
    # first sidelobe of sin(x)/x, found numerically, against the printed "about -13 dB"
    x = np.linspace(np.pi + 1e-6, 2 * np.pi - 1e-6, 200001)
    peak = np.max(np.abs(np.sin(x) / x))
    db = 20 * np.log10(peak)
    fact = _facts()["unweighted_sidelobe_db"]
    assert abs(db - fact["printed"]) < fact["tolerance_db"]
    assert abs(db - (-13.26)) < 0.005


def test_oracle_regression_fixture():
    import sys
    sys.path.insert(0, GOLD)
    import make_golden
    img = make_golden.compute()
    with open(os.path.join(GOLD, "oracle_point_patch.json")) as f:
        ref = json.load(f)
    want = np.array(ref["re"]) + 1j * np.array(ref["im"])
    assert np.abs(img - want).max() <= 1e-8 * np.abs(want).max()
