"""Writes oracle_point_patch.json: a regression fixture computed by the oracle alone.

A noise-free scatterer on a pixel centre of the tiny stripmap geometry, cut
to 32 pulses; the fixture holds the 5x5 image patch around the scatterer.  Any
later change to the oracle's arithmetic must regenerate it with this script and
name the passage that justifies the change.
"""
import dataclasses
import json
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402
from synth.scenes import add_echoes  # noqa: E402


def compute():
    cfg = dataclasses.replace(synth.SCENES[1], n_pulses=32, prf=300.0 / 8)
    radar, grid = cfg.radar(), cfg.grid()
    pos = synth.track(cfg)
    xyz = torch.tensor([[grid.x0 + 64 * grid.dx, grid.y0 + 64 * grid.dy, 0.0]], dtype=torch.float64)
    raw = torch.zeros(cfg.n_pulses, cfg.n_range, dtype=torch.complex64)
    add_echoes(raw, pos, xyz, torch.tensor([1.0 + 0j], dtype=torch.complex128), radar)
    rc = oracle.range_compress(radar, raw.numpy())
    patch = synth.Grid(grid.x0 + 62 * grid.dx, grid.y0 + 62 * grid.dy, grid.z0, grid.dx, grid.dy, 5, 5)
    return oracle.backproject(radar, patch, rc, pos.numpy())


if __name__ == "__main__":
    img = compute()
    with open(os.path.join(HERE, "oracle_point_patch.json"), "w") as f:
        json.dump({"_about": __doc__.strip().splitlines()[0],
                   "re": np.round(img.real, 9).tolist(), "im": np.round(img.imag, 9).tolist()}, f, indent=1)
