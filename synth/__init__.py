"""Seeded synthetic SAR inputs shared by the oracle-side tests and the CUDA library's tests and bench."""
from .scenes import (C0, SCENES, RC_SWEEP_NR, Grid, Radar, SceneConfig, chirp_count, make_rc_sweep,
                     make_scene, track, targets, clutter)
