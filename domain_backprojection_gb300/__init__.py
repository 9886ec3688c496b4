"""GB300-native SAR image formation: fused range compression and time-domain
backprojection as hand-written CUDA kernels for sm_103a behind a small C ABI
(include/sar.h).  This package is the thin Python binding of that ABI; the
function names are the C entry points'."""
from ._binding import (SAR_ACCUM_COMPENSATED, SAR_ACCUM_FP32, SAR_INTERP_LINEAR, SAR_INTERP_SINC8, SAR_OK,
                       SAR_RC_NATURAL, SAR_RC_POLYPHASE, SAR_STAGE_FP16, SAR_STAGE_FP32, SAR_WINDOW_HAMMING,
                       SAR_WINDOW_NONE, SAR_WINDOW_TAYLOR, Plan, SarError, declared_symbols, lib, library_path,
                       sar_backproject, sar_form_image, sar_form_image_host, sar_plan_create, sar_plan_destroy,
                       sar_plan_kernel_times, sar_plan_last_launches, sar_plan_set_accumulation,
                       sar_plan_set_interpolation, sar_plan_set_pulse_weights, sar_plan_set_range_window,
                       sar_plan_set_range_doppler, sar_plan_set_rc_layout, sar_plan_set_stage_precision, sar_plan_set_timing,
                       sar_plan_sync, sar_range_compress, sar_range_doppler, sar_range_doppler_workspace_size,
                       sar_status_string, sar_workspace_size)
from .build import build as build_library

__all__ = ["SAR_ACCUM_COMPENSATED", "SAR_ACCUM_FP32", "SAR_INTERP_LINEAR", "SAR_INTERP_SINC8", "SAR_OK",
           "SAR_RC_NATURAL", "SAR_RC_POLYPHASE", "SAR_STAGE_FP16", "SAR_STAGE_FP32", "SAR_WINDOW_HAMMING",
           "SAR_WINDOW_NONE", "SAR_WINDOW_TAYLOR", "Plan", "SarError", "build_library", "declared_symbols", "lib",
           "library_path", "sar_backproject", "sar_form_image", "sar_form_image_host", "sar_plan_create",
           "sar_plan_destroy", "sar_plan_kernel_times", "sar_plan_last_launches", "sar_plan_set_accumulation",
           "sar_plan_set_interpolation", "sar_plan_set_pulse_weights", "sar_plan_set_range_window",
           "sar_plan_set_range_doppler", "sar_plan_set_rc_layout", "sar_plan_set_stage_precision", "sar_plan_set_timing",
           "sar_plan_sync", "sar_range_compress", "sar_range_doppler", "sar_range_doppler_workspace_size",
           "sar_status_string", "sar_workspace_size"]
