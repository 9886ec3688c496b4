"""ctypes binding of the C ABI in include/sar.h.

Argument marshalling only: every function below checks tensor dtypes, devices
and shapes, passes raw pointers and the current torch stream to the native
library, and turns status codes into exceptions.  All arithmetic runs in the
CUDA kernels of ``libsar.so``; there is no fallback.  If the library is missing
and cannot be built, importing the first entry point raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import build as _build

_lib = None

SAR_OK = 0
SAR_RC_NATURAL = 0
SAR_RC_POLYPHASE = 1
STATUS_NAMES = {0: "SAR_OK", 1: "SAR_ERR_INVALID_ARG", 2: "SAR_ERR_UNSUPPORTED", 3: "SAR_ERR_NO_MEMORY",
                4: "SAR_ERR_CUDA", 5: "SAR_ERR_TIMEOUT", 6: "SAR_ERR_INTERNAL"}


class SarError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS_NAMES.get(self.status, self.status)} ({sar_status_string(self.status)})")


class sar_radar(ctypes.Structure):
    _fields_ = [("fc", ctypes.c_double), ("bandwidth", ctypes.c_double), ("pulse_width", ctypes.c_double),
                ("fs", ctypes.c_double), ("range_start", ctypes.c_double),
                ("n_pulses", ctypes.c_int32), ("n_range", ctypes.c_int32), ("upsample", ctypes.c_int32)]


class sar_grid(ctypes.Structure):
    _fields_ = [("x0", ctypes.c_double), ("y0", ctypes.c_double), ("z0", ctypes.c_double),
                ("dx", ctypes.c_double), ("dy", ctypes.c_double), ("nx", ctypes.c_int32), ("ny", ctypes.c_int32)]


def library_path() -> str:
    return _build.LIB


def declared_symbols() -> list:
    """Entry points declared in include/sar.h."""
    with open(os.path.join(_build.ROOT, "include", "sar.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(sar_\w+)\s*\(", text, re.M)))


def load_library(path: str):
    """Load a build of libsar.so at `path` and declare its entry points' signatures."""
    L = ctypes.CDLL(path)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "sar_plan_create": ([P, P, ctypes.c_int, P], ctypes.c_int),
        "sar_plan_destroy": ([P], ctypes.c_int),
        "sar_workspace_size": ([P, P], ctypes.c_int),
        "sar_range_compress": ([P, P, P, I64, P], ctypes.c_int),
        "sar_backproject": ([P, P, P, I32, I32, P, ctypes.c_int, P], ctypes.c_int),
        "sar_form_image": ([P, P, P, P, P, SZ, P], ctypes.c_int),
        "sar_form_image_host": ([P, P, P, P, P], ctypes.c_int),
        "sar_plan_sync": ([P, P], ctypes.c_int),
        "sar_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "sar_plan_last_launches": ([P], I32),
        "sar_plan_set_rc_layout": ([P, ctypes.c_int], ctypes.c_int),
        "sar_plan_set_timing": ([P, ctypes.c_int], ctypes.c_int),
        "sar_plan_set_range_window": ([P, ctypes.c_int, I32, ctypes.c_double], ctypes.c_int),
        "sar_plan_set_pulse_weights": ([P, P], ctypes.c_int),
        "sar_plan_kernel_times": ([P, P, P, P, P], ctypes.c_int),
        "sar_plan_set_accumulation": ([P, ctypes.c_int], ctypes.c_int),
        "sar_plan_set_stage_precision": ([P, ctypes.c_int], ctypes.c_int),
        "sar_plan_set_interpolation": ([P, ctypes.c_int], ctypes.c_int),
        "sar_plan_set_range_doppler": ([P, ctypes.c_double], ctypes.c_int),
        "sar_range_doppler_workspace_size": ([P, P], ctypes.c_int),
        "sar_range_doppler": ([P, P, P, P, SZ, P], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = load_library(_build.build())
    return _lib


def _check(status, where):
    if status != SAR_OK:
        raise SarError(status, where)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev_tensor(t, dtype, name, device):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous CUDA tensor of dtype {dtype}")
    if t.device.index != device:
        raise ValueError(f"{name} is on cuda:{t.device.index}, the plan on cuda:{device}")
    return ctypes.c_void_p(t.data_ptr())


class Plan:
    """Owns a native sar_plan handle; destroyed with the object or by sar_plan_destroy."""

    def __init__(self, handle, radar, grid, device):
        self.handle = handle
        self.radar = radar
        self.grid = grid
        self.device = device

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.sar_plan_destroy(self.handle)
            self.handle = None

    @property
    def samples(self):
        return self.radar.n_range * self.radar.upsample


def _to_radar(r) -> sar_radar:
    return sar_radar(float(r.fc), float(r.bandwidth), float(r.pulse_width), float(r.fs), float(r.range_start),
                     int(r.n_pulses), int(r.n_range), int(r.upsample))


def _to_grid(g) -> sar_grid:
    return sar_grid(float(g.x0), float(g.y0), float(g.z0), float(g.dx), float(g.dy), int(g.nx), int(g.ny))


def sar_status_string(status: int) -> str:
    return lib().sar_status_string(int(status)).decode()


def sar_plan_create(radar, grid=None, device: int = 0) -> Plan:
    r = _to_radar(radar)
    g = _to_grid(grid) if grid is not None else None
    h = ctypes.c_void_p()
    _check(lib().sar_plan_create(ctypes.byref(r), ctypes.byref(g) if g is not None else None, int(device),
                                 ctypes.byref(h)), "sar_plan_create")
    return Plan(h, r, g, int(device))


def sar_plan_destroy(plan: Plan) -> None:
    if plan.handle:
        _check(lib().sar_plan_destroy(plan.handle), "sar_plan_destroy")
        plan.handle = None


def sar_workspace_size(plan: Plan) -> int:
    n = ctypes.c_size_t()
    _check(lib().sar_workspace_size(plan.handle, ctypes.byref(n)), "sar_workspace_size")
    return int(n.value)


def sar_range_compress(plan: Plan, raw: torch.Tensor, rc: torch.Tensor = None, stream=None) -> torch.Tensor:
    """raw [lines][Nr] complex64 (CUDA) -> rc [lines][U Nr] complex64."""
    if raw.dim() != 2 or raw.shape[1] != plan.radar.n_range:
        raise ValueError(f"raw must be [lines][{plan.radar.n_range}]")
    lines = raw.shape[0]
    if rc is None:
        rc = torch.empty(lines, plan.samples, dtype=torch.complex64, device=raw.device)
    if tuple(rc.shape) != (lines, plan.samples):
        raise ValueError(f"rc must be [{lines}][{plan.samples}]")
    _check(lib().sar_range_compress(plan.handle, _dev_tensor(raw, torch.complex64, "raw", plan.device),
                                    _dev_tensor(rc, torch.complex64, "rc", plan.device), lines, _stream(stream)),
           "sar_range_compress")
    return rc


def sar_backproject(plan: Plan, rc: torch.Tensor, pos: torch.Tensor, pulse_begin: int = 0, pulse_count=None,
                    image: torch.Tensor = None, accumulate: bool = False, stream=None) -> torch.Tensor:
    """rc [Na][U Nr] complex64, pos [Na][3] float64 (CUDA) -> image [ny][nx] complex64."""
    na = plan.radar.n_pulses
    if tuple(rc.shape) != (na, plan.samples):
        raise ValueError(f"rc must be [{na}][{plan.samples}]")
    if tuple(pos.shape) != (na, 3):
        raise ValueError(f"pos must be [{na}][3]")
    if plan.grid is None:
        raise SarError(2, "sar_backproject (plan has no grid)")
    if pulse_count is None:
        pulse_count = na - pulse_begin
    if image is None:
        image = (torch.zeros if accumulate else torch.empty)(plan.grid.ny, plan.grid.nx, dtype=torch.complex64,
                                                             device=rc.device)
    if tuple(image.shape) != (plan.grid.ny, plan.grid.nx):
        raise ValueError(f"image must be [{plan.grid.ny}][{plan.grid.nx}]")
    _check(lib().sar_backproject(plan.handle, _dev_tensor(rc, torch.complex64, "rc", plan.device),
                                 _dev_tensor(pos, torch.float64, "pos", plan.device), int(pulse_begin),
                                 int(pulse_count), _dev_tensor(image, torch.complex64, "image", plan.device),
                                 int(bool(accumulate)), _stream(stream)), "sar_backproject")
    return image


def sar_form_image(plan: Plan, raw: torch.Tensor, pos: torch.Tensor, image: torch.Tensor = None,
                   workspace: torch.Tensor = None, stream=None) -> torch.Tensor:
    """raw [Na][Nr] complex64, pos [Na][3] float64 (CUDA) -> image [ny][nx] complex64."""
    na = plan.radar.n_pulses
    if tuple(raw.shape) != (na, plan.radar.n_range) or tuple(pos.shape) != (na, 3):
        raise ValueError("raw must be [Na][Nr] and pos [Na][3]")
    if plan.grid is None:
        raise SarError(2, "sar_form_image (plan has no grid)")
    ws_bytes = sar_workspace_size(plan)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=raw.device)
    if workspace.dtype != torch.uint8 or workspace.numel() < ws_bytes or not workspace.is_cuda:
        raise ValueError(f"workspace must be a CUDA uint8 tensor of at least {ws_bytes} bytes")
    if image is None:
        image = torch.empty(plan.grid.ny, plan.grid.nx, dtype=torch.complex64, device=raw.device)
    _check(lib().sar_form_image(plan.handle, _dev_tensor(raw, torch.complex64, "raw", plan.device),
                                _dev_tensor(pos, torch.float64, "pos", plan.device),
                                _dev_tensor(image, torch.complex64, "image", plan.device),
                                _dev_tensor(workspace, torch.uint8, "workspace", plan.device),
                                workspace.numel(), _stream(stream)), "sar_form_image")
    return image


def sar_form_image_host(plan: Plan, raw: torch.Tensor, pos: torch.Tensor, image: torch.Tensor = None,
                        stream=None) -> torch.Tensor:
    """Host (ideally pinned) raw [Na][Nr] complex64 and pos [Na][3] float64 -> host image [ny][nx] complex64."""
    na = plan.radar.n_pulses
    for t, name, dt in ((raw, "raw", torch.complex64), (pos, "pos", torch.float64)):
        if t.is_cuda or t.dtype != dt or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous host tensor of dtype {dt}")
    if tuple(raw.shape) != (na, plan.radar.n_range) or tuple(pos.shape) != (na, 3):
        raise ValueError("raw must be [Na][Nr] and pos [Na][3]")
    if image is None:
        image = torch.empty(plan.grid.ny, plan.grid.nx, dtype=torch.complex64, pin_memory=True)
    if image.is_cuda or image.dtype != torch.complex64 or tuple(image.shape) != (plan.grid.ny, plan.grid.nx):
        raise TypeError("image must be a host complex64 tensor [ny][nx]")
    _check(lib().sar_form_image_host(plan.handle, ctypes.c_void_p(raw.data_ptr()), ctypes.c_void_p(pos.data_ptr()),
                                     ctypes.c_void_p(image.data_ptr()), _stream(stream)), "sar_form_image_host")
    return image


def sar_plan_sync(plan: Plan, stream=None) -> None:
    _check(lib().sar_plan_sync(plan.handle, _stream(stream)), "sar_plan_sync")


def sar_plan_set_rc_layout(plan: Plan, layout: int) -> None:
    """SAR_RC_NATURAL (sample U m + u at U m + u) or SAR_RC_POLYPHASE (at u Nr + m)."""
    _check(lib().sar_plan_set_rc_layout(plan.handle, int(layout)), "sar_plan_set_rc_layout")
    plan.layout = int(layout)


def sar_plan_last_launches(plan: Plan) -> int:
    return int(lib().sar_plan_last_launches(plan.handle))


def sar_plan_set_timing(plan: Plan, enable: bool = True) -> None:
    """Record CUDA events around each later call's main kernel (see sar_plan_kernel_times)."""
    _check(lib().sar_plan_set_timing(plan.handle, 1 if enable else 0), "sar_plan_set_timing")


def sar_plan_kernel_times(plan: Plan) -> dict:
    """Summed durations (ms) and call counts of the kernels recorded since timing was enabled or
    last read: {"rc_ms", "rc_calls", "bp_ms", "bp_calls"}; the record is then cleared."""
    rc_ms, bp_ms = ctypes.c_double(), ctypes.c_double()
    rc_n, bp_n = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().sar_plan_kernel_times(plan.handle, ctypes.byref(rc_ms), ctypes.byref(rc_n), ctypes.byref(bp_ms),
                                       ctypes.byref(bp_n)), "sar_plan_kernel_times")
    return {"rc_ms": rc_ms.value, "rc_calls": rc_n.value, "bp_ms": bp_ms.value, "bp_calls": bp_n.value}


SAR_WINDOW_NONE, SAR_WINDOW_HAMMING, SAR_WINDOW_TAYLOR = 0, 1, 2


def sar_plan_set_range_window(plan: Plan, window: int, taylor_nbar: int = 4, taylor_sll_db: float = 35.0) -> None:
    """Weight the plan's matched filter: SAR_WINDOW_NONE, SAR_WINDOW_HAMMING or SAR_WINDOW_TAYLOR."""
    _check(lib().sar_plan_set_range_window(plan.handle, int(window), int(taylor_nbar), float(taylor_sll_db)),
           "sar_plan_set_range_window")


def sar_plan_set_pulse_weights(plan: Plan, weights) -> None:
    """Per-pulse real weights for later backprojections: a CUDA float32 tensor [Na] (kept referenced by
    the plan while set), or None for unit weights."""
    if weights is None:
        _check(lib().sar_plan_set_pulse_weights(plan.handle, None), "sar_plan_set_pulse_weights")
        plan.weights = None
        return
    if tuple(weights.shape) != (plan.radar.n_pulses,):
        raise ValueError(f"weights must be [{plan.radar.n_pulses}]")
    _check(lib().sar_plan_set_pulse_weights(plan.handle, _dev_tensor(weights, torch.float32, "weights", plan.device)),
           "sar_plan_set_pulse_weights")
    plan.weights = weights


SAR_ACCUM_FP32, SAR_ACCUM_COMPENSATED = 0, 1
SAR_STAGE_FP32, SAR_STAGE_FP16 = 0, 1
SAR_INTERP_LINEAR, SAR_INTERP_SINC8 = 0, 1


def sar_plan_set_accumulation(plan: Plan, accumulation: int) -> None:
    """SAR_ACCUM_FP32 (plain float32 pulse sums) or SAR_ACCUM_COMPENSATED (batch sums folded into Kahan totals)."""
    _check(lib().sar_plan_set_accumulation(plan.handle, int(accumulation)), "sar_plan_set_accumulation")


def sar_plan_set_stage_precision(plan: Plan, precision: int) -> None:
    """SAR_STAGE_FP32 or SAR_STAGE_FP16 (float16 staged interpolation entries, float32 arithmetic)."""
    _check(lib().sar_plan_set_stage_precision(plan.handle, int(precision)), "sar_plan_set_stage_precision")


def sar_plan_set_interpolation(plan: Plan, interpolation: int) -> None:
    """SAR_INTERP_LINEAR or SAR_INTERP_SINC8 (8-tap Hann-tapered sinc, weights normalised to unit sum)."""
    _check(lib().sar_plan_set_interpolation(plan.handle, int(interpolation)), "sar_plan_set_interpolation")


def sar_plan_set_range_doppler(plan: Plan, pulse_spacing: float) -> None:
    """Azimuth tables for range-Doppler image formation of pulses `pulse_spacing` metres apart."""
    _check(lib().sar_plan_set_range_doppler(plan.handle, float(pulse_spacing)), "sar_plan_set_range_doppler")


def sar_range_doppler_workspace_size(plan: Plan) -> int:
    n = ctypes.c_size_t()
    _check(lib().sar_range_doppler_workspace_size(plan.handle, ctypes.byref(n)), "sar_range_doppler_workspace_size")
    return n.value


def sar_range_doppler(plan: Plan, raw: torch.Tensor, image: torch.Tensor = None, workspace: torch.Tensor = None,
                      stream=None) -> torch.Tensor:
    """Range-Doppler image [Nr][Na] complex64 of raw [Na][Nr] complex64 (see include/sar.h)."""
    r = plan.radar
    if tuple(raw.shape) != (r.n_pulses, r.n_range):
        raise ValueError(f"raw must be [{r.n_pulses}][{r.n_range}]")
    ws_bytes = sar_range_doppler_workspace_size(plan)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=raw.device)
    if workspace.dtype != torch.uint8 or workspace.numel() < ws_bytes or not workspace.is_cuda:
        raise ValueError(f"workspace must be a CUDA uint8 tensor of at least {ws_bytes} bytes")
    if image is None:
        image = torch.empty(r.n_range, r.n_pulses, dtype=torch.complex64, device=raw.device)
    if tuple(image.shape) != (r.n_range, r.n_pulses):
        raise ValueError(f"image must be [{r.n_range}][{r.n_pulses}]")
    _check(lib().sar_range_doppler(plan.handle, _dev_tensor(raw, torch.complex64, "raw", plan.device),
                                   _dev_tensor(image, torch.complex64, "image", plan.device),
                                   _dev_tensor(workspace, torch.uint8, "workspace", plan.device),
                                   workspace.numel(), _stream(stream)), "sar_range_doppler")
    return image
