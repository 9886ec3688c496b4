"""fp64 CPU oracle for SAR range compression and time-domain backprojection.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
bench's CPU-baseline leg, never by the CUDA library.  The arithmetic lives in
``sar_oracle.c``; this module only marshals numpy arrays through ctypes.
"""
import ctypes
import os

import numpy as np

from .build import build as _build

_lib = None


class OrRadar(ctypes.Structure):
    _fields_ = [("fc", ctypes.c_double), ("bandwidth", ctypes.c_double), ("pulse_width", ctypes.c_double),
                ("fs", ctypes.c_double), ("range_start", ctypes.c_double),
                ("n_pulses", ctypes.c_int32), ("n_range", ctypes.c_int32), ("upsample", ctypes.c_int32)]


class OrGrid(ctypes.Structure):
    _fields_ = [("x0", ctypes.c_double), ("y0", ctypes.c_double), ("z0", ctypes.c_double),
                ("dx", ctypes.c_double), ("dy", ctypes.c_double), ("nx", ctypes.c_int32), ("ny", ctypes.c_int32)]


def lib():
    global _lib
    if _lib is None:
        path = _build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        L.or_dft.argtypes = [P, ctypes.c_int64, ctypes.c_int]
        L.or_chirp_count.argtypes = [P]
        L.or_chirp_count.restype = ctypes.c_int32
        L.or_matched_filter.argtypes = [P, ctypes.c_int32, P]
        L.or_range_compress.argtypes = [P, P, ctypes.c_int64, P, ctypes.c_int]
        L.or_window.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_double, P]
        L.or_matched_filter_w.argtypes = [P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_double, P]
        L.or_range_compress_w.argtypes = [P, P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_double, P,
                                          ctypes.c_int]
        L.or_backproject.argtypes = [P, P, P, P, ctypes.c_int32, ctypes.c_int32, P, ctypes.c_int64, P,
                                     ctypes.c_int, ctypes.c_int]
        L.or_backproject_interp.argtypes = [P, P, P, P, ctypes.c_int32, ctypes.c_int32, P, ctypes.c_int64, P,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.or_sinc8_kernel.argtypes = [ctypes.c_double]
        L.or_sinc8_kernel.restype = ctypes.c_double
        L.or_interp_line.argtypes = [P, ctypes.c_int64, P, ctypes.c_int64, ctypes.c_int, P]
        L.or_range_doppler.argtypes = [P, ctypes.c_double, P, P, ctypes.c_int, ctypes.c_int]
        L.or_range_doppler.restype = ctypes.c_int
        L.or_max_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _radar(r, upsample=None, n_range=None):
    return OrRadar(r.fc, r.bandwidth, r.pulse_width, r.fs, r.range_start, r.n_pulses,
                   r.n_range if n_range is None else n_range, r.upsample if upsample is None else upsample)


def _grid(g):
    return OrGrid(g.x0, g.y0, g.z0, g.dx, g.dy, g.nx, g.ny)


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def dft(x, sign=-1):
    """sum_j x[j] exp(sign 2 pi i j k / n) for any n (radix-2, or Bluestein on radix-2)."""
    z = np.ascontiguousarray(x, dtype=np.complex128).copy()
    lib().or_dft(_ptr(z), z.size, int(sign))
    return z


def chirp_count(radar):
    return int(lib().or_chirp_count(ctypes.byref(_radar(radar))))


WINDOW_NONE, WINDOW_HAMMING, WINDOW_TAYLOR = 0, 1, 2


def window(kind, nc, nbar=4, sll_db=35.0):
    """The nc range weights of the reference chirp (kind: WINDOW_NONE / _HAMMING / _TAYLOR)."""
    w = np.zeros(nc, dtype=np.float64)
    lib().or_window(int(kind), int(nc), int(nbar), float(sll_db), _ptr(w))
    return w


def matched_filter(radar, n=None, window=WINDOW_NONE, nbar=4, sll_db=35.0):
    n = radar.n_range if n is None else n
    H = np.zeros(n, dtype=np.complex128)
    lib().or_matched_filter_w(ctypes.byref(_radar(radar, n_range=n)), n, int(window), int(nbar), float(sll_db),
                              _ptr(H))
    return H


def range_compress(radar, raw, upsample=None, threads=0, window=WINDOW_NONE, nbar=4, sll_db=35.0):
    """raw [lines][N] complex64 -> rc [lines][U N] complex128 (matched filter weighted by `window`)."""
    raw = np.ascontiguousarray(raw, dtype=np.complex64)
    lines, n = raw.shape
    U = radar.upsample if upsample is None else upsample
    r = _radar(radar, upsample=U, n_range=n)
    rc = np.zeros((lines, U * n), dtype=np.complex128)
    lib().or_range_compress_w(ctypes.byref(r), _ptr(raw), lines, int(window), int(nbar), float(sll_db), _ptr(rc),
                              int(threads))
    return rc


INTERP_LINEAR, INTERP_SINC8 = 0, 1


def sinc8_kernel(d):
    """The 8-tap sinc interpolation kernel h(d) (or_sinc8_kernel)."""
    return float(lib().or_sinc8_kernel(float(d)))


def interp_line(line, q, interp=INTERP_LINEAR):
    """Interpolate one complex line at fractional sample indices q (or_interp_line)."""
    line = np.ascontiguousarray(line, dtype=np.complex128)
    q = np.ascontiguousarray(q, dtype=np.float64)
    out = np.zeros(q.shape, dtype=np.complex128)
    lib().or_interp_line(_ptr(line), line.size, _ptr(q), q.size, int(interp), _ptr(out))
    return out


def backproject(radar, grid, rc, pos, pulse_begin=0, pulse_count=None, pixels=None, out=None,
                accumulate=False, threads=0, interp=INTERP_LINEAR):
    """rc [pulses][U N] (widened to complex128), pos [pulses][3] float64 -> image.

    pixels None: returns the full [ny][nx] complex128 image; otherwise a flat
    array of the listed pixels (flat index iy * nx + ix).  interp: INTERP_LINEAR
    or INTERP_SINC8."""
    rc = np.ascontiguousarray(rc, dtype=np.complex128)
    pos = np.ascontiguousarray(pos, dtype=np.float64)
    if pulse_count is None:
        pulse_count = rc.shape[0] - pulse_begin
    U = rc.shape[1] // radar.n_range
    r = _radar(radar, upsample=U)
    if pixels is None:
        shape, pix, npix = (grid.ny, grid.nx), None, grid.nx * grid.ny
    else:
        pix = np.ascontiguousarray(pixels, dtype=np.int64)
        shape, npix = pix.shape, pix.size
    if out is None:
        out = np.zeros(shape, dtype=np.complex128)
    lib().or_backproject_interp(ctypes.byref(r), ctypes.byref(_grid(grid)), _ptr(rc), _ptr(pos),
                                int(pulse_begin), int(pulse_count), None if pix is None else _ptr(pix), npix,
                                _ptr(out), int(bool(accumulate)), int(interp), int(threads))
    return out


def range_doppler(radar, rc, pulse_spacing, rcmc=True, threads=0):
    """Range-Doppler image [Nr][Na] complex128 of range-compressed lines rc [Na][Nr] (upsample 1) from a
    straight track with `pulse_spacing` metres between pulses (or_range_doppler)."""
    rc = np.ascontiguousarray(rc, dtype=np.complex128)
    na, nr = rc.shape
    r = _radar(radar, upsample=1, n_range=nr)
    r.n_pulses = na
    img = np.zeros((nr, na), dtype=np.complex128)
    st = lib().or_range_doppler(ctypes.byref(r), float(pulse_spacing), _ptr(rc), _ptr(img), int(bool(rcmc)),
                                int(threads))
    if st != 0:
        raise ValueError("pulse spacing too small for the range-Doppler model (lambda / (4 du) >= 1)")
    return img


def form_image(radar, grid, raw, pos, threads=0):
    rc = range_compress(radar, raw, threads=threads)
    return backproject(radar, grid, rc, pos, threads=threads)


def max_threads():
    return int(lib().or_max_threads())
