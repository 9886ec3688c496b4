"""Pins for the oracle's range weighting ("GPU-accelerated backprojection SAR imaging", section 3.1:
an unweighted matched filter leaves about -13 dB range sidelobes, and a Hamming or Taylor weight
lowers them at the cost of a wider main lobe).  The weights are checked against an independent
implementation (scipy), the weighted compression of an on-grid echo against its direct time-domain
correlation, and the compressed point response against the windows' known sidelobe levels."""
import dataclasses
import math

import numpy as np
import pytest

import oracle
from test_oracle_rc import BETA, RADAR, on_grid_echo

windows = pytest.importorskip("scipy.signal.windows")


@pytest.mark.parametrize("nc", [360, 361, 64])
def test_weights_match_an_independent_implementation(nc):
    assert np.array_equal(oracle.window(oracle.WINDOW_NONE, nc), np.ones(nc))
    assert np.abs(oracle.window(oracle.WINDOW_HAMMING, nc) - windows.hamming(nc, sym=True)).max() < 1e-13
    for nbar, sll in ((4, 35.0), (5, 40.0), (6, 30.0)):
        ref = windows.taylor(nc, nbar=nbar, sll=sll, norm=False, sym=True)
        assert np.abs(oracle.window(oracle.WINDOW_TAYLOR, nc, nbar, sll) - ref).max() < 1e-13


@pytest.mark.parametrize("kind", [oracle.WINDOW_HAMMING, oracle.WINDOW_TAYLOR])
def test_weighted_compression_equals_direct_correlation(kind):
    # rc[m0 + l] = sum_s echo(m0 + l + s) conj(w_s h(s)) for the on-grid echo echo(m0 + k) = h(k)
    # (the echo as stored, complex64, so that both sides see the same input)
    n, m0 = 1024, 500
    r = dataclasses.replace(RADAR, n_range=n, upsample=1)
    x = on_grid_echo(n, m0, 1.0)
    rc = oracle.range_compress(r, x[None, :], window=kind)[0]
    s = np.arange(-180, 180)
    h = np.exp(1j * math.pi * BETA * s.astype(float) ** 2)
    w = oracle.window(kind, 360)
    xd = x.astype(np.complex128)
    for lag in range(-400, 401, 7):
        k = m0 + lag + s
        echo = np.where((k >= 0) & (k < n), xd[np.clip(k, 0, n - 1)], 0)
        want = np.sum(echo * np.conj(w * h))
        assert abs(rc[m0 + lag] - want) <= 1e-10 * 360
    assert abs(rc[m0] - w.sum()) <= 1e-5                  # coherent gain of the weight (input in float32)


def _lobe_db(mag, pk):
    """-3 dB main-lobe width (samples) and the highest sidelobe (dB) of a compressed response."""
    db = 20 * np.log10(mag / mag[pk] + 1e-300)
    edges, worst = [], -300.0
    for side in (+1, -1):
        i = pk
        while db[i + side] > -3.0:
            i += side
        # interpolate the -3 dB crossing between samples i and i + side
        frac = (db[i] + 3.0) / (db[i] - db[i + side])
        edges.append(i + side * frac)
        while db[i + side] < db[i]:               # down to the first null
            i += side
        lo, hi = (i, i + 40 * 8) if side > 0 else (i - 40 * 8, i + 1)
        worst = max(worst, db[lo:hi].max())
    return abs(edges[0] - edges[1]), worst


def test_point_response_sidelobes_and_width():
    n, U = 1024, 8
    r = dataclasses.replace(RADAR, n_range=n, upsample=U)
    raw = on_grid_echo(n, 500, 1.0)[None, :]
    res = {}
    for kind, nbar, sll in ((oracle.WINDOW_NONE, 4, 35.0), (oracle.WINDOW_HAMMING, 4, 35.0),
                            (oracle.WINDOW_TAYLOR, 4, 35.0)):
        mag = np.abs(oracle.range_compress(r, raw, window=kind, nbar=nbar, sll_db=sll)[0])
        pk = int(mag.argmax())
        assert pk == 500 * U
        res[kind] = _lobe_db(mag, pk)
    w0, s0 = res[oracle.WINDOW_NONE]
    wh, sh = res[oracle.WINDOW_HAMMING]
    wt, st = res[oracle.WINDOW_TAYLOR]
    assert abs(s0 - (-13.26)) < 0.5                        # unweighted: the sinc's first sidelobe
    assert sh < -38.0                                      # Hamming: about -42 dB
    assert -37.5 < st < -32.5                              # Taylor: its design level, -35 dB
    assert 1.35 < wh / w0 < 1.6 and 1.15 < wt / w0 < 1.45  # the main lobe widens
