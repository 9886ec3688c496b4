"""Comparison helpers shared by the GPU parity tests (no method arithmetic here)."""
import os

import numpy as np

import oracle

ORACLE_THREADS = int(os.environ.get("SAR_ORACLE_THREADS", "0"))   # 0 = all cores

RC_TOL = 2e-4       # relative L2, range compression
IMG_TOL = 1e-3      # relative L2, image
PEAK_DB_TOL = 0.05  # peak magnitude, dB
SNR_DB_TOL = 0.05   # per-target peak-to-background ratio, dB
SNR_HALF = 10       # SNR window: (2 SNR_HALF + 1)^2 pixels centred on the target's pixel
SNR_LOBE = 3        # main lobe excluded from the background: pixels within this Chebyshev distance of the peak


def rel_l2(got, ref):
    got = np.asarray(got, dtype=np.complex128)
    ref = np.asarray(ref, dtype=np.complex128)
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))


def oracle_image_pixels(radar, grid, raw, pos, pixels, chunk=2048, interp=oracle.INTERP_LINEAR):
    """Oracle image at the listed flat pixel indices, range-compressing and
    backprojecting the pulses in chunks so that float64 lines never exceed a
    few GB of host memory."""
    raw = np.ascontiguousarray(raw)
    pos = np.ascontiguousarray(pos)
    na = raw.shape[0]
    out = np.zeros(np.asarray(pixels).shape, dtype=np.complex128)
    for n0 in range(0, na, chunk):
        n1 = min(na, n0 + chunk)
        rc = oracle.range_compress(radar, raw[n0:n1], threads=ORACLE_THREADS)
        oracle.backproject(radar, grid, rc, pos[n0:n1], pixels=pixels, out=out, accumulate=True,
                           threads=ORACLE_THREADS, interp=interp)
    return out


def window_pixels(grid, centres, half):
    """Flat indices of the (2 half + 1)^2 windows around integer pixel centres (ix, iy), clipped."""
    idx = []
    for ix, iy in centres:
        for dy in range(-half, half + 1):
            for dx in range(-half, half + 1):
                x, y = ix + dx, iy + dy
                if 0 <= x < grid.nx and 0 <= y < grid.ny:
                    idx.append(y * grid.nx + x)
    return np.unique(np.array(idx, dtype=np.int64))


def check_peaks(img_gpu, img_ref, grid, centres, half):
    """Per point target: the peak pixel inside its window must be the same in both images (when the
    oracle's top two are within 1e-3 the GPU may pick either), and the peak magnitude must agree
    within PEAK_DB_TOL dB.  Images are full [ny][nx] arrays (pixels outside windows unused)."""
    worst = 0.0
    for ix, iy in centres:
        y0, y1 = max(0, iy - half), min(grid.ny, iy + half + 1)
        x0, x1 = max(0, ix - half), min(grid.nx, ix + half + 1)
        ref = np.abs(img_ref[y0:y1, x0:x1])
        got = np.abs(img_gpu[y0:y1, x0:x1])
        order = np.argsort(ref.ravel())[::-1]
        best = order[0]
        ties = [i for i in order[:4] if ref.ravel()[i] >= ref.ravel()[best] * (1 - 1e-3)]
        g = int(np.argmax(got))
        assert g in ties, f"target ({ix},{iy}): GPU peak {np.unravel_index(g, got.shape)} vs oracle " \
                          f"{np.unravel_index(best, ref.shape)}"
        db = abs(20 * np.log10(got.ravel()[g] / ref.ravel()[best]))
        worst = max(worst, db)
        assert db <= PEAK_DB_TOL, f"target ({ix},{iy}): peak differs by {db:.4f} dB"
    return worst


def target_pixels(scene):
    """Nearest pixel centre of every point target."""
    g = scene["grid"]
    xyz = scene["target_xyz"].numpy()
    ix = np.rint((xyz[:, 0] - g.x0) / g.dx).astype(int)
    iy = np.rint((xyz[:, 1] - g.y0) / g.dy).astype(int)
    return list(zip(ix.tolist(), iy.tolist()))


def target_snr_db(img, grid, centre, half=SNR_HALF, lobe=SNR_LOBE, peak_at=None):
    """Peak-to-background ratio (dB) of one point target: the largest magnitude in the window of
    half-width `half` around `centre`, over the RMS magnitude of the window's pixels farther than
    `lobe` pixels (Chebyshev distance) from the peak (the main lobe excluded).  `peak_at` fixes the
    peak pixel (window coordinates) instead of searching for it.  Returns (snr_db, peak_index)."""
    ix, iy = centre
    y0, y1 = max(0, iy - half), min(grid.ny, iy + half + 1)
    x0, x1 = max(0, ix - half), min(grid.nx, ix + half + 1)
    a = np.abs(np.asarray(img)[y0:y1, x0:x1])
    py, px = np.unravel_index(int(np.argmax(a)), a.shape) if peak_at is None else peak_at
    yy, xx = np.mgrid[0:a.shape[0], 0:a.shape[1]]
    bg = a[np.maximum(np.abs(yy - py), np.abs(xx - px)) > lobe]
    return 20.0 * np.log10(a[py, px] / np.sqrt(np.mean(bg ** 2))), (py, px)


def check_snr(img_gpu, img_ref, grid, centres):
    """Per point target, the GPU image's peak-to-background ratio must match the oracle's within
    SNR_DB_TOL dB (both measured around the oracle's peak pixel).  Returns the largest difference."""
    worst = 0.0
    for c in centres:
        ref_db, peak = target_snr_db(img_ref, grid, c)
        got_db, _ = target_snr_db(img_gpu, grid, c, peak_at=peak)
        d = abs(got_db - ref_db)
        worst = max(worst, d)
        assert d <= SNR_DB_TOL, f"target {c}: SNR {got_db:.4f} dB vs oracle {ref_db:.4f} dB"
    return worst
