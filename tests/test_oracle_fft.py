"""Pins for the oracle's transforms: its own radix-2 FFT and the Bluestein
(chirp-z) transform for other lengths ("Ultra-high-resolution airborne SAR on
CUDA", section 5.1), checked against brute-force DFT sums, closed forms,
identities and numpy's FFT -- never against the oracle itself."""
import numpy as np
import pytest

import oracle


def brute_dft(x, sign=-1):
    """O(N^2) DFT with exact integer reduction of j*k mod N before the exponential."""
    n = x.size
    jk = np.outer(np.arange(n), np.arange(n)) % n
    return np.exp(sign * 2j * np.pi * jk / n) @ x


def rand_c(n, seed):
    g = np.random.default_rng(seed)
    return g.standard_normal(n) + 1j * g.standard_normal(n)


@pytest.mark.parametrize("n", [1, 2, 8, 64, 256])
@pytest.mark.parametrize("sign", [-1, +1])
def test_pow2_matches_brute_force(n, sign):
    x = rand_c(n, n)
    ref = brute_dft(x, sign)
    got = oracle.dft(x, sign)
    assert np.linalg.norm(got - ref) <= 1e-12 * max(1.0, np.linalg.norm(ref))


@pytest.mark.parametrize("n", [3, 5, 15, 60, 375, 1000])
@pytest.mark.parametrize("sign", [-1, +1])
def test_bluestein_matches_brute_force(n, sign):
    x = rand_c(n, 7 * n)
    ref = brute_dft(x, sign)
    got = oracle.dft(x, sign)
    assert np.linalg.norm(got - ref) <= 1e-11 * np.linalg.norm(ref)


def test_bluestein_6000_sampled_bins():
    # the non-power-of-two range length of the range-compression sweep
    n = 6000
    x = rand_c(n, 6000)
    got = oracle.dft(x, -1)
    j = np.arange(n)
    for k in [0, 1, 2, 1499, 2999, 3000, 3001, 4567, 5999]:
        ref = np.sum(x * np.exp(-2j * np.pi * ((j * k) % n) / n))
        assert abs(got[k] - ref) <= 1e-10 * np.linalg.norm(x) * np.sqrt(n)


@pytest.mark.parametrize("n", [4096, 6000, 48000])
def test_matches_numpy_fft(n):
    x = rand_c(n, n + 1)
    assert np.linalg.norm(oracle.dft(x, -1) - np.fft.fft(x)) <= 1e-11 * np.linalg.norm(np.fft.fft(x))
    assert np.linalg.norm(oracle.dft(x, +1) - n * np.fft.ifft(x)) <= 1e-11 * np.linalg.norm(np.fft.fft(x))


@pytest.mark.parametrize("n", [1024, 6000])
def test_inverse_and_parseval(n):
    x = rand_c(n, 3)
    X = oracle.dft(x, -1)
    assert np.allclose(oracle.dft(X, +1) / n, x, rtol=0, atol=1e-12 * np.abs(x).max())
    assert abs(np.sum(np.abs(X) ** 2) / n - np.sum(np.abs(x) ** 2)) <= 1e-11 * np.sum(np.abs(x) ** 2)


@pytest.mark.parametrize("n", [512, 6000])
def test_conj_identity(n):
    # IFFT(x) = conj(FFT(conj(x))) / N  ("Fused FFT -> filter -> IFFT ...", section 3.2)
    x = rand_c(n, 11)
    lhs = oracle.dft(x, +1) / n
    rhs = np.conj(oracle.dft(np.conj(x), -1)) / n
    assert np.allclose(lhs, rhs, rtol=0, atol=1e-13 * np.abs(lhs).max())


@pytest.mark.parametrize("n", [1024, 6000])
def test_impulse_and_tone(n):
    d = np.zeros(n, complex)
    d[0] = 1.0
    assert np.allclose(oracle.dft(d, -1), 1.0, rtol=0, atol=1e-13)
    k0 = n // 3 + 1
    tone = np.exp(2j * np.pi * ((np.arange(n) * k0) % n) / n)
    X = oracle.dft(tone, -1)
    expect = np.zeros(n, complex)
    expect[k0] = n
    assert np.abs(X - expect).max() <= 1e-9 * n
