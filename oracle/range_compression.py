"""Plain FP64 range compression (matched filtering). TEST INFRASTRUCTURE ONLY.

SARBP-GPU §3.1 (the page "基于GPU的SAR后向投影成像优化与CUDA加速实践"): FFT each
pulse along range, multiply by the matched filter's frequency response, apply a
Hamming (or Taylor) window in the frequency domain to lower the sidelobes,
inverse FFT; the FFTs of all pulses form one batch.

Definition used here (reading of the page's steps):
    rc[n][k] = sum_{l=0}^{L-1} raw[n][k + l] * conj(ref[l]),   0 <= k < ns,
with raw taken as zero beyond its last sample, i.e. the linear
cross-correlation, computed as ifft(fft(raw, N) * conj(fft(ref, N)) * W)[:ns]
with N the smallest power of two >= ns + L - 1 (no circular wrap). W = 1, or
the Hamming weighting 0.54 + 0.46 cos(2 pi f / b) over the centred band
|f| <= b/2 (f = signed frequency in cycles per sample, b = band fraction) and
0 outside it. numpy's FFT is a library step of that definition.

Pinned by: the direct correlation sum on small sizes (brute force), the
closed-form peak a * sum |ref|^2 at an integer delay, shift equivariance,
linearity, and the sidelobe / mainlobe figures the page quotes (about -13 dB
peak sidelobe without a window; Hamming widens the mainlobe 1.3-1.5x)
(tests/test_range_compression_oracle.py).
"""

from __future__ import annotations

import numpy as np


def fft_size(ns: int, nref: int) -> int:
    n = 1
    while n < ns + nref - 1:
        n *= 2
    return n


def window_weights(n: int, window: str = "none", band_fraction: float = 1.0) -> np.ndarray:
    f = np.fft.fftfreq(n)                      # signed cycles per sample
    if window == "none":
        return np.ones(n)
    if window == "hamming":
        inside = np.abs(f) <= band_fraction / 2.0
        return np.where(inside, 0.54 + 0.46 * np.cos(2.0 * np.pi * f / band_fraction), 0.0)
    raise ValueError(window)


def range_compress(raw: np.ndarray, ref: np.ndarray, window: str = "none",
                   band_fraction: float = 1.0) -> np.ndarray:
    """complex128 [na, ns] from raw [na, ns] and reference chirp [L]."""
    raw = np.asarray(raw, dtype=np.complex128)
    ref = np.asarray(ref, dtype=np.complex128)
    na, ns = raw.shape
    n = fft_size(ns, ref.size)
    h = np.conj(np.fft.fft(ref, n)) * window_weights(n, window, band_fraction)
    spec = np.fft.fft(raw, n, axis=1) * h[None, :]
    return np.fft.ifft(spec, axis=1)[:, :ns]


def direct_correlation(raw: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """The definition as a plain double loop (small sizes only)."""
    raw = np.asarray(raw, dtype=np.complex128)
    ref = np.asarray(ref, dtype=np.complex128)
    na, ns = raw.shape
    out = np.zeros((na, ns), dtype=np.complex128)
    for n in range(na):
        for k in range(ns):
            acc = 0j
            for l in range(ref.size):
                if k + l < ns:
                    acc += raw[n, k + l] * np.conj(ref[l])
            out[n, k] = acc
    return out
