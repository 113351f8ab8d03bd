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
a weighting over the centred band |f| <= b/2 (f = signed frequency in cycles
per sample, b = band fraction) and 0 outside it: Hamming
0.54 + 0.46 cos(2 pi f / b), or Taylor (nbar = 5, 35 dB sidelobes)
1 + 2 sum_m F_m cos(2 pi m f / b) with Taylor's coefficients F_m. numpy's FFT
is a library step of that definition.

Pinned by: the direct correlation sum on small sizes (brute force), the
closed-form peak a * sum |ref|^2 at an integer delay, shift equivariance,
linearity, and the sidelobe / mainlobe figures the page quotes (about -13 dB
peak sidelobe without a window; Hamming widens the mainlobe 1.3-1.5x), and for
the Taylor weighting its design sidelobe level, its unit mean over the band
and a mainlobe between those of no window and Hamming
(tests/test_range_compression_oracle.py).
"""

from __future__ import annotations

import numpy as np


def fft_size(ns: int, nref: int) -> int:
    n = 1
    while n < ns + nref - 1:
        n *= 2
    return n


TAYLOR_NBAR = 5          # terms kept (Taylor's n-bar; 35 dB needs nbar >= 2 A^2 + 1/2 = 5)
TAYLOR_SLL_DB = 35.0     # design sidelobe level below the peak


def taylor_coefficients(nbar: int = TAYLOR_NBAR, sll_db: float = TAYLOR_SLL_DB) -> np.ndarray:
    """F_1 .. F_(nbar-1) of Taylor's weighting w(x) = 1 + 2 sum F_m cos(2 pi m x).

    With A = acosh(10^(sll/20)) / pi and the stretch sigma^2 = nbar^2 / (A^2 + (nbar - 1/2)^2),
    F_m = (-1)^(m+1) prod_i (1 - m^2 / (sigma^2 (A^2 + (i - 1/2)^2)))
          / (2 prod_(i != m) (1 - m^2 / i^2)),  i, m = 1 .. nbar - 1.
    """
    a = np.arccosh(10.0 ** (sll_db / 20.0)) / np.pi
    sigma2 = nbar ** 2 / (a ** 2 + (nbar - 0.5) ** 2)
    out = np.zeros(nbar - 1)
    for m in range(1, nbar):
        num = 1.0
        den = 1.0
        for i in range(1, nbar):
            num *= 1.0 - m ** 2 / (sigma2 * (a ** 2 + (i - 0.5) ** 2))
            if i != m:
                den *= 1.0 - m ** 2 / i ** 2
        out[m - 1] = (-1.0) ** (m + 1) * num / (2.0 * den)
    return out


def window_weights(n: int, window: str = "none", band_fraction: float = 1.0) -> np.ndarray:
    f = np.fft.fftfreq(n)                      # signed cycles per sample
    if window == "none":
        return np.ones(n)
    inside = np.abs(f) <= band_fraction / 2.0
    x = f / band_fraction
    if window == "hamming":
        return np.where(inside, 0.54 + 0.46 * np.cos(2.0 * np.pi * x), 0.0)
    if window == "taylor":
        w = np.ones(n)
        for m, fm in enumerate(taylor_coefficients(), start=1):
            w += 2.0 * fm * np.cos(2.0 * np.pi * m * x)
        return np.where(inside, w, 0.0)
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
