"""Raw (uncompressed) SAR echoes: linear-FM pulses from point targets.

SARBP-GPU §3.1 (the page "基于GPU的SAR后向投影成像优化与CUDA加速实践"): the
backprojection input is produced by range compression of raw echoes with a
matched filter. This module makes the raw side: a transmitted baseband chirp
s(t) = exp(j pi K (t - T/2)^2), 0 <= t < T, K = B / T (frequency sweeping
-B/2 .. B/2), sampled at the range-bin rate
dt = 2 dr / c, and echoes a * s(t - tau) * exp(-j 4 pi R / lambda) delayed by
tau = (R - r0) * 2 / c. Input generation only.
"""

from __future__ import annotations

import numpy as np

from .scenes import C_LIGHT, DR, WAVELENGTH

BANDWIDTH = 150e6          # Hz (rho = c / 2B = 0.999 m)
PULSE_LENGTH = 2e-6        # s


def chirp(bandwidth: float = BANDWIDTH, pulse_length: float = PULSE_LENGTH,
          dr: float = DR) -> np.ndarray:
    """Reference chirp sampled at the range-bin rate (complex128)."""
    dt = 2.0 * dr / C_LIGHT
    n = int(np.floor(pulse_length / dt))
    t = np.arange(n) * dt - pulse_length / 2.0
    k = bandwidth / pulse_length
    return np.exp(1j * np.pi * k * t * t)


def raw_echoes(antenna_pos: np.ndarray, target_xyz: np.ndarray, amps: np.ndarray, r0: float,
               ns: int, dr: float = DR, wavelength: float = WAVELENGTH,
               bandwidth: float = BANDWIDTH, pulse_length: float = PULSE_LENGTH) -> np.ndarray:
    """Raw echoes (complex128 [na, ns]): every target's delayed chirp with its carrier phase."""
    na = antenna_pos.shape[0]
    dt = 2.0 * dr / C_LIGHT
    kk = bandwidth / pulse_length
    out = np.zeros((na, ns), dtype=np.complex128)
    t = np.arange(ns) * dt
    for j in range(target_xyz.shape[0]):
        rng = np.linalg.norm(antenna_pos - target_xyz[j][None, :], axis=1)   # [na]
        tau = 2.0 * (rng - r0) / C_LIGHT
        tl = t[None, :] - tau[:, None]
        inside = (tl >= 0.0) & (tl < pulse_length)
        tc = tl - pulse_length / 2.0
        ph = np.pi * kk * tc * tc - 4.0 * np.pi * rng[:, None] / wavelength
        out += np.where(inside, amps[j] * np.exp(1j * ph), 0.0)
    return out
