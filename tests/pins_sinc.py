"""Pins for the 8-tap windowed-sinc oracle (SARBP-GPU §2.2: sinc interpolation).

The kernel is h(t) = sinc(t) (1/2 + 1/2 cos(2 pi t / 8)) over the stencil
k-3 .. k+4; its values used below follow from that formula by hand:
h(0) = 1, h(integer != 0) = 0, h(1/2) = (2/pi)(1 + cos(pi/8))/2,
h(-5/2) = (2/(5 pi))(1 + cos(5 pi/8))/2. Geometry as in hand_cases.json:
lambda = 1/32 m, dr = 1/64 m, r0 = 999.83984375 m, so ranges and phases are exact.
"""

from __future__ import annotations

import math

import numpy as np

from synth import scenes
from tests import pins

R0, DR, LAM, NR = 999.83984375, 0.015625, 0.03125, 16


def _one_pulse(u, samples):
    """Single pixel at the origin, antenna straight above at range r0 + u dr."""
    params = dict(nx=1, ny=1, na=1, nr=NR, x0=0.0, y0=0.0, z0=0.0, dx=1.0, dy=1.0,
                  r0=R0, dr=DR, wavelength=LAM)
    pos = np.array([[0.0, 0.0, R0 + u * DR]])
    echo = np.zeros((1, NR), dtype=np.complex64)
    for k, v in samples.items():
        echo[0, k] = v
    phase_turns = (2.0 * (R0 + u * DR) / LAM) % 1.0          # exact on this dyadic grid
    return params, echo, pos, np.exp(2j * np.pi * phase_turns)


def pin_sinc_on_sample(bp):
    """u = 10: every tap but the centre sits on a zero of sinc; the value is e[10]."""
    poison = {m: complex(3 * (m + 1), 5 * (m + 1)) for m in range(NR)}
    poison[10] = 1 + 2j
    params, echo, pos, rot = _one_pulse(10.0, poison)
    got = bp(params, echo, pos, np.array([0]))[0]
    want = (1 + 2j) * rot
    return abs(got - want) < 1e-9, f"got {got}, want {want}"


def pin_sinc_half_sample(bp):
    """u = 10.5 with a single nonzero sample at 6, 7, 10, 11, 13 or 14.

    The stencil is 7 .. 14: samples 7 and 14 sit at t = +-3.5, where
    h = -(2/(7 pi)) (1 + cos(7 pi/8)) / 2; sample 6 is outside and gets weight 0.
    """
    h_half = (2 / math.pi) * (1 + math.cos(math.pi / 8)) / 2
    h_m25 = (2 / (5 * math.pi)) * (1 + math.cos(5 * math.pi / 8)) / 2
    h_35 = -(2 / (7 * math.pi)) * (1 + math.cos(7 * math.pi / 8)) / 2
    bad = []
    for k, h in ((10, h_half), (11, h_half), (13, h_m25), (7, h_35), (14, h_35), (6, 0.0)):
        params, echo, pos, rot = _one_pulse(10.5, {k: 1.0 + 0j})
        got = bp(params, echo, pos, np.array([0]))[0]
        if abs(got - h * rot) > 1e-9:
            bad.append(f"sample {k}: got {got}, want {h * rot}")
    return (not bad), "; ".join(bad)


def pin_sinc_window_rule(bp):
    """The whole stencil k-3 .. k+4 must lie in 0 .. nr-1."""
    ones = {m: 1.0 + 0j for m in range(NR)}
    bad = []
    for u, inside in ((2.5, False), (3.5, True), (11.5, True), (12.5, False)):
        params, echo, pos, _ = _one_pulse(u, ones)
        got = bp(params, echo, pos, np.array([0]))[0]
        if (got != 0) != inside:
            bad.append(f"u={u}: got {got}")
    return (not bad), "; ".join(bad)


def pin_sinc_fine_target(bp):
    """Isolated noiseless target on 0.2 m bins (5x oversampled): the sinc-interpolated
    echo at the target's own range is 1, and the phases cancel, so I = a Na, real."""
    na, amp = 64, 0.7
    params, _, pos, txyz, _ = pins.single_target_scene(na=na, nx=8, ny=8, target=(4, 4))
    dr = 0.2
    nr = 4096
    r0 = float(np.linalg.norm(pos[na // 2] - txyz)) - (nr // 2) * dr
    params = dict(params, dr=dr, nr=nr, r0=r0)
    echo = scenes.simulate_echoes(pos, txyz[None, :], np.array([amp]), r0, dr, nr).astype(np.complex64)
    got = bp(params, echo, pos, np.array([4 * 8 + 4]))[0]
    want = amp * na
    ok = abs(got - want) < 1e-3 * want
    return ok, f"got {got}, want {want}"


SINC_PINS = [pin_sinc_on_sample, pin_sinc_half_sample, pin_sinc_window_rule, pin_sinc_fine_target,
             pins.pin_zero_echo, pins.pin_linearity, pins.pin_pulse_permutation,
             pins.pin_focusing, pins.pin_mirror_symmetry]
