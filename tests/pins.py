"""Checks that pin the FP64 oracle to facts fixed outside itself.

Each check takes a backprojection callable ``bp(params, echoes, antenna_pos,
pixels=None)`` and returns ``(ok, detail)``. The same checks run against the
real oracle (they must all pass) and against copies of the oracle with a
planted mistake (at least one must fail), so a pin that cannot see a plausible
error is noticed.

SARBP-GPU = the page "基于GPU的SAR后向投影成像优化与CUDA加速实践".
"""

from __future__ import annotations

import json
import os

import numpy as np

from synth import scenes

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_cases.json")


def load_hand_cases():
    with open(GOLDEN) as fh:
        doc = json.load(fh)
    common = doc["common"]
    out = []
    for case in doc["cases"]:
        pos = np.array(case["antenna_pos"], dtype=np.float64)
        na, nr = pos.shape[0], common["nr"]
        echo = np.full((na, nr), complex(*common["poison"]), dtype=np.complex64)
        for n, k, re, im in case["samples"]:
            echo[n, k] = complex(re, im)
        params = dict(case["geometry"], na=na, nr=nr, r0=common["r0"], dr=common["dr"],
                      wavelength=common["wavelength"])
        expected = np.array([complex(re, im) for re, im in case["expected"]])
        out.append((case["name"], params, echo, pos, np.array(case["pixels"]), expected))
    return out


def pin_hand_cases(bp):
    """Hand-derived values (tests/golden/hand_cases.json), SARBP-GPU §1.1, §2.2, §3.3."""
    bad = []
    for name, params, echo, pos, pix, expected in load_hand_cases():
        got = bp(params, echo, pos, pix)
        if not np.allclose(got, expected, rtol=0, atol=1e-9):
            bad.append(f"{name}: got {got}, want {expected}")
    return (not bad), "; ".join(bad)


def closed_form_peak(params, pos, target_xyz, amp, rho=scenes.RHO):
    """Value at an isolated on-grid target with a noiseless sinc echo.

    The echo is a*sinc((r_k - R_n)/rho)*exp(-j 4 pi R_n / lambda); the phase
    compensation exp(+j 4 pi R_n / lambda) cancels it exactly, so the pixel value
    is real: a * sum_n [(1 - f_n) sinc((r_k - R_n)/rho) + f_n sinc((r_{k+1} - R_n)/rho)].
    """
    d = pos - target_xyz[None, :]
    rng = np.sqrt(np.sum(d * d, axis=1))
    u = (rng - params["r0"]) / params["dr"]
    k = np.floor(u)
    f = u - k
    rk = params["r0"] + k * params["dr"]
    lo = np.sinc((rk - rng) / rho)
    hi = np.sinc((rk + params["dr"] - rng) / rho)
    return amp * np.sum((1.0 - f) * lo + f * hi)


def single_target_scene(na=96, nx=24, ny=20, spacing=0.5, step=0.5, target=(11, 9), amp=0.8):
    """A noiseless one-target spotlight scene on the page-style geometry (SARBP-GPU §3.2)."""
    pos = scenes.straight_track(na, step)
    geo = scenes.image_geometry(nx, ny, spacing)
    nr = 512
    r_mid = float(np.linalg.norm(pos[na // 2]))
    r0 = r_mid - (nr // 2) * scenes.DR
    params = dict(nx=nx, ny=ny, na=na, nr=nr, r0=r0, dr=scenes.DR,
                  wavelength=scenes.WAVELENGTH, **geo)
    txyz = np.array([[geo["x0"] + target[0] * spacing, geo["y0"] + target[1] * spacing, 0.0]])
    echo = scenes.simulate_echoes(pos, txyz, np.array([amp]), r0, scenes.DR, nr).astype(np.complex64)
    return params, echo, pos, txyz[0], amp


def pin_closed_form(bp, tol=1e-6):
    """Isolated target: value equals a * sum L_n and is real (SARBP-GPU §1.1, §4.2)."""
    params, echo, pos, txyz, amp = single_target_scene()
    pix = np.array([9 * params["nx"] + 11])
    got = bp(params, echo, pos, pix)[0]
    want = closed_form_peak(params, pos, txyz, amp)
    ok = abs(got - want) <= tol * abs(want) and abs(got.imag) <= tol * abs(want)
    return ok, f"got {got}, closed form {want}"


def pin_zero_echo(bp):
    """No echo energy gives an exactly zero image."""
    params, echo, pos, _, _ = single_target_scene()
    got = bp(params, np.zeros_like(echo), pos, None)
    return bool(np.all(got == 0)), f"max |I| = {np.abs(got).max()}"


def pin_linearity(bp, tol=1e-12):
    """BP(2 E1 + j E2) = 2 BP(E1) + j BP(E2); inputs chosen so the combination is exact in complex64."""
    params, _, pos, _, _ = single_target_scene(nx=10, ny=8)
    rng = np.random.default_rng(7)
    shape = (params["na"], params["nr"])
    e1 = (rng.integers(-512, 512, shape) + 1j * rng.integers(-512, 512, shape)) / 1024.0
    e2 = (rng.integers(-512, 512, shape) + 1j * rng.integers(-512, 512, shape)) / 1024.0
    e1, e2 = e1.astype(np.complex64), e2.astype(np.complex64)
    mix = (2 * e1.astype(np.complex128) + 1j * e2.astype(np.complex128)).astype(np.complex64)
    lhs = bp(params, mix, pos, None)
    rhs = 2 * bp(params, e1, pos, None) + 1j * bp(params, e2, pos, None)
    err = np.abs(lhs - rhs).max() / max(np.abs(rhs).max(), 1e-300)
    return err < tol, f"relative difference {err:.3e}"


def pin_pulse_permutation(bp, tol=1e-12):
    """The sum over pulses does not depend on their order."""
    params, echo, pos, _, _ = single_target_scene(nx=10, ny=8)
    perm = np.random.default_rng(3).permutation(params["na"])
    a = bp(params, echo, pos, None)
    b = bp(params, echo[perm], pos[perm], None)
    err = np.abs(a - b).max() / np.abs(a).max()
    return err < tol, f"relative difference {err:.3e}"


def pin_focusing(bp):
    """Noiseless on-grid targets focus exactly at their own pixel (SARBP-GPU §3.2, §4.2).

    Range bins are 0.1 m here: with bins much wider than a pixel, a linearly
    interpolated sinc peaks at a sample rather than at the true range, which moves
    the range peak by up to half a bin. Fine bins remove that bias, so an error in
    geometry, wavelength or phase sign is what would move the peak.
    """
    cfg = scenes.shrink(scenes.CONFIGS[1], na=256, nx=128, ny=128, nr=4096,
                        pulse_step=200.0 / 256, n_targets=4)
    sc = scenes.make_scene(cfg, noise=False)
    dr = 0.1
    r0 = float(np.linalg.norm(sc.antenna_pos[cfg.na // 2])) - (cfg.nr // 2) * dr
    params = dict(sc.params, r0=r0, dr=dr)
    txyz = np.zeros((len(sc.targets), 3))
    txyz[:, 0] = params["x0"] + sc.targets[:, 0] * params["dx"]
    txyz[:, 1] = params["y0"] + sc.targets[:, 1] * params["dy"]
    echo = scenes.simulate_echoes(sc.antenna_pos, txyz, sc.amps, r0, dr,
                                  cfg.nr).astype(np.complex64)
    img = np.abs(bp(params, echo, sc.antenna_pos, None))
    bad = []
    for ix, iy in sc.targets:
        win = img[iy - 4:iy + 5, ix - 4:ix + 5]
        jy, jx = np.unravel_index(np.argmax(win), win.shape)
        if (jx - 4, jy - 4) != (0, 0):
            bad.append(f"target ({ix},{iy}) peaks at offset ({jx - 4},{jy - 4})")
    return (not bad), "; ".join(bad)


def pin_mirror_symmetry(bp, tol=1e-10):
    """Target at the scene centre under a symmetric straight track: |I| is even in x."""
    # image_geometry puts pixel (10, 4) of a 21 x 9 grid on the origin and
    # straight_track is symmetric about x = 0 (pulse n mirrors pulse na-1-n)
    params, echo, pos, _, _ = single_target_scene(na=64, nx=21, ny=9, target=(10, 4))
    img = np.abs(bp(params, echo, pos, None))
    err = np.abs(img - img[:, ::-1]).max() / img.max()
    return err < tol, f"relative asymmetry {err:.3e}"


def pin_resolution(bp):
    """Point response width near the textbook values (loose, SARBP-GPU §4.2).

    Range (ground y): 0.886 rho / sin(look) with sin(look) = 7000/R.
    Azimuth (x): 0.886 lambda R / (2 L) for a synthetic aperture of length L.
    Linear interpolation and the discrete aperture widen both a little; +-30 %.
    """
    na, step, spacing = 512, 0.5, 0.05
    params, echo, pos, txyz, amp = single_target_scene(na=na, nx=161, ny=161, spacing=spacing,
                                                       step=step, target=(80, 80))
    img = np.abs(bp(params, echo, pos, None))
    peak = img[80, 80]

    def width(profile):
        above = np.nonzero(profile >= peak / np.sqrt(2.0))[0]
        return (above.max() - above.min() + 1) * spacing

    r = float(np.linalg.norm(pos[na // 2] - txyz))
    want_y = 0.886 * scenes.RHO / (scenes.GROUND_OFFSET / r)
    want_x = 0.886 * scenes.WAVELENGTH * r / (2.0 * na * step)
    wy, wx = width(img[:, 80]), width(img[80, :])
    ok = abs(wy / want_y - 1) < 0.3 and abs(wx / want_x - 1) < 0.3
    return ok, f"range width {wy:.3f} m (textbook {want_y:.3f}), azimuth {wx:.3f} m ({want_x:.3f})"


ALL_PINS = [pin_hand_cases, pin_closed_form, pin_zero_echo, pin_linearity,
            pin_pulse_permutation, pin_focusing, pin_mirror_symmetry, pin_resolution]
