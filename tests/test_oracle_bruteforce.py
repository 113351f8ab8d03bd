"""Marshalling check: the compiled oracle against a direct Python loop on a tiny grid.

This re-types the definition, so it is not one of the pins (tests/pins.py holds
those); it only shows that the C library receives what the caller means.
"""

import math

import numpy as np

import oracle
from tests import pins


def _python_loop(p, echo, pos):
    img = np.zeros((p["ny"], p["nx"]), dtype=np.complex128)
    for iy in range(p["ny"]):
        for ix in range(p["nx"]):
            x, y, z = p["x0"] + ix * p["dx"], p["y0"] + iy * p["dy"], p["z0"]
            acc = 0j
            for n in range(p["na"]):
                r = math.sqrt((x - pos[n, 0]) ** 2 + (y - pos[n, 1]) ** 2 + (z - pos[n, 2]) ** 2)
                u = (r - p["r0"]) / p["dr"]
                k = math.floor(u)
                if k < 0 or k + 1 > p["nr"] - 1:
                    continue
                f = u - k
                w = (1 - f) * complex(echo[n, k]) + f * complex(echo[n, k + 1])
                acc += w * complex(math.cos(4 * math.pi * r / p["wavelength"]),
                                   math.sin(4 * math.pi * r / p["wavelength"]))
            img[iy, ix] = acc
    return img


def test_bruteforce_tiny():
    params, echo, pos, _, _ = pins.single_target_scene(na=16, nx=12, ny=9)
    rng = np.random.default_rng(1)
    echo = echo + (rng.standard_normal(echo.shape) * 0.1).astype(np.complex64)
    got = oracle.backproject(params, echo, pos)
    want = _python_loop(params, echo, pos)
    assert np.abs(got - want).max() <= 1e-12 * np.abs(want).max()
