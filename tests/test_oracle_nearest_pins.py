"""The nearest-neighbour oracle against facts fixed outside itself (no GPU needed).

SARBP-GPU §2.2 lists nearest-neighbour interpolation as the fastest and least
accurate choice. Values below follow by hand from k = floor(u + 1/2) on the
dyadic geometry of hand_cases.json (exact ranges and phases).
"""

import os
import shutil

import numpy as np
import pytest

import oracle
from tests import pins, pins_sinc


def _bp(params, echo, pos, pixels=None, library=None):
    return oracle.backproject(params, echo, pos, pixels, interp="nearest", library=library)


def pin_nearest_rounding(bp):
    """u = 10.25 and 10.49 take sample 10; u = 10.5 and 10.75 take sample 11."""
    samples = {m: complex(m + 1, -(m + 2)) for m in range(pins_sinc.NR)}
    bad = []
    for u, k in ((10.25, 10), (10.5, 11), (10.75, 11), (10.0, 10)):
        params, echo, pos, rot = pins_sinc._one_pulse(u, samples)
        got = bp(params, echo, pos, np.array([0]))[0]
        want = samples[k] * rot
        if abs(got - want) > 1e-9:
            bad.append(f"u={u}: got {got}, want {want}")
    return (not bad), "; ".join(bad)


def pin_nearest_window(bp):
    """Sample 0 is reached from u >= -0.5, sample nr-1 until u < nr - 0.5."""
    ones = {m: 1.0 + 0j for m in range(pins_sinc.NR)}
    bad = []
    for u, inside in ((-0.75, False), (-0.5, True), (15.25, True), (15.5, False)):
        params, echo, pos, _ = pins_sinc._one_pulse(u, ones)
        got = bp(params, echo, pos, np.array([0]))[0]
        if (got != 0) != inside:
            bad.append(f"u={u}: got {got}")
    return (not bad), "; ".join(bad)


NEAREST_PINS = [pin_nearest_rounding, pin_nearest_window, pins.pin_zero_echo, pins.pin_linearity,
                pins.pin_pulse_permutation, pins.pin_mirror_symmetry]


@pytest.mark.parametrize("pin", NEAREST_PINS, ids=lambda p: p.__name__)
def test_nearest_pin(pin):
    ok, detail = pin(_bp)
    assert ok, detail


SRC = os.path.join(os.path.dirname(oracle.__file__), "sarbp_oracle.c")
HDR = os.path.join(os.path.dirname(oracle.__file__), "sarbp_oracle.h")
MUTATIONS = {
    "floor_not_round": [("const double k = floor(u + 0.5);", "const double k = floor(u);")],
    "ceil_rounding": [("const double k = floor(u + 0.5);", "const double k = ceil(u - 0.5);")],
    "last_sample_dropped": [("k <= (double)(g->nr - 1)))\n            continue;                      /* nearest",
                             "k < (double)(g->nr - 1)))\n            continue;                      /* nearest")],
    "imag_ignored": [("acc_re += (double)e[0] * c - (double)e[1] * s;", "acc_re += (double)e[0] * c;")],
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_nearest_mutation_is_caught(tmp_path, name):
    src = open(SRC).read()
    for old, new in MUTATIONS[name]:
        assert src.count(old) >= 1, f"mutation {name}: text not found"
        src = src.replace(old, new, 1)
    (tmp_path / "sarbp_oracle.c").write_text(src)
    shutil.copy(HDR, tmp_path / "sarbp_oracle.h")
    lib = oracle.load_library(oracle.compile_library(src=str(tmp_path / "sarbp_oracle.c"),
                                                     out=str(tmp_path / "m.so")))

    def bp(params, echo, pos, pixels=None):
        return _bp(params, echo, pos, pixels, library=lib)

    failed = [p.__name__ for p in NEAREST_PINS if not p(bp)[0]]
    assert failed, f"no pin rejects the planted mistake '{name}'"
