"""Planted mistakes in a copy of the oracle must each be caught by a pin.

Each case edits one expression of oracle/sarbp_oracle.c in a temporary copy,
compiles it with gcc, and runs every pin in tests/pins.py against it. A pin
set that let any of these through would not be pinning what it claims to.
All of this runs on the CPU; the real oracle source is never modified.
"""

import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from tests import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "sarbp_oracle.c")
HDR = os.path.join(os.path.dirname(oracle.__file__), "sarbp_oracle.h")

MUTATIONS = {
    "phase_sign": [("acc_re += w_re * c - w_im * s;", "acc_re += w_re * c + w_im * s;"),
                   ("acc_im += w_re * s + w_im * c;", "acc_im += -w_re * s + w_im * c;")],
    "two_pi_not_four_pi": [("4.0 * ORACLE_PI", "2.0 * ORACLE_PI")],
    "wavelength_multiplied": [("range / g->wavelength", "range * g->wavelength")],
    "lerp_weights_swapped": [("(1.0 - f) * (double)e0[0] + f * (double)e1[0]",
                              "f * (double)e0[0] + (1.0 - f) * (double)e1[0]"),
                             ("(1.0 - f) * (double)e0[1] + f * (double)e1[1]",
                              "f * (double)e0[1] + (1.0 - f) * (double)e1[1]")],
    "round_not_floor": [("floor(u)", "round(u)")],
    "bin_spacing_multiplied": [("(range - g->r0) / g->dr", "(range - g->r0) * g->dr")],
    "first_bin_dropped": [("k >= 0.0 &&", "k >= 1.0 &&")],
    "last_bin_dropped": [("k + 1.0 <= (double)(g->nr - 1)", "k + 1.0 < (double)(g->nr - 1)")],
    "pixel_axes_swapped": [("const int64_t ix = pixel % g->nx;", "const int64_t ix = pixel / g->nx;"),
                           ("const int64_t iy = pixel / g->nx;", "const int64_t iy = pixel % g->nx;")],
    "x_difference_sign": [("x - a[0]", "x + a[0]")],
    "height_ignored": [("const double z = g->z0;", "const double z = 0.0;")],
    "last_pulse_dropped": [("n < g->na;", "n + 1 < g->na;")],
    "imag_part_dropped": [("(1.0 - f) * (double)e0[1] + f * (double)e1[1]", "0.0")],
    "cos_for_sin": [("const double s = sin(phase);", "const double s = cos(phase);")],
    "next_sample_wrong": [("const float* e1 = e0 + 2;", "const float* e1 = e0;")],
}


def _compile(tmp_path, name, edits):
    src = open(SRC).read()
    for old, new in edits:
        assert src.count(old) >= 1, f"mutation {name}: '{old}' not in the oracle source"
        src = src.replace(old, new)
    d = tmp_path / name
    d.mkdir()
    (d / "sarbp_oracle.c").write_text(src)
    shutil.copy(HDR, d / "sarbp_oracle.h")
    out = str(d / "libmut.so")
    oracle.compile_library(src=str(d / "sarbp_oracle.c"), out=out)
    return oracle.load_library(out)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(tmp_path, name):
    lib = _compile(tmp_path, name, MUTATIONS[name])

    def bp(params, echo, pos, pixels=None):
        return oracle.backproject(params, echo, pos, pixels, library=lib)

    failed = []
    for pin in pins.ALL_PINS:
        ok, _ = pin(bp)
        if not ok:
            failed.append(pin.__name__)
    assert failed, f"no pin rejects the planted mistake '{name}'"


def test_unmutated_copy_passes(tmp_path):
    lib = _compile(tmp_path, "identity", [])

    def bp(params, echo, pos, pixels=None):
        return oracle.backproject(params, echo, pos, pixels, library=lib)

    for pin in pins.ALL_PINS:
        ok, detail = pin(bp)
        assert ok, f"{pin.__name__}: {detail}"
