"""The windowed-sinc oracle against facts fixed outside itself (no GPU needed)."""

import os
import shutil

import pytest

import oracle
from tests import pins_sinc


def _bp(params, echo, pos, pixels=None):
    return oracle.backproject(params, echo, pos, pixels, interp="sinc8")


@pytest.mark.parametrize("pin", pins_sinc.SINC_PINS, ids=lambda p: p.__name__)
def test_sinc_pin(pin):
    ok, detail = pin(_bp)
    assert ok, detail


SRC = os.path.join(os.path.dirname(oracle.__file__), "sarbp_oracle.c")
HDR = os.path.join(os.path.dirname(oracle.__file__), "sarbp_oracle.h")

MUTATIONS = {
    "stencil_shifted": [("for (int64_t m = kk - 3; m <= kk + 4; ++m)",
                         "for (int64_t m = kk - 4; m <= kk + 3; ++m)")],
    "tap_dropped": [("for (int64_t m = kk - 3; m <= kk + 4; ++m)",
                     "for (int64_t m = kk - 3; m <= kk + 3; ++m)")],
    "window_too_narrow": [("cos(2.0 * ORACLE_PI * t / 8.0)", "cos(2.0 * ORACLE_PI * t / 4.0)")],
    "window_dropped": [("const double window = 0.5 + 0.5 * cos(2.0 * ORACLE_PI * t / 8.0);",
                        "const double window = 1.0;")],
    "sinc_unnormalised": [("sin(ORACLE_PI * t) / (ORACLE_PI * t)", "sin(t) / t")],
    "window_rule_loose": [("k - 3.0 >= 0.0 && k + 4.0 <= (double)(g->nr - 1)",
                           "k - 2.0 >= 0.0 && k + 4.0 <= (double)(g->nr - 1)")],
    "sinc_phase_sign": [("acc_im += w_re * s + w_im * c;\n    }\n    out[0] = acc_re;\n    out[1] = acc_im;\n}\n\n/* One pixel, all pulses, nearest",
                         "acc_im += -w_re * s + w_im * c;\n    }\n    out[0] = acc_re;\n    out[1] = acc_im;\n}\n\n/* One pixel, all pulses, nearest")],
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_sinc_mutation_is_caught(tmp_path, name):
    src = open(SRC).read()
    for old, new in MUTATIONS[name]:
        assert src.count(old) >= 1, f"mutation {name}: text not found"
        src = src.replace(old, new, 1)
    (tmp_path / "sarbp_oracle.c").write_text(src)
    shutil.copy(HDR, tmp_path / "sarbp_oracle.h")
    so = oracle.compile_library(src=str(tmp_path / "sarbp_oracle.c"), out=str(tmp_path / "m.so"))
    lib = oracle.load_library(so)

    def bp(params, echo, pos, pixels=None):
        return oracle.backproject(params, echo, pos, pixels, library=lib, interp="sinc8")

    failed = [p.__name__ for p in pins_sinc.SINC_PINS if not p(bp)[0]]
    assert failed, f"no pin rejects the planted mistake '{name}'"
