"""The FP64 oracle against facts fixed outside itself (no GPU needed)."""

import numpy as np
import pytest

import oracle
from tests import pins


def _bp(params, echo, pos, pixels=None):
    return oracle.backproject(params, echo, pos, pixels)


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    ok, detail = pin(_bp)
    assert ok, detail


def test_threads_do_not_change_result():
    params, echo, pos, _, _ = pins.single_target_scene(nx=13, ny=7)
    a = oracle.backproject(params, echo, pos, None, threads=1)
    b = oracle.backproject(params, echo, pos, None, threads=5)
    assert np.array_equal(a, b)


def test_pixel_subset_matches_full_image():
    params, echo, pos, _, _ = pins.single_target_scene(nx=13, ny=7)
    full = oracle.backproject(params, echo, pos, None)
    pix = np.array([0, 5, 44, 90])
    sub = oracle.backproject(params, echo, pos, pix)
    assert np.array_equal(sub, full.reshape(-1)[pix])


def test_rejects_bad_pixel_index():
    params, echo, pos, _, _ = pins.single_target_scene(nx=4, ny=4)
    with pytest.raises(ValueError):
        oracle.backproject(params, echo, pos, np.array([16]))


def test_no_pulses_gives_zero():
    params, echo, pos, _, _ = pins.single_target_scene(nx=4, ny=4)
    p = dict(params, na=0)
    img = oracle.backproject(p, echo[:0], pos[:0], None)
    assert np.all(img == 0)
