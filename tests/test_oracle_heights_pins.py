"""The non-planar-grid oracle against facts fixed outside itself (no GPU needed).

SARBP-GPU §3.3 (the page "基于GPU的SAR后向投影成像优化与CUDA加速实践") notes that
the range history may need terrain elevation. Pixel (ix, iy) sits at
(x0 + ix dx, y0 + iy dy, z0 + h[iy, ix]).
"""

import os
import shutil

import numpy as np
import pytest

import oracle
from synth import scenes
from tests import pins


def _scene():
    return pins.single_target_scene(na=48, nx=14, ny=11)


def pin_zero_heights_reduce_to_planar(bp):
    params, echo, pos, _, _ = _scene()
    h = np.zeros((params["ny"], params["nx"]), dtype=np.float32)
    ok = np.array_equal(bp(params, echo, pos, h), oracle.backproject(params, echo, pos))
    return ok, "zero heights differ from the planar grid"


def pin_constant_height_is_a_shifted_plane(bp):
    params, echo, pos, _, _ = _scene()
    h = np.full((params["ny"], params["nx"]), 7.25, dtype=np.float32)
    want = oracle.backproject(dict(params, z0=params["z0"] + 7.25), echo, pos)
    return np.array_equal(bp(params, echo, pos, h), want), "constant height != raised plane"


def pin_hand_raised_pixel(bp):
    """pixel_mapping of hand_cases.json raised by 3 m, antenna raised by 3 m: R = 1000."""
    case = [c for c in pins.load_hand_cases() if c[0] == "pixel_mapping"][0]
    _, params, echo, pos, pix, expected = case
    h = np.zeros((params["ny"], params["nx"]), dtype=np.float32)
    h.reshape(-1)[pix] = 3.0
    h.reshape(-1)[0] = -11.0                      # other pixels move elsewhere
    got = bp(params, echo, pos + np.array([0.0, 0.0, 3.0]), h)
    ok = abs(got.reshape(-1)[pix][0] - expected[0]) < 1e-9
    return ok, f"got {got.reshape(-1)[pix]}, want {expected}"


def pin_focusing_on_rough_surface(bp):
    """Targets on a rough surface focus on their pixels with the right heights,
    and away from them on a flat grid (a 25 m height error moves the image of a
    target by about 25 * 5000 / 7000 m in ground range)."""
    nx = ny = 96
    spacing = 0.5
    cfg = scenes.shrink(scenes.CONFIGS[1], na=256, nx=nx, ny=ny, nr=4096, spacing=spacing,
                        pulse_step=200.0 / 256, n_targets=3)
    sc = scenes.make_scene(cfg, noise=False)
    yy, xx = np.mgrid[0:ny, 0:nx]
    h = (25.0 + 10.0 * np.sin(xx / 13.0) * np.cos(yy / 17.0)).astype(np.float32)
    dr = 0.1
    r0 = float(np.linalg.norm(sc.antenna_pos[cfg.na // 2])) - (cfg.nr // 2) * dr
    params = dict(sc.params, r0=r0, dr=dr)
    txyz = np.zeros((len(sc.targets), 3))
    txyz[:, 0] = params["x0"] + sc.targets[:, 0] * spacing
    txyz[:, 1] = params["y0"] + sc.targets[:, 1] * spacing
    txyz[:, 2] = h[sc.targets[:, 1], sc.targets[:, 0]]
    echo = scenes.simulate_echoes(sc.antenna_pos, txyz, sc.amps, r0, dr, cfg.nr).astype(np.complex64)
    right = np.abs(bp(params, echo, sc.antenna_pos, h))
    flat = np.abs(bp(params, echo, sc.antenna_pos, np.zeros_like(h)))
    bad = []
    for ix, iy in sc.targets:
        w = right[iy - 4:iy + 5, ix - 4:ix + 5]
        if np.unravel_index(np.argmax(w), w.shape) != (4, 4):
            bad.append(f"({ix},{iy}) not focused")
        if flat[iy, ix] > 0.5 * right[iy, ix]:
            bad.append(f"({ix},{iy}) still focused on the flat grid")
    return (not bad), "; ".join(bad)


HEIGHT_PINS = [pin_zero_heights_reduce_to_planar, pin_constant_height_is_a_shifted_plane,
               pin_hand_raised_pixel, pin_focusing_on_rough_surface]


def _bp(params, echo, pos, heights, library=None):
    return oracle.backproject_heights(params, echo, pos, heights, library=library)


@pytest.mark.parametrize("pin", HEIGHT_PINS, ids=lambda p: p.__name__)
def test_height_pin(pin):
    ok, detail = pin(_bp)
    assert ok, detail


@pytest.mark.parametrize("interp", ["sinc8", "nearest"])
def test_interpolation_variants_reduce_to_the_planar_ones(interp):
    """Zero heights give the planar variant bit for bit; a constant height gives
    the planar variant on the raised plane; a mixed map gives each pixel the
    planar value of its own height."""
    params, echo, pos, _, _ = _scene()
    ny, nx = params["ny"], params["nx"]
    zero = np.zeros((ny, nx), dtype=np.float32)
    assert np.array_equal(oracle.backproject_heights(params, echo, pos, zero, interp=interp),
                          oracle.backproject(params, echo, pos, interp=interp))
    const = np.full((ny, nx), 7.25, dtype=np.float32)
    assert np.array_equal(oracle.backproject_heights(params, echo, pos, const, interp=interp),
                          oracle.backproject(dict(params, z0=params["z0"] + 7.25), echo, pos,
                                             interp=interp))
    mixed = np.where((np.arange(ny)[:, None] + np.arange(nx)[None, :]) % 2 == 0, 0.0, 3.5)
    mixed = mixed.astype(np.float32)
    got = oracle.backproject_heights(params, echo, pos, mixed, interp=interp)
    raised = oracle.backproject(dict(params, z0=params["z0"] + 3.5), echo, pos, interp=interp)
    flat = oracle.backproject(params, echo, pos, interp=interp)
    assert np.array_equal(got, np.where(mixed == 0, flat, raised))


SRC = os.path.join(os.path.dirname(oracle.__file__), "sarbp_oracle.c")
HDR = os.path.join(os.path.dirname(oracle.__file__), "sarbp_oracle.h")
MUTATIONS = {
    "heights_ignored": [("raised.z0 = g->z0 + (double)heights[pixel];", "raised.z0 = g->z0;")],
    "heights_negated": [("raised.z0 = g->z0 + (double)heights[pixel];",
                         "raised.z0 = g->z0 - (double)heights[pixel];")],
    "heights_transposed": [("raised.z0 = g->z0 + (double)heights[pixel];",
                            "raised.z0 = g->z0 + (double)heights[(pixel % g->nx) * g->ny + pixel / g->nx];")],
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_height_mutation_is_caught(tmp_path, name):
    src = open(SRC).read()
    for old, new in MUTATIONS[name]:
        assert src.count(old) == 1, f"mutation {name}: text not found"
        src = src.replace(old, new)
    (tmp_path / "sarbp_oracle.c").write_text(src)
    shutil.copy(HDR, tmp_path / "sarbp_oracle.h")
    lib = oracle.load_library(oracle.compile_library(src=str(tmp_path / "sarbp_oracle.c"),
                                                     out=str(tmp_path / "m.so")))
    failed = [p.__name__ for p in HEIGHT_PINS
              if not p(lambda *a: _bp(*a, library=lib))[0]]
    assert failed, f"no pin rejects the planted mistake '{name}'"
