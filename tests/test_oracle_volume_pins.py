"""The voxel-grid oracle against three-dimensional focusing (no GPU needed).

SARBP-GPU §3.3 (the page "基于GPU的SAR后向投影成像优化与CUDA加速实践") notes that
the pixel grid may leave the ground plane; a voxel grid is a stack of planes
z0 + iz dz. With a single straight pass the height of a target is not
resolved (every point of a circle about the track has the same range
history); with passes stacked vertically (a two-dimensional aperture) it is,
to about lambda R / (2 B_perp). Targets on grid voxels, noiseless echoes on
fine range bins: the magnitude peaks at each target's voxel, and a volume
made from one pass only does not separate the heights.
"""

import numpy as np

import oracle
from synth import scenes


def _scene(passes, baseline=40.0):
    nx = ny = 24
    nz, dz, spacing = 7, 0.5, 0.5
    na_pass = 48
    pos = scenes.multipass_track(na_pass, passes, 2.0, baseline)
    geo = scenes.image_geometry(nx, ny, spacing)
    geo["z0"] = -1.5
    vox = np.array([[6, 8, 1], [15, 14, 3], [10, 18, 5]])        # (ix, iy, iz)
    txyz = np.stack([geo["x0"] + vox[:, 0] * spacing, geo["y0"] + vox[:, 1] * spacing,
                     geo["z0"] + vox[:, 2] * dz], axis=1).astype(np.float64)
    dr, nr = 0.1, 2048
    r0 = float(np.linalg.norm(pos[len(pos) // 2])) - (nr // 2) * dr
    echo = scenes.simulate_echoes(pos, txyz, np.ones(len(vox)), r0, dr, nr).astype(np.complex64)
    params = dict(nx=nx, ny=ny, na=len(pos), nr=nr, r0=r0, dr=dr,
                  wavelength=scenes.WAVELENGTH, **geo)
    return params, echo, pos, vox, nz, dz


def test_volume_is_a_stack_of_planes():
    params, echo, pos, _, nz, dz = _scene(passes=3)
    vol = oracle.backproject_volume(params, echo, pos, nz, dz)
    assert vol.shape == (nz, params["ny"], params["nx"])
    for iz in (0, nz - 1):
        plane = oracle.backproject(dict(params, z0=params["z0"] + iz * dz), echo, pos)
        assert np.array_equal(vol[iz], plane)


def pin_focus(bpv):
    params, echo, pos, vox, nz, dz = _scene(passes=10)
    mag = np.abs(bpv(params, echo, pos, nz, dz))
    bad = []
    for ix, iy, iz in vox:
        w = mag[:, iy - 3:iy + 4, ix - 3:ix + 4]
        got = np.unravel_index(np.argmax(w), w.shape)
        if got != (iz, 3, 3):
            bad.append(((ix, iy, iz), got))
    return not bad, bad


def test_targets_focus_at_their_voxels_with_a_vertical_aperture():
    ok, bad = pin_focus(oracle.backproject_volume)
    assert ok, bad


def _planes(params, echo, pos, heights):
    return np.stack([oracle.backproject(dict(params, z0=h), echo, pos) for h in heights])


MISTAKES = {
    "planes_reversed": lambda p, e, a, nz, dz: _planes(p, e, a, [p["z0"] + (nz - 1 - i) * dz for i in range(nz)]),
    "dz_sign": lambda p, e, a, nz, dz: _planes(p, e, a, [p["z0"] - i * dz for i in range(nz)]),
    "dz_ignored": lambda p, e, a, nz, dz: _planes(p, e, a, [p["z0"]] * nz),
    "half_dz": lambda p, e, a, nz, dz: _planes(p, e, a, [p["z0"] + 0.5 * i * dz for i in range(nz)]),
}


def test_focus_pin_rejects_plausible_mistakes():
    for name, bpv in MISTAKES.items():
        assert not pin_focus(bpv)[0], f"the focusing pin accepts '{name}'"


def test_one_pass_does_not_resolve_height():
    params, echo, pos, vox, nz, dz = _scene(passes=1)
    mag = np.abs(oracle.backproject_volume(params, echo, pos, nz, dz))
    # along the layover circle the focus moves with height: the peak over each
    # plane's neighbourhood stays within 10 % of the best plane's for every height
    ix, iy, iz = vox[1]
    best = [mag[z, iy - 6:iy + 7, ix - 6:ix + 7].max() for z in range(nz)]
    assert min(best) > 0.9 * max(best)
