"""The seeded scene generator (input generation only, no backprojection)."""

import numpy as np

from synth import scenes


def _small(**kw):
    base = dict(na=48, nr=512, nx=64, ny=64, n_targets=3)
    base.update(kw)
    return scenes.shrink(scenes.CONFIGS[0], **base)


def test_seeded_determinism():
    a = scenes.make_scene(_small())
    b = scenes.make_scene(_small())
    assert np.array_equal(a.echoes, b.echoes)
    assert np.array_equal(a.antenna_pos, b.antenna_pos)
    assert np.array_equal(a.targets, b.targets)
    c = scenes.make_scene(_small(), seed=99)
    assert not np.array_equal(a.echoes, c.echoes)


def test_targets_on_grid_spaced_and_inside():
    sc = scenes.make_scene(scenes.shrink(scenes.CONFIGS[1], na=4, nr=64, n_targets=16))
    t = sc.targets
    assert t.shape == (16, 2)
    assert t.min() >= scenes.TARGET_BORDER
    assert t[:, 0].max() < sc.params["nx"] - scenes.TARGET_BORDER
    for i in range(len(t)):
        for j in range(i):
            assert np.abs(t[i] - t[j]).max() >= scenes.TARGET_SPACING


def test_echo_peak_in_nearest_bin_and_support():
    pos = scenes.straight_track(5, 1.0)
    txyz = np.array([[3.0, -2.0, 0.0]])
    r0, dr, nr = 8500.0, scenes.DR, 512
    e = scenes.simulate_echoes(pos, txyz, np.array([1.0]), r0, dr, nr)
    for n in range(5):
        rng = np.linalg.norm(pos[n] - txyz[0])
        k_near = int(np.round((rng - r0) / dr))
        assert np.argmax(np.abs(e[n])) == k_near
        nz = np.nonzero(e[n])[0]
        rk = r0 + nz * dr
        assert np.all(np.abs(rk - rng) <= 16 * scenes.RHO + 1e-9)
        # every bin within the support is present
        k_all = np.arange(nr)
        inside = np.abs(r0 + k_all * dr - rng) <= 16 * scenes.RHO
        assert np.array_equal(np.nonzero(inside)[0], nz)
        # phase of the echo is -4 pi R / lambda at the peak bin (sinc > 0 there)
        ph = np.angle(e[n, k_near] * np.exp(1j * 4 * np.pi * rng / scenes.WAVELENGTH))
        assert abs(ph) < 1e-9


def test_noise_power():
    cfg = _small(n_targets=0 if False else 1, noise_sigma=0.5, na=256, nr=1024)
    sc = scenes.make_scene(cfg)
    clean = scenes.make_scene(cfg, noise=False)
    n = (sc.echoes - clean.echoes).astype(np.complex128)
    assert abs(np.mean(np.abs(n) ** 2) / 0.25 - 1) < 0.02
    assert abs(np.var(n.real) / np.var(n.imag) - 1) < 0.03


def test_motion_bounded():
    sc = scenes.make_scene(scenes.shrink(scenes.CONFIGS[4], na=512, nr=64, nx=64, ny=64,
                                         n_targets=1))
    straight = scenes.straight_track(512, 0.1)
    d = sc.antenna_pos - straight
    assert np.abs(d).max() <= 0.5
    assert np.abs(d).max() > 0.01


def test_range_window_centred():
    sc = scenes.make_scene(_small())
    p = sc.params
    r_mid = np.linalg.norm(sc.antenna_pos[p["na"] // 2])
    assert abs(p["r0"] + (p["nr"] // 2) * p["dr"] - r_mid) < 1e-9


def test_compared_pixels():
    cfg = scenes.shrink(scenes.CONFIGS[2], na=4, nr=64)
    sc = scenes.make_scene(cfg, noise=False)
    pix = scenes.compared_pixels(sc)
    assert np.all(np.diff(pix) > 0)
    for ix, iy in sc.targets:
        assert iy * cfg.nx + ix in set(pix.tolist())
    assert len(pix) >= 4096
