"""Backprojection over a height map (sarbp_backproject_heights) against the FP64 oracle.

SARBP-GPU §3.3 (the page "基于GPU的SAR后向投影成像优化与CUDA加速实践") notes
that the range history may need the terrain elevation; pixel (ix, iy) sits
at (x0 + ix dx, y0 + iy dy, z0 + h[iy, ix]). Acceptance as for the planar
path (tests/parity.py): relative L2 <= 1e-3, max |error| <= 1e-3 of the
peak, the same argmax at every target.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from domain_backprojection_sarbp_gb300 import Plan, SarbpError, _native  # noqa: E402
from synth import scenes  # noqa: E402
from tests import parity  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
KNIFE = 1e-5     # bins from a half bin within which two nearest samples are both valid


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def _dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=dtype)).to(DEV)


def heights_image(params, echoes, pos, heights, h_range, init=None, accumulate=False, plan=None,
                  interp="linear"):
    img = torch.full((params["ny"], params["nx"]), complex(7.0, -3.0), dtype=torch.complex64,
                     device=DEV)
    if init is not None:
        img.copy_(torch.from_numpy(init.astype(np.complex64)))
    own = plan is None
    plan = plan or Plan(params, height_range=h_range)
    try:
        plan.backproject_heights(img, _dev(echoes, np.complex64), _dev(pos, np.float64),
                                 _dev(heights, np.float32), params=params, accumulate=accumulate,
                                 interp=interp)
        torch.cuda.synchronize()
    finally:
        if own:
            plan.close()
    return img.cpu().numpy()


def terrain_scene(cfg, relief, mean=20.0, noise=True):
    h = scenes.terrain(cfg.nx, cfg.ny, cfg.spacing, cfg.seed + 77, relief=relief, mean=mean)
    return scenes.make_scene(cfg, noise=noise, heights=h), h


# ------------------------------------------------ several tiles, ragged tails
@pytest.mark.parametrize("relief", [10.0, 40.0])
def test_terrain_several_tiles(relief):
    # 100 x 600 pixels: four 32-wide tiles (the last 4 wide) by two 512-high
    # tiles (the last 88 high)
    cfg = scenes.shrink(scenes.CONFIGS[1], na=512, nx=100, ny=600, n_targets=6)
    sc, h = terrain_scene(cfg, relief)
    h_range = (float(h.min()), float(h.max()))
    got = heights_image(sc.params, sc.echoes, sc.antenna_pos, h, h_range)
    ref = oracle.backproject_heights(sc.params, sc.echoes, sc.antenna_pos, h)
    print(parity.assert_parity(got, ref, f"terrain relief {relief}"))
    assert not parity.argmax_mismatches(got, ref, sc.targets)


def two_bin_fraction(params, pos, h, pulses, span=0.9):
    """Share of (thread row of 32 pixels, pulse) pairs whose range index u
    spans less than ``span`` bins: below 0.9 the pixels fall in two adjacent
    bins, the rows the linear path serves from two table entries; the others
    take one gather per pixel."""
    p = params
    ny, nx = h.shape
    xs = p["x0"] + np.arange(nx) * p["dx"]
    ys = p["y0"] + np.arange(ny) * p["dy"]
    px = np.broadcast_to(xs[None, :], (ny, nx))
    py = np.broadcast_to(ys[:, None], (ny, nx))
    pz = p["z0"] + h.astype(np.float64)
    full = (nx // 32) * 32
    spans = []
    for n in pulses:
        u = np.sqrt((px - pos[n, 0]) ** 2 + (py - pos[n, 1]) ** 2 + (pz - pos[n, 2]) ** 2)
        u = ((u - p["r0"]) / p["dr"])[:, :full].reshape(ny, -1, 32)
        spans.append((u.max(axis=2) - u.min(axis=2)).ravel())
    return float((np.concatenate(spans) < span).mean())


@pytest.mark.parametrize("relief", [40.0, 80.0, 240.0])
def test_terrain_two_entry_and_gathered_rows(relief):
    """Terrain where about 60 % (40 m), 40 % (80 m) and 7 % (240 m) of the
    (row, pulse) pairs lie in two range bins (two-entry form) and the rest in
    more (a gather per pixel); all against the oracle in full."""
    cfg = scenes.shrink(scenes.CONFIGS[1], na=384, nx=96, ny=700, n_targets=6)
    sc, h = terrain_scene(cfg, relief, mean=5.0)
    share2 = two_bin_fraction(sc.params, sc.antenna_pos, h, range(0, cfg.na, 48))
    share3 = two_bin_fraction(sc.params, sc.antenna_pos, h, range(0, cfg.na, 48), span=1.9)
    print("two-bin share", share2, "three-bin share", share3)
    assert 0.05 < share2 < share3 < 0.99, (share2, share3)
    got = heights_image(sc.params, sc.echoes, sc.antenna_pos, h, (float(h.min()), float(h.max())))
    ref = oracle.backproject_heights(sc.params, sc.echoes, sc.antenna_pos, h)
    print(parity.assert_parity(got, ref, f"gentle terrain relief {relief}"))
    assert not parity.argmax_mismatches(got, ref, sc.targets)


def assert_nearest_parity(got, ref, p, e, pos, h, label):
    """Nearest sample on a height map: where a pulse's range lies within KNIFE
    bins of a half bin, the float32 and float64 paths may take different
    samples and both are valid; such pixels are held to the sum of
    |e_k - e_k+1| over those pulses, the rest to the usual tolerances."""
    err = np.abs(got - ref).reshape(-1)
    tol = parity.MAX_ERR * np.abs(ref).max()
    explained = []
    for pix in np.nonzero(err > tol)[0]:
        ix, iy = pix % p["nx"], pix // p["nx"]
        pt = np.array([p["x0"] + ix * p["dx"], p["y0"] + iy * p["dy"], p["z0"] + float(h[iy, ix])])
        u = (np.linalg.norm(pos - pt[None, :], axis=1) - p["r0"]) / p["dr"]
        kk = np.floor(u).astype(np.int64)
        knife = (np.abs(u - kk - 0.5) < KNIFE) & (kk >= -1) & (kk <= p["nr"] - 1)
        gap = sum(abs(complex(e[n, kk[n]] if kk[n] >= 0 else 0) -
                      complex(e[n, kk[n] + 1] if kk[n] + 1 <= p["nr"] - 1 else 0))
                  for n in np.nonzero(knife)[0])
        assert err[pix] <= gap + tol, (int(pix), err[pix], gap)
        explained.append(pix)
    keep = np.setdiff1d(np.arange(err.size), np.array(explained, dtype=np.int64))
    m = parity.compare(got.reshape(-1)[keep], ref.reshape(-1)[keep])
    print(label, m, len(explained), "knife-edge pixels")
    assert m["rel_l2"] <= parity.REL_L2 and m["max_err"] <= parity.MAX_ERR, m


# the widest spread of u over a row that the sinc kernel serves with one
# polynomial (degree 6 on seven nodes); below one bin, the two-sample nearest rows
SINC_SPAN6 = 0.80


@pytest.mark.parametrize("interp,relief", [("sinc8", 2.0), ("sinc8", 20.0), ("nearest", 2.0),
                                           ("nearest", 20.0)])
def test_terrain_with_other_interpolations(interp, relief):
    """Windowed sinc and nearest sample on terrain, against the oracle. On 2 m
    of relief every (row, pulse) pair lies within SINC_SPAN6 bins (one
    polynomial per row for sinc, of degree 2 to 6 by the span) and within two
    bins (one table entry per row for nearest); on 20 m about 67 % (sinc)
    and 73 % (nearest) do, the rest take the per-pixel path."""
    cfg = scenes.shrink(scenes.CONFIGS[1], na=512, nx=100, ny=600, n_targets=6)
    sc, h = terrain_scene(cfg, relief)
    span = SINC_SPAN6 if interp == "sinc8" else 0.9
    share = two_bin_fraction(sc.params, sc.antenna_pos, h, range(0, cfg.na, 64), span=span)
    print(interp, relief, "row share", share)
    if relief < 5.0:
        assert share > 0.99, share
    else:
        assert 0.2 < share < 0.9, share
    img = torch.zeros((cfg.ny, cfg.nx), dtype=torch.complex64, device=DEV)
    with Plan(sc.params, height_range=(float(h.min()), float(h.max()))) as plan:
        plan.backproject_heights(img, _dev(sc.echoes, np.complex64), _dev(sc.antenna_pos, np.float64),
                                 _dev(h, np.float32), interp=interp)
        torch.cuda.synchronize()
    got = img.cpu().numpy()
    ref = oracle.backproject_heights(sc.params, sc.echoes, sc.antenna_pos, h, interp=interp)
    if interp == "sinc8":
        print(interp, parity.assert_parity(got, ref, f"terrain {relief} m, sinc8"))
        assert not parity.argmax_mismatches(got, ref, sc.targets)
        return
    assert_nearest_parity(got, ref, sc.params, sc.echoes, sc.antenna_pos, h, interp)


def test_focusing_pin_on_the_gpu():
    """The oracle's focusing pin (targets on a rough surface focus on their
    pixels with the right heights and not on a flat grid), run on this path."""
    from tests.test_oracle_heights_pins import pin_focusing_on_rough_surface

    def gpu_bp(params, echo, pos, h):
        return heights_image(params, echo, pos, h, (float(h.min()), float(h.max())))
    ok, detail = pin_focusing_on_rough_surface(gpu_bp)
    assert ok, detail


def test_constant_height_is_the_raised_plane():
    sc = scenes.make_scene(scenes.CONFIGS[0])
    p = sc.params
    h = np.full((p["ny"], p["nx"]), 7.25, dtype=np.float32)
    got = heights_image(p, sc.echoes, sc.antenna_pos, h, (0.0, 10.0))
    ref = oracle.backproject(dict(p, z0=p["z0"] + 7.25), sc.echoes, sc.antenna_pos)
    parity.assert_parity(got, ref, "constant height")


@pytest.mark.parametrize("interp", ["linear", "sinc8", "nearest"])
def test_wide_height_range(interp):
    """A 500 m height range widens every table row; pixels at both extremes
    still receive every pulse's echo. (The tile reach this range gives sends
    the records to the float64 path; for sinc the terrain cost split prices
    them so.)"""
    cfg = scenes.shrink(scenes.CONFIGS[1], na=256, nx=96, ny=96, n_targets=4)
    base = scenes.terrain(cfg.nx, cfg.ny, cfg.spacing, cfg.seed + 5, relief=4.0, mean=0.0)
    h = base.copy()
    h[:48] += -100.0
    h[48:] += 400.0
    sc = scenes.make_scene(cfg, heights=h)
    got = heights_image(sc.params, sc.echoes, sc.antenna_pos, h, (-110.0, 410.0), interp=interp)
    ref = oracle.backproject_heights(sc.params, sc.echoes, sc.antenna_pos, h, interp=interp)
    if interp == "nearest":
        assert_nearest_parity(got, ref, sc.params, sc.echoes, sc.antenna_pos, h, "wide height range")
    else:
        print(parity.assert_parity(got, ref, f"wide height range, {interp}"))


@pytest.mark.parametrize("interp", ["linear", "sinc8", "nearest"])
def test_near_field_uses_the_exact_rows(interp):
    """Antenna 40-60 m from the pixels: the range series does not apply
    (|t| > 0.01) and every row takes the float64 reference with an exact
    float32 difference per pixel."""
    na, nx, ny = 48, 70, 530
    pos = np.zeros((na, 3))
    pos[:, 0] = np.linspace(-20, 20, na)
    pos[:, 1] = -30.0
    pos[:, 2] = 40.0
    geo = scenes.image_geometry(nx, ny, 0.1)
    p = dict(nx=nx, ny=ny, na=na, nr=512, r0=10.0, dr=0.25, wavelength=scenes.WAVELENGTH, **geo)
    echo = (np.random.default_rng(8).standard_normal((na, 512)) * (1 + 1j)).astype(np.complex64)
    h = scenes.terrain(nx, ny, 0.1, 99, relief=3.0, mean=1.0)
    got = heights_image(p, echo, pos, h, (float(h.min()), float(h.max())), interp=interp)
    ref = oracle.backproject_heights(p, echo, pos, h, interp=interp)
    if interp == "nearest":
        assert_nearest_parity(got, ref, p, echo, pos, h, "near field on terrain")
    else:
        print(parity.assert_parity(got, ref, f"near field on terrain, {interp}"))


def test_heights_are_clamped_to_the_plan_range():
    cfg = scenes.shrink(scenes.CONFIGS[1], na=128, nx=64, ny=80, n_targets=2)
    sc, h = terrain_scene(cfg, 30.0)
    wild = h.copy()
    wild[3, 5] = 1.0e6
    wild[7, 9] = -1.0e6
    wild[11, 13] = np.nan
    wild[2, 40] = np.inf
    lo, hi = 10.0, 25.0
    tame = np.clip(wild, lo, hi)
    tame[11, 13] = lo                     # a NaN height is taken as the lower bound
    with Plan(sc.params, height_range=(lo, hi)) as plan:
        a = heights_image(sc.params, sc.echoes, sc.antenna_pos, wild, None, plan=plan)
        b = heights_image(sc.params, sc.echoes, sc.antenna_pos, tame, None, plan=plan)
    assert np.all(np.isfinite(a))
    assert np.array_equal(a, b)
    ref = oracle.backproject_heights(sc.params, sc.echoes, sc.antenna_pos, tame)
    parity.assert_parity(a, ref, "clamped heights")


@pytest.mark.parametrize("interp", ["linear", "sinc8", "nearest"])
def test_accumulate_and_determinism(interp):
    """Repeated calls give the same bits (for sinc with the terrain cost split,
    which is computed in integers and so the same on every run), and
    accumulation adds the image to what the buffer held."""
    cfg = scenes.shrink(scenes.CONFIGS[1], na=256, nx=70, ny=530, n_targets=3)
    sc, h = terrain_scene(cfg, 20.0)
    rng = np.random.default_rng(3)
    init = (rng.standard_normal((cfg.ny, cfg.nx)) + 1j * rng.standard_normal((cfg.ny, cfg.nx)))
    init = init.astype(np.complex64)
    rng_h = (float(h.min()), float(h.max()))
    with Plan(sc.params, height_range=rng_h) as plan:
        one = heights_image(sc.params, sc.echoes, sc.antenna_pos, h, None, plan=plan, interp=interp)
        two = heights_image(sc.params, sc.echoes, sc.antenna_pos, h, None, plan=plan, interp=interp)
        acc = heights_image(sc.params, sc.echoes, sc.antenna_pos, h, None, init=init,
                            accumulate=True, plan=plan, interp=interp)
    assert np.array_equal(one, two)
    scale = np.abs(one).max()
    assert np.abs(acc - (init + one)).max() <= 1e-5 * scale


# ------------------------------------------- full size, sampled pixels
@pytest.mark.slow
@pytest.mark.parametrize("interp", ["linear", "sinc8"])
def test_page_spotlight_on_terrain_sampled(interp):
    """4096 pulses onto 1024 x 1024 pixels on 40 m of relief, in the launch
    configuration the bench uses (for sinc: polynomial rows of degree 2 to 6,
    per-pixel rows in the steep tiles, the terrain cost split); compared on
    sampled pixels."""
    cfg = scenes.CONFIGS[2]
    sc, h = terrain_scene(cfg, 40.0)
    got = heights_image(sc.params, sc.echoes, sc.antenna_pos, h, (float(h.min()), float(h.max())),
                        interp=interp)
    pix = scenes.compared_pixels(sc)
    ref = oracle.backproject_heights(sc.params, sc.echoes, sc.antenna_pos, h, pixels=pix,
                                     interp=interp)
    print(parity.assert_parity(got.reshape(-1)[pix], ref, f"page_spotlight on terrain, {interp}"))
    full = np.zeros(cfg.nx * cfg.ny, dtype=np.complex128)
    full[pix] = ref
    assert not parity.argmax_mismatches(got, full.reshape(cfg.ny, cfg.nx), sc.targets)


# ------------------------------------------------------------ the interface
def test_plans_do_not_mix():
    sc = scenes.make_scene(scenes.CONFIGS[0])
    p = sc.params
    h = np.zeros((p["ny"], p["nx"]), dtype=np.float32)
    img = torch.zeros((p["ny"], p["nx"]), dtype=torch.complex64, device=DEV)
    e, a, hd = _dev(sc.echoes, np.complex64), _dev(sc.antenna_pos, np.float64), _dev(h, np.float32)
    with Plan(p, height_range=(0.0, 1.0)) as hp, Plan(p) as fp:
        with pytest.raises(SarbpError) as ex:
            hp.backproject(img, e, a)
        assert ex.value.status == _native.SARBP_ERR_PLAN_MISMATCH
        with pytest.raises(SarbpError) as ex:
            hp.backproject_host(np.zeros((p["ny"], p["nx"]), np.complex64), sc.echoes,
                                sc.antenna_pos)
        assert ex.value.status == _native.SARBP_ERR_PLAN_MISMATCH
        with pytest.raises(SarbpError) as ex:
            fp.backproject_heights(img, e, a, hd)
        assert ex.value.status == _native.SARBP_ERR_PLAN_MISMATCH


def test_bad_height_arguments():
    sc = scenes.make_scene(scenes.CONFIGS[0])
    p = sc.params
    lib = _native.lib()
    prm = _native.Params.from_dict(p)
    h = ctypes.c_void_p()
    for lo, hi in ((1.0, 0.0), (float("nan"), 1.0), (0.0, float("inf"))):
        assert lib.sarbp_plan_heights(ctypes.byref(h), ctypes.byref(prm), lo, hi) == \
            _native.SARBP_ERR_INVALID_ARG
        assert not h.value
    img = torch.zeros((p["ny"], p["nx"]), dtype=torch.complex64, device=DEV)
    e, a = _dev(sc.echoes, np.complex64), _dev(sc.antenna_pos, np.float64)
    hd = torch.zeros(p["ny"] * p["nx"] + 1, dtype=torch.float32, device=DEV)
    with Plan(p, height_range=(0.0, 1.0)) as plan:
        # heights that are not 4-byte aligned, and missing heights
        odd = ctypes.c_void_p(hd.data_ptr() + 2)
        for ptr in (odd, ctypes.c_void_p(None)):
            st = lib.sarbp_backproject_heights(
                plan.handle, ctypes.c_void_p(img.data_ptr()), ctypes.c_void_p(e.data_ptr()),
                ctypes.c_void_p(a.data_ptr()), ptr, ctypes.byref(prm), None)
            assert st == _native.SARBP_ERR_INVALID_ARG
        with pytest.raises(SarbpError):
            plan.backproject_heights(img, e, a, hd[:-1].reshape(p["ny"], p["nx"]),
                                     params=dict(p, flags=_native.SARBP_NEAREST | _native.SARBP_SINC8))
