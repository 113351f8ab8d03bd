"""libsarbp (CUDA, sm_103a) against the FP64 oracle, through the C-ABI.

Acceptance (tests/parity.py): relative L2 <= 1e-3, max |error| <= 1e-3 of the
oracle's peak, identical per-target argmax. SARBP-GPU §4.2 (the page
"基于GPU的SAR后向投影成像优化与CUDA加速实践") asks for the same check: run the
same backprojection on CPU and GPU over simulated point targets and compare.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from domain_backprojection_sarbp_gb300 import Plan, SarbpError, _native  # noqa: E402
from synth import scenes  # noqa: E402
from tests import parity, pins  # noqa: E402

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def gpu_image(params, echoes, pos, plan=None, accumulate=False, init=None, stream=None,
              interp="linear"):
    p = dict(params)
    e = torch.from_numpy(np.ascontiguousarray(echoes, dtype=np.complex64)).to(DEV)
    a = torch.from_numpy(np.ascontiguousarray(pos, dtype=np.float64)).to(DEV)
    img = torch.full((p["ny"], p["nx"]), complex(7.0, -3.0), dtype=torch.complex64, device=DEV)
    if init is not None:
        img.copy_(torch.from_numpy(init.astype(np.complex64)))
    own = plan is None
    plan = plan or Plan(p)
    try:
        plan.backproject(img, e, a, params=p, accumulate=accumulate, stream=stream, interp=interp)
        torch.cuda.synchronize()
    finally:
        if own:
            plan.close()
    return img.cpu().numpy()


# ---------------------------------------------------------------- hand values
@pytest.mark.parametrize("case", [c for c in pins.load_hand_cases() if c[0] != "first_bin"],
                         ids=lambda c: c[0])
def test_hand_cases(case):
    # "first_bin" sits exactly on u = 0, the edge of the window rule, where a
    # float32 range one ulp low flips the value to zero; it stays an oracle pin.
    name, params, echo, pos, pix, expected = case
    img = gpu_image(params, echo, pos).reshape(-1)
    got = img[pix]
    assert np.allclose(got, expected, rtol=0, atol=2e-4 * max(1.0, np.abs(expected).max())), \
        f"{name}: {got} vs {expected}"


# ---------------------------------------------------------------- the configs
def _check_scene(sc, img):
    pix = scenes.compared_pixels(sc)
    ref = oracle.backproject(sc.params, sc.echoes, sc.antenna_pos, pix)
    got = img.reshape(-1)[pix]
    m = parity.assert_parity(got, ref, sc.cfg.name)
    nx, ny = sc.params["nx"], sc.params["ny"]
    ref_img = np.zeros(nx * ny, dtype=np.complex128)
    ref_img[pix] = ref
    bad = parity.argmax_mismatches(img, ref_img.reshape(ny, nx), sc.targets)
    assert not bad, f"{sc.cfg.name}: argmax differs at {bad}"
    return m


@pytest.mark.parametrize("index", [1, 2])
def test_config_full_image(index):
    sc = scenes.make_scene(scenes.CONFIGS[index - 1])
    img = gpu_image(sc.params, sc.echoes, sc.antenna_pos)
    m = _check_scene(sc, img)
    print(sc.cfg.name, m)


@pytest.mark.slow
@pytest.mark.parametrize("index", [3, 4, 5])
def test_config_full_size_sampled(index):
    sc = scenes.make_scene(scenes.CONFIGS[index - 1])
    img = gpu_image(sc.params, sc.echoes, sc.antenna_pos)
    assert np.all(np.isfinite(img))
    m = _check_scene(sc, img)
    print(sc.cfg.name, m)


@pytest.mark.slow
def test_page_scene_every_pixel():
    """The benchmark's scene compared at all 1,048,576 pixels (4.3e9 updates of
    the oracle, a few seconds on the host's cores), not only a sample."""
    sc = scenes.make_scene(scenes.CONFIGS[2])
    img = gpu_image(sc.params, sc.echoes, sc.antenna_pos)
    ref = oracle.backproject(sc.params, sc.echoes, sc.antenna_pos)
    print(sc.cfg.name, "all pixels", parity.assert_parity(img, ref, "page scene, every pixel"))
    assert not parity.argmax_mismatches(img, ref, sc.targets)


# ---------------------------------------------------------------- edge cases
def _small_scene(nx, ny, na=40, nr=512, spacing=0.5, step=0.5, seed=5, noise=0.05):
    cfg = scenes.shrink(scenes.CONFIGS[0], nx=nx, ny=ny, na=na, nr=nr, spacing=spacing,
                        pulse_step=step, n_targets=0, noise_sigma=noise)
    return scenes.make_scene(cfg, seed=seed)


@pytest.mark.parametrize("shape", [(37, 201), (1, 1), (3, 2), (33, 129), (200, 7)])
def test_ragged_and_tiny_images(shape):
    sc = _small_scene(*shape)
    img = gpu_image(sc.params, sc.echoes, sc.antenna_pos)
    ref = oracle.backproject(sc.params, sc.echoes, sc.antenna_pos)
    parity.assert_parity(img, ref, f"shape {shape}")


@pytest.mark.slow
def test_maximum_image_size():
    """The largest image a plan accepts, 2^30 pixels (32768 x 32768, 8 GiB on the
    device), 16 pulses of clutter; sampled pixels against the oracle. One pixel
    more is refused."""
    nx = ny = 32768
    na, nr = 16, 4096
    spacing = 0.05
    rng = np.random.default_rng(30)
    pos = scenes.straight_track(na, 1.0)
    geo = scenes.image_geometry(nx, ny, spacing)
    corner = np.array([geo["x0"], geo["y0"] + ny * spacing, 0.0])
    rmin = float(np.min(np.linalg.norm(pos - np.array([0.0, geo["y0"], 0.0]), axis=1))) - 50.0
    p = dict(nx=nx, ny=ny, na=na, nr=nr, r0=rmin, dr=scenes.DR, wavelength=scenes.WAVELENGTH, **geo)
    assert float(np.max(np.linalg.norm(pos - corner, axis=1))) < rmin + (nr - 2) * scenes.DR
    echo = (rng.standard_normal((na, nr)) + 1j * rng.standard_normal((na, nr))).astype(np.complex64)
    img = torch.empty((ny, nx), dtype=torch.complex64, device=DEV)
    with Plan(p) as plan:
        plan.backproject(img, torch.from_numpy(echo).to(DEV), torch.from_numpy(pos).to(DEV))
        torch.cuda.synchronize()
    pix = np.unique(np.concatenate([rng.choice(nx * ny, 4000, replace=False),
                                    [0, nx - 1, nx * ny - nx, nx * ny - 1]])).astype(np.int64)
    got = img.reshape(-1)[torch.from_numpy(pix).to(DEV)].cpu().numpy()
    del img
    ref = oracle.backproject(p, echo, pos, pix)
    parity.assert_parity(got, ref, "2^30 pixels")
    with pytest.raises(SarbpError) as ex:
        Plan(dict(p, ny=ny + 1))
    assert ex.value.status == _native.SARBP_ERR_INVALID_ARG


@pytest.mark.parametrize("field,value", [("na", 0), ("nr", 0), ("nr", 1)])
def test_no_contribution_gives_zero(field, value):
    sc = _small_scene(40, 20)
    p = dict(sc.params, **{field: value})
    echo = sc.echoes[:p["na"], :p["nr"]]
    pos = sc.antenna_pos[:p["na"]]
    img = gpu_image(p, echo, pos)
    assert np.all(img == 0)
    init = np.full((20, 40), 2 + 1j)
    img = gpu_image(p, echo, pos, accumulate=True, init=init)
    assert np.all(img == init.astype(np.complex64))


def test_empty_image():
    sc = _small_scene(40, 20)
    p = dict(sc.params, nx=0)
    with Plan(p) as plan:
        e = torch.from_numpy(sc.echoes).to(DEV)
        a = torch.from_numpy(sc.antenna_pos).to(DEV)
        img = torch.empty((20, 0), dtype=torch.complex64, device=DEV)
        plan.backproject(img, e, a)
        torch.cuda.synchronize()


def test_accumulate_pulse_batches():
    sc = _small_scene(70, 150, na=96)
    half = 40
    p1 = dict(sc.params, na=half)
    p2 = dict(sc.params, na=sc.params["na"] - half)
    first = gpu_image(p1, sc.echoes[:half], sc.antenna_pos[:half])
    both = gpu_image(p2, sc.echoes[half:], sc.antenna_pos[half:], accumulate=True, init=first)
    ref = oracle.backproject(sc.params, sc.echoes, sc.antenna_pos)
    parity.assert_parity(both, ref, "two batches")


@pytest.mark.parametrize("interp", ["linear", "sinc8"])
def test_bitwise_deterministic(interp):
    """Same inputs, same bits: the pulse sum has a fixed order, and the sinc
    call's cost-weighted work split is computed in integers."""
    sc = scenes.make_scene(scenes.shrink(scenes.CONFIGS[1], na=300, nx=300, ny=260, nr=2048))
    with Plan(sc.params) as plan:
        a = gpu_image(sc.params, sc.echoes, sc.antenna_pos, plan=plan, interp=interp)
        b = gpu_image(sc.params, sc.echoes, sc.antenna_pos, plan=plan, interp=interp)
    assert np.array_equal(a.view(np.uint64), b.view(np.uint64))


def test_nan_guard_bands_untouched():
    sc = _small_scene(64, 130, na=50)
    na, nr = sc.echoes.shape
    guard = 4096
    flat = torch.full((na * nr + 2 * guard,), complex(float("nan"), float("nan")),
                      dtype=torch.complex64, device=DEV)
    flat[guard:guard + na * nr] = torch.from_numpy(sc.echoes.reshape(-1)).to(DEV)
    echoes = flat[guard:guard + na * nr].view(na, nr)
    pos = torch.from_numpy(sc.antenna_pos).to(DEV)
    img = torch.zeros((sc.params["ny"], sc.params["nx"]), dtype=torch.complex64, device=DEV)
    with Plan(sc.params) as plan:
        plan.backproject(img, echoes, pos)
        torch.cuda.synchronize()
    got = img.cpu().numpy()
    assert np.all(np.isfinite(got))
    parity.assert_parity(got, oracle.backproject(sc.params, sc.echoes, sc.antenna_pos), "guards")


@pytest.mark.parametrize("interp", ["linear", "sinc8", "nearest"])
def test_unreachable_nonfinite_samples_are_ignored(interp):
    """Samples more than 8 bins outside the ranges a pulse can reach from the
    image (nearest and farthest point of the image rectangle) are set to NaN
    and infinity: the image must be the clean one bit for bit."""
    sc = scenes.make_scene(scenes.CONFIGS[1])
    p = sc.params
    xa, xb = p["x0"], p["x0"] + (p["nx"] - 1) * p["dx"]
    ya, yb = p["y0"], p["y0"] + (p["ny"] - 1) * p["dy"]
    dirty = sc.echoes.copy()
    k = np.arange(p["nr"])
    for n, (ax, ay, az) in enumerate(sc.antenna_pos):
        dz = p["z0"] - az
        rmin = np.sqrt((np.clip(ax, xa, xb) - ax) ** 2 + (np.clip(ay, ya, yb) - ay) ** 2 + dz * dz)
        rmax = np.sqrt(max(abs(xa - ax), abs(xb - ax)) ** 2 + max(abs(ya - ay), abs(yb - ay)) ** 2
                       + dz * dz)
        lo = np.floor((rmin - p["r0"]) / p["dr"]) - 8
        hi = np.floor((rmax - p["r0"]) / p["dr"]) + 9
        out = (k < lo) | (k > hi)
        dirty[n, out & (k % 2 == 0)] = complex(np.nan, np.nan)
        dirty[n, out & (k % 2 == 1)] = complex(np.inf, -np.inf)
    assert np.isnan(dirty).sum() > dirty.size // 4
    clean = gpu_image(p, sc.echoes, sc.antenna_pos, interp=interp)
    got = gpu_image(p, dirty, sc.antenna_pos, interp=interp)
    assert np.array_equal(got, clean), interp


def test_range_window_edges_full_window():
    # a short range axis that the image overruns at both ends: every rule of
    # the window (k < 0, k + 1 > nr - 1) is exercised, and the table spans the
    # whole axis
    sc = _small_scene(96, 300, na=24, nr=48, spacing=0.5, noise=0.3)
    p = dict(sc.params)
    centre = np.linalg.norm(sc.antenna_pos[12])
    p["r0"] = centre - 20 * p["dr"]
    with Plan(p) as plan:
        assert plan.describe()["full_window"] == 1
        img = gpu_image(p, sc.echoes, sc.antenna_pos, plan=plan)
    ref = oracle.backproject(p, sc.echoes, sc.antenna_pos)
    assert np.any(ref == 0) and np.any(ref != 0)
    parity.assert_parity(img, ref, "window edges")


@pytest.mark.parametrize("interp", ["linear", "sinc8"])
def test_non_finite_antenna_position_skips_pulse(interp):
    """Pulses with a non-finite antenna position contribute nothing (for sinc
    they also carry no weight in the work split)."""
    sc = _small_scene(40, 130, na=30)
    pos = sc.antenna_pos.copy()
    pos[7, 1] = np.nan
    pos[19, 2] = np.inf
    img = gpu_image(sc.params, sc.echoes, pos, interp=interp)
    ref = oracle.backproject(sc.params, sc.echoes, pos, interp=interp)
    assert np.all(np.isfinite(img))
    parity.assert_parity(img, ref, "non-finite antenna " + interp)


def test_sinc_all_antenna_positions_non_finite():
    """No finite pulse at all: the sinc work split has zero total cost and
    falls back to the equal split; the image is zero."""
    sc = _small_scene(40, 130, na=30)
    pos = np.full_like(sc.antenna_pos, np.nan)
    img = gpu_image(sc.params, sc.echoes, pos, interp="sinc8")
    assert np.array_equal(img, np.zeros_like(img))


def test_near_field_exact_path():
    # antenna 40 m above a 32 m wide scene: the Taylor remainder is far above
    # the fast-path bound, so every (tile, pulse) takes the exact path
    na, nx, ny = 48, 64, 130
    pos = np.zeros((na, 3))
    pos[:, 0] = np.linspace(-20, 20, na)
    pos[:, 1] = -30.0
    pos[:, 2] = 40.0
    geo = scenes.image_geometry(nx, ny, 0.25)
    nr = 256
    r0 = 20.0
    p = dict(nx=nx, ny=ny, na=na, nr=nr, r0=r0, dr=0.5, wavelength=scenes.WAVELENGTH, **geo)
    txyz = np.array([[geo["x0"] + 20 * 0.25, geo["y0"] + 70 * 0.25, 0.0]])
    echo = scenes.simulate_echoes(pos, txyz, np.array([1.0]), r0, 0.5, nr).astype(np.complex64)
    echo += (np.random.default_rng(2).standard_normal(echo.shape) * 0.05).astype(np.complex64)
    img = gpu_image(p, echo, pos)
    ref = oracle.backproject(p, echo, pos)
    parity.assert_parity(img, ref, "near field")


def test_host_entry_point_matches_device():
    sc = _small_scene(64, 200, na=64)
    with Plan(sc.params) as plan:
        dev_img = gpu_image(sc.params, sc.echoes, sc.antenna_pos, plan=plan)
        host_img = np.zeros((sc.params["ny"], sc.params["nx"]), dtype=np.complex64)
        plan.backproject_host(host_img, sc.echoes, sc.antenna_pos)
        parity.assert_parity(host_img, dev_img, "host entry point")
        parity.assert_parity(host_img, oracle.backproject(sc.params, sc.echoes, sc.antenna_pos),
                             "host entry point vs oracle")
        h2d, d2h = plan.host_transfer_bytes()
        # only the band of bins the image reaches is copied, not all 512 per pulse
        assert h2d < sc.echoes.nbytes // 2 and d2h == host_img.nbytes
        again = host_img.copy()
        plan.backproject_host(again, sc.echoes, sc.antenna_pos, accumulate=True)
        parity.assert_parity(again, 2 * host_img.astype(np.complex128), "host accumulate")


def test_host_entry_point_at_range_axis_edges():
    sc = _small_scene(96, 300, na=24, nr=48, spacing=0.5, noise=0.3)
    p = dict(sc.params)
    p["r0"] = np.linalg.norm(sc.antenna_pos[12]) - 20 * p["dr"]
    with Plan(p) as plan:
        img = np.zeros((p["ny"], p["nx"]), dtype=np.complex64)
        plan.backproject_host(img, sc.echoes, sc.antenna_pos, params=p)
    parity.assert_parity(img, oracle.backproject(p, sc.echoes, sc.antenna_pos), "host, axis edges")


def test_host_entry_point_no_reachable_bin():
    sc = _small_scene(40, 20, na=8)
    p = dict(sc.params, r0=sc.params["r0"] + 1.0e5)      # every range is below the axis
    with Plan(p) as plan:
        img = np.full((20, 40), 3 + 3j, dtype=np.complex64)
        plan.backproject_host(img, sc.echoes, sc.antenna_pos, params=p)
        assert np.all(img == 0)
        assert plan.host_transfer_bytes()[0] == sc.antenna_pos.nbytes


def test_non_default_stream():
    sc = _small_scene(64, 130, na=40)
    s = torch.cuda.Stream()
    img = gpu_image(sc.params, sc.echoes, sc.antenna_pos, stream=s)
    parity.assert_parity(img, oracle.backproject(sc.params, sc.echoes, sc.antenna_pos), "stream")


def test_timing_api_counts_launches():
    sc = _small_scene(64, 130, na=40)
    with Plan(sc.params) as plan:
        plan.set_timing(True)
        for _ in range(3):
            gpu_image(sc.params, sc.echoes, sc.antenna_pos, plan=plan)
        ms, n = plan.kernel_times()
        assert n == 3 and ms > 0
        assert plan.kernel_times() == (0.0, 0)


def test_plan_mismatch_and_alignment_errors():
    sc = _small_scene(64, 130, na=40)
    with Plan(sc.params) as plan:
        e = torch.from_numpy(sc.echoes).to(DEV)
        a = torch.from_numpy(sc.antenna_pos).to(DEV)
        img = torch.zeros((130, 64), dtype=torch.complex64, device=DEV)
        with pytest.raises(SarbpError) as ei:
            plan.backproject(img[:, :32].contiguous(), e, a, params=dict(sc.params, nx=32))
        assert ei.value.status == _native.SARBP_ERR_PLAN_MISMATCH
        p = _native.Params.from_dict(sc.params)
        raw = torch.zeros(64 * 130 * 2 + 1, dtype=torch.float32, device=DEV)
        st = _native.lib().sarbp_backproject(plan.handle, ctypes.c_void_p(raw.data_ptr() + 4),
                                             ctypes.c_void_p(e.data_ptr()),
                                             ctypes.c_void_p(a.data_ptr()), ctypes.byref(p), None)
        assert st == _native.SARBP_ERR_INVALID_ARG
        torch.cuda.synchronize()
