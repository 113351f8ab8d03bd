"""Windowed-sinc interpolation (SARBP_SINC8) against the FP64 sinc oracle.

SARBP-GPU §2.2 (the page "基于GPU的SAR后向投影成像优化与CUDA加速实践") names sinc
interpolation as the more accurate alternative to linear; same acceptance as
the linear path: relative L2 <= 1e-3, max |error| <= 1e-3 of the peak,
identical per-target argmax.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from domain_backprojection_sarbp_gb300 import Plan, _native  # noqa: E402
from synth import scenes  # noqa: E402
from tests import parity  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def sinc_image(params, echoes, pos):
    e = torch.from_numpy(np.ascontiguousarray(echoes, dtype=np.complex64)).to(DEV)
    a = torch.from_numpy(np.ascontiguousarray(pos, dtype=np.float64)).to(DEV)
    img = torch.full((params["ny"], params["nx"]), complex(7.0, -3.0), dtype=torch.complex64,
                     device=DEV)
    with Plan(params) as plan:
        plan.backproject(img, e, a, params=params, interp="sinc8")
        torch.cuda.synchronize()
    return img.cpu().numpy()


def _check(sc, img, pix=None):
    pix = scenes.compared_pixels(sc) if pix is None else pix
    ref = oracle.backproject(sc.params, sc.echoes, sc.antenna_pos, pix, interp="sinc8")
    m = parity.assert_parity(img.reshape(-1)[pix], ref, sc.cfg.name + " sinc8")
    nx, ny = sc.params["nx"], sc.params["ny"]
    ref_img = np.zeros(nx * ny, dtype=np.complex128)
    ref_img[pix] = ref
    bad = parity.argmax_mismatches(img, ref_img.reshape(ny, nx), sc.targets)
    assert not bad, f"argmax differs at {bad}"
    return m


@pytest.mark.parametrize("index", [1, 2])
def test_sinc_config_full_image(index):
    sc = scenes.make_scene(scenes.CONFIGS[index - 1])
    print(_check(sc, sinc_image(sc.params, sc.echoes, sc.antenna_pos)))


@pytest.mark.slow
def test_sinc_page_scene_full_size():
    sc = scenes.make_scene(scenes.CONFIGS[2])
    print(_check(sc, sinc_image(sc.params, sc.echoes, sc.antenna_pos)))


@pytest.mark.slow
@pytest.mark.parametrize("index", [4, 5])
def test_sinc_wide_scenes_sampled(index):
    """The 2048^2 and 4096^2 scenes: a thread's 32 pixels span up to about a
    range bin per pulse at the image's far x edges, so these run the
    wide-geometry sinc kernel (one polynomial of degree 5 or 6 per thread and
    pulse where its pixels span more than 0.34 bin)."""
    sc = scenes.make_scene(scenes.CONFIGS[index - 1])
    print(_check(sc, sinc_image(sc.params, sc.echoes, sc.antenna_pos)))


def _small(nx, ny, na=40, nr=512, noise=0.05):
    cfg = scenes.shrink(scenes.CONFIGS[0], nx=nx, ny=ny, na=na, nr=nr, spacing=0.5,
                        pulse_step=0.5, n_targets=0, noise_sigma=noise)
    return scenes.make_scene(cfg, seed=11)


def test_sinc_range_axis_edges():
    sc = _small(96, 300, na=24, nr=48, noise=0.3)
    p = dict(sc.params, r0=np.linalg.norm(sc.antenna_pos[12]) - 20 * sc.params["dr"])
    img = sinc_image(p, sc.echoes, sc.antenna_pos)
    ref = oracle.backproject(p, sc.echoes, sc.antenna_pos, interp="sinc8")
    assert np.any(ref == 0) and np.any(ref != 0)
    parity.assert_parity(img, ref, "sinc window edges")


def test_sinc_ragged_image():
    sc = _small(37, 201)
    img = sinc_image(sc.params, sc.echoes, sc.antenna_pos)
    parity.assert_parity(img, oracle.backproject(sc.params, sc.echoes, sc.antenna_pos,
                                                 interp="sinc8"), "sinc ragged")


def test_more_tiles_than_split_cells():
    """3 x 33,554,944 pixels at 0.1 mm: 65,537 tiles of 32 x 512, one more than
    the cells of the cost-weighted work split, so the call takes the even
    split (every CTA covers hundreds of whole tiles); sampled pixels and the
    image's corners against the oracle."""
    nx, ny = 3, 65537 * 512
    na, nr = 8, 4096
    spacing = 1.0e-4
    rng = np.random.default_rng(65537)
    pos = scenes.straight_track(na, 0.5)
    geo = scenes.image_geometry(nx, ny, spacing)
    near = np.array([0.0, geo["y0"], 0.0])
    far = np.array([0.0, geo["y0"] + ny * spacing, 0.0])
    rmin = float(np.min(np.linalg.norm(pos - near, axis=1))) - 20.0
    p = dict(nx=nx, ny=ny, na=na, nr=nr, r0=rmin, dr=scenes.DR, wavelength=scenes.WAVELENGTH, **geo)
    assert float(np.max(np.linalg.norm(pos - far, axis=1))) < rmin + (nr - 8) * scenes.DR
    echo = (rng.standard_normal((na, nr)) + 1j * rng.standard_normal((na, nr))).astype(np.complex64)
    img = torch.empty((ny, nx), dtype=torch.complex64, device=DEV)
    with Plan(p, interp="sinc8") as plan:
        assert plan.describe()["tiles"] == 65537
        plan.backproject(img, torch.from_numpy(echo).to(DEV), torch.from_numpy(pos).to(DEV),
                         interp="sinc8")
        torch.cuda.synchronize()
    pix = np.unique(np.concatenate([rng.choice(nx * ny, 3000, replace=False),
                                    [0, nx - 1, nx * ny - nx, nx * ny - 1]])).astype(np.int64)
    got = img.reshape(-1)[torch.from_numpy(pix).to(DEV)].cpu().numpy()
    del img
    ref = oracle.backproject(p, echo, pos, pix, interp="sinc8")
    parity.assert_parity(got, ref, "65537 tiles, sinc8")


def test_sinc_near_field_exact_path():
    na, nx, ny = 48, 64, 130
    pos = np.zeros((na, 3))
    pos[:, 0] = np.linspace(-20, 20, na)
    pos[:, 1] = -30.0
    pos[:, 2] = 40.0
    geo = scenes.image_geometry(nx, ny, 0.25)
    nr, r0, dr = 256, 20.0, 0.5
    p = dict(nx=nx, ny=ny, na=na, nr=nr, r0=r0, dr=dr, wavelength=scenes.WAVELENGTH, **geo)
    txyz = np.array([[geo["x0"] + 20 * 0.25, geo["y0"] + 70 * 0.25, 0.0]])
    echo = scenes.simulate_echoes(pos, txyz, np.array([1.0]), r0, dr, nr).astype(np.complex64)
    echo += (np.random.default_rng(2).standard_normal(echo.shape) * 0.05).astype(np.complex64)
    img = sinc_image(p, echo, pos)
    parity.assert_parity(img, oracle.backproject(p, echo, pos, interp="sinc8"), "sinc near field")


def test_sinc_host_entry_point():
    sc = _small(64, 200, na=64)
    with Plan(sc.params) as plan:
        host = np.zeros((sc.params["ny"], sc.params["nx"]), dtype=np.complex64)
        plan.backproject_host(host, sc.echoes, sc.antenna_pos, interp="sinc8")
    parity.assert_parity(host, oracle.backproject(sc.params, sc.echoes, sc.antenna_pos,
                                                  interp="sinc8"), "sinc host entry point")


def test_sinc_differs_from_linear():
    sc = scenes.make_scene(scenes.CONFIGS[0])
    lin = oracle.backproject(sc.params, sc.echoes, sc.antenna_pos)
    img = sinc_image(sc.params, sc.echoes, sc.antenna_pos)
    assert np.linalg.norm(img - lin) > 1e-2 * np.linalg.norm(lin)


def test_noalloc_rejects_sinc():
    sc = _small(32, 32, na=4)
    e = torch.from_numpy(sc.echoes).to(DEV)
    a = torch.from_numpy(sc.antenna_pos).to(DEV)
    img = torch.zeros((32, 32), dtype=torch.complex64, device=DEV)
    p = _native.Params.from_dict(sc.params, flags=_native.SARBP_SINC8)
    st = _native.lib().sarbp_backproject_noalloc(
        ctypes.c_void_p(img.data_ptr()), ctypes.c_void_p(e.data_ptr()),
        ctypes.c_void_p(a.data_ptr()), ctypes.byref(p), None)
    assert st == _native.SARBP_ERR_INVALID_ARG
