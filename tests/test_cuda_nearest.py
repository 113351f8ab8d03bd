"""Nearest-neighbour interpolation (SARBP_NEAREST) against the FP64 oracle.

SARBP-GPU §2.2 (the page "基于GPU的SAR后向投影成像优化与CUDA加速实践") lists it
as the fastest, least accurate choice. The nearest sample is an integer
decision taken from the range: where a range lies within KNIFE bins of a
half-bin, the float32 kernel and the float64 oracle may pick different
samples and both are valid. So: relative L2 <= 1e-3 over the image, and
max |error| <= 1e-3 of the peak at every pixel none of whose ranges is such a
knife edge (checked in float64).
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from domain_backprojection_sarbp_gb300 import Plan  # noqa: E402
from synth import scenes  # noqa: E402
from tests import parity  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
KNIFE = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def nearest_image(params, echoes, pos):
    e = torch.from_numpy(np.ascontiguousarray(echoes, dtype=np.complex64)).to(DEV)
    a = torch.from_numpy(np.ascontiguousarray(pos, dtype=np.float64)).to(DEV)
    img = torch.full((params["ny"], params["nx"]), complex(7.0, -3.0), dtype=torch.complex64,
                     device=DEV)
    with Plan(params) as plan:
        plan.backproject(img, e, a, params=params, interp="nearest")
        torch.cuda.synchronize()
    return img.cpu().numpy()


def _knife_gap(params, echoes, pos, pixel):
    """Largest change the two valid choices at knife-edge pulses can make at a pixel:
    sum over pulses whose range is within KNIFE of a half-bin of |e[k] - e[k+1]|."""
    ix, iy = pixel % params["nx"], pixel // params["nx"]
    p = np.array([params["x0"] + ix * params["dx"], params["y0"] + iy * params["dy"], params["z0"]])
    u = (np.linalg.norm(pos - p[None, :], axis=1) - params["r0"]) / params["dr"]
    k = np.floor(u).astype(np.int64)
    knife = (np.abs(u - k - 0.5) < KNIFE) & (k >= -1) & (k <= params["nr"] - 1)
    gap = 0.0
    for n in np.nonzero(knife)[0]:
        lo = echoes[n, k[n]] if k[n] >= 0 else 0.0
        hi = echoes[n, k[n] + 1] if k[n] + 1 <= params["nr"] - 1 else 0.0
        gap += abs(complex(lo) - complex(hi))
    return gap


def check(params, echoes, pos, img, pix=None, targets=None):
    nx, ny = params["nx"], params["ny"]
    pix = np.arange(nx * ny) if pix is None else pix
    ref = oracle.backproject(params, echoes, pos, pix, interp="nearest")
    got = img.reshape(-1)[pix]
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    tol = parity.MAX_ERR * np.abs(ref).max()
    suspect = np.nonzero(err > min(tol, 1e-3 * np.abs(ref).max()))[0]
    explained = []
    for i in suspect:
        gap = _knife_gap(params, echoes, pos, int(pix[i]))
        assert err[i] <= gap + tol, f"pixel {int(pix[i])}: error {err[i]:.3e} beyond knife edges"
        if gap > 0:
            explained.append(i)
    keep = np.setdiff1d(np.arange(pix.size), np.array(explained, dtype=np.int64))
    m = parity.compare(got[keep], ref[keep])
    assert m["rel_l2"] <= parity.REL_L2 and m["max_err"] <= parity.MAX_ERR, m
    if targets is not None:
        ref_img = np.zeros(nx * ny, dtype=np.complex128)
        ref_img[pix] = ref
        assert not parity.argmax_mismatches(img, ref_img.reshape(ny, nx), targets)
    return m, len(explained)


@pytest.mark.parametrize("index", [1, 2])
def test_nearest_config_full_image(index):
    sc = scenes.make_scene(scenes.CONFIGS[index - 1])
    img = nearest_image(sc.params, sc.echoes, sc.antenna_pos)
    print(check(sc.params, sc.echoes, sc.antenna_pos, img, targets=sc.targets))


@pytest.mark.slow
def test_nearest_page_scene_full_size():
    """4096 pulses onto 1024 x 1024 pixels, the bench's launch configuration;
    compared on the sampled pixel set."""
    sc = scenes.make_scene(scenes.CONFIGS[2])
    img = nearest_image(sc.params, sc.echoes, sc.antenna_pos)
    print(check(sc.params, sc.echoes, sc.antenna_pos, img, pix=scenes.compared_pixels(sc),
                targets=sc.targets))


def _small(nx, ny, na=40, nr=512, noise=0.05):
    cfg = scenes.shrink(scenes.CONFIGS[0], nx=nx, ny=ny, na=na, nr=nr, spacing=0.5,
                        pulse_step=0.5, n_targets=0, noise_sigma=noise)
    return scenes.make_scene(cfg, seed=13)


def test_nearest_range_axis_edges():
    sc = _small(96, 300, na=24, nr=48, noise=0.3)
    p = dict(sc.params, r0=np.linalg.norm(sc.antenna_pos[12]) - 20 * sc.params["dr"])
    print(check(p, sc.echoes, sc.antenna_pos, nearest_image(p, sc.echoes, sc.antenna_pos)))


def test_nearest_ragged():
    sc = _small(37, 201)
    print(check(sc.params, sc.echoes, sc.antenna_pos,
                nearest_image(sc.params, sc.echoes, sc.antenna_pos)))


def test_nearest_near_field():
    na, nx, ny = 48, 64, 130
    pos = np.zeros((na, 3))
    pos[:, 0] = np.linspace(-20, 20, na)
    pos[:, 1] = -30.0
    pos[:, 2] = 40.0
    geo = scenes.image_geometry(nx, ny, 0.25)
    p = dict(nx=nx, ny=ny, na=na, nr=256, r0=20.0, dr=0.5, wavelength=scenes.WAVELENGTH, **geo)
    echo = (np.random.default_rng(4).standard_normal((na, 256)) * (1 + 1j)).astype(np.complex64)
    print(check(p, echo, pos, nearest_image(p, echo, pos)))
