"""Parity across radar bands and flight geometries the five configurations do not cover.

The kernel picks, per thread and pulse, between its hinge, gather and exact
forms from bounds on the range polynomial; these cases move those bounds:
long and short wavelengths, fine and coarse range bins, a squinted and a
circular aperture, a low near-field pass, and an image far off broadside.
Each image is compared in full with the FP64 oracle (tests/parity.py), for
the linear path and, on some cases, the windowed sinc and nearest sample.
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
C = scenes.C_LIGHT


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def _track_line(na, step, x_centre=0.0, y=-7000.0, z=5000.0):
    pos = np.zeros((na, 3))
    pos[:, 0] = x_centre + (np.arange(na) - (na - 1) / 2) * step
    pos[:, 1] = y
    pos[:, 2] = z
    return pos


def _track_circle(na, radius, z, arc):
    th = np.linspace(-arc / 2, arc / 2, na) - np.pi / 2
    return np.stack([radius * np.cos(th), radius * np.sin(th), np.full(na, z)], axis=1)


def _scene(pos, fc, dr, spacing, nx=160, ny=530, nr=None, centre=(0.0, 0.0), seed=0):
    lam = C / fc
    rng = np.random.default_rng(seed)
    geo = scenes.image_geometry(nx, ny, spacing)
    geo["x0"] += centre[0]
    geo["y0"] += centre[1]
    corners = np.array([[geo["x0"] + a * (nx - 1) * spacing, geo["y0"] + b * (ny - 1) * spacing, 0.0]
                        for a in (0, 1) for b in (0, 1)])
    d = np.linalg.norm(pos[:, None, :] - corners[None, :, :], axis=2)
    near = max(float(np.min(np.linalg.norm(pos - np.array([*centre, 0.0]), axis=1))) - 0.75 *
               float(np.linalg.norm([nx * spacing, ny * spacing])), 1.0)
    r0 = near - 20 * dr
    nr = nr or int(np.ceil((d.max() - r0) / dr)) + 40
    tx = rng.integers(12, nx - 12, 6)
    ty = rng.integers(12, ny - 12, 6)
    txyz = np.stack([geo["x0"] + tx * spacing, geo["y0"] + ty * spacing, np.zeros(6)], axis=1)
    echo = scenes.simulate_echoes(pos, txyz, rng.uniform(0.5, 1.0, 6), r0, dr, nr, wavelength=lam,
                                  rho=max(dr, 0.3))
    echo += 0.05 * (rng.standard_normal(echo.shape) + 1j * rng.standard_normal(echo.shape))
    params = dict(nx=nx, ny=ny, na=len(pos), nr=nr, r0=r0, dr=dr, wavelength=lam, **geo)
    return params, echo.astype(np.complex64), pos


CASES = {
    # name: (antenna positions, fc, dr, pixel spacing, image centre)
    "l_band": (_track_line(256, 2.0), 1.25e9, 1.0, 1.0, (0.0, 0.0)),
    "ka_band": (_track_line(512, 0.02), 35e9, 0.15, 0.05, (0.0, 0.0)),
    "fine_bins": (_track_line(256, 0.1), 9.6e9, 0.05, 0.05, (0.0, 0.0)),
    "coarse_bins": (_track_line(256, 0.4), 9.6e9, 3.0, 1.0, (0.0, 0.0)),
    "squint_25deg": (_track_line(384, 0.1, x_centre=-3700.0), 9.6e9, 0.8333, 0.15, (0.0, 0.0)),
    "circular_arc": (_track_circle(720, 6000.0, 4000.0, np.deg2rad(30.0)), 9.6e9, 0.5, 0.1, (0.0, 0.0)),
    "low_pass": (_track_line(256, 0.2, y=-400.0, z=250.0), 9.6e9, 0.3, 0.1, (0.0, 0.0)),
    "off_broadside": (_track_line(256, 0.1), 9.6e9, 0.8333, 0.25, (2500.0, 1500.0)),
}

# slant ranges at and beyond the ~10 km the float32 phase must hold at
# (SARBP-GPU §2.2, range-computation precision): X band at 12.8 km (8000 m
# altitude, 10 km ground offset) and Ka band (lambda = 8.6 mm, 4.5 rad of phase
# per millimetre of range) at 10 km (6000 m, 8 km)
LONG_RANGE = {
    "x_band_12800m": (_track_line(512, 0.1, y=-10000.0, z=8000.0), 9.6e9, 0.8333, 0.15, (0.0, 0.0)),
    "ka_band_10km": (_track_line(512, 0.02, y=-8000.0, z=6000.0), 35e9, 0.15, 0.05, (0.0, 0.0)),
}


def test_anisotropic_pixels_and_raised_plane():
    """dx != dy, an image plane 120 m above the origin and a descending track."""
    pos = _track_line(300, -0.3, y=-6000.0, z=4500.0)
    params, echo, pos = _scene(pos, 9.6e9, 0.6, 0.1, nx=150, ny=400)
    params = dict(params, dy=0.35, z0=120.0)
    got = _gpu(params, echo, pos, "linear")
    ref = oracle.backproject(params, echo, pos)
    print("anisotropic", parity.assert_parity(got, ref, "anisotropic, raised plane"))


@pytest.mark.parametrize("interp", ["linear", "sinc8", "nearest"])
def test_accumulated_pulse_batches_equal_one_call(interp):
    """Two calls over halves of the pulses with SARBP_ACCUMULATE give the
    one-call image to float32 rounding, for every interpolation."""
    pos, fc, dr, spacing, centre = CASES["circular_arc"]
    params, echo, pos = _scene(pos, fc, dr, spacing, centre=centre, nx=96, ny=200, seed=3)
    na = params["na"]
    whole = _gpu(params, echo, pos, interp)
    half = na // 2
    img = torch.zeros((params["ny"], params["nx"]), dtype=torch.complex64, device=DEV)
    for lo, hi in ((0, half), (half, na)):
        p = dict(params, na=hi - lo)
        with Plan(p) as plan:
            plan.backproject(img, torch.from_numpy(np.ascontiguousarray(echo[lo:hi])).to(DEV),
                             torch.from_numpy(np.ascontiguousarray(pos[lo:hi])).to(DEV),
                             accumulate=lo > 0, interp=interp)
            torch.cuda.synchronize()
    two = img.cpu().numpy()
    assert np.abs(two - whole).max() <= 2e-5 * np.abs(whole).max()


def _gpu(params, echo, pos, interp):
    img = torch.zeros((params["ny"], params["nx"]), dtype=torch.complex64, device=DEV)
    with Plan(params) as plan:
        plan.backproject(img, torch.from_numpy(echo).to(DEV), torch.from_numpy(pos).to(DEV),
                         interp=interp)
        torch.cuda.synchronize()
    return img.cpu().numpy()


@pytest.mark.parametrize("name", sorted(CASES))
def test_linear(name):
    pos, fc, dr, spacing, centre = CASES[name]
    params, echo, pos = _scene(pos, fc, dr, spacing, centre=centre)
    got = _gpu(params, echo, pos, "linear")
    ref = oracle.backproject(params, echo, pos)
    print(name, parity.assert_parity(got, ref, name))


@pytest.mark.parametrize("name", ["l_band", "squint_25deg", "circular_arc", "low_pass"])
def test_sinc8(name):
    pos, fc, dr, spacing, centre = CASES[name]
    params, echo, pos = _scene(pos, fc, dr, spacing, centre=centre, seed=1)
    got = _gpu(params, echo, pos, "sinc8")
    ref = oracle.backproject(params, echo, pos, interp="sinc8")
    print(name, parity.assert_parity(got, ref, name))


@pytest.mark.parametrize("name", ["ka_band", "coarse_bins", "off_broadside"])
def test_nearest(name):
    pos, fc, dr, spacing, centre = CASES[name]
    params, echo, pos = _scene(pos, fc, dr, spacing, centre=centre, seed=2)
    got = _gpu(params, echo, pos, "nearest")
    ref = oracle.backproject(params, echo, pos, interp="nearest")
    # a sample chosen at a half-bin knife edge may differ (both valid); the
    # image-wide error stays within the tolerance
    m = parity.compare(got, ref)
    print(name, m)
    assert m["rel_l2"] <= parity.REL_L2 and m["max_err"] <= parity.MAX_ERR, m


@pytest.mark.parametrize("name", ["squint_25deg", "low_pass"])
def test_sinc8_wide_geometry_at_range_axis_edges(name):
    """A geometry where a thread's 32 pixels span more than 0.34 bin, the
    widest polynomial of the narrow sinc kernel (so the wide kernel, with its
    degree-5 and degree-6 polynomials and per-pixel taps, runs), with the recorded range
    axis cut so that it starts and ends inside the image: stencils that reach
    past either end contribute nothing, per pixel and per part."""
    pos, fc, dr, spacing, centre = CASES[name]
    params, echo, pos = _scene(pos, fc, dr, spacing, centre=centre, seed=4)
    xs = params["x0"] + np.array([0.0, params["nx"] - 1]) * params["dx"]
    rmin = np.min(np.linalg.norm(pos, axis=1)) - np.hypot(params["nx"] * spacing, params["ny"] * spacing)
    spread = 31 * params["dx"] * np.max(np.abs(xs[None, :] - pos[:, :1])) / (rmin * dr)
    assert spread > 0.34, spread
    # keep the middle half of the bins the middle pulse sees the image in: its
    # ranges then run past both ends of the cut axis
    gx, gy = np.meshgrid(params["x0"] + np.arange(params["nx"]) * params["dx"],
                         params["y0"] + np.arange(params["ny"]) * params["dy"])
    a = pos[len(pos) // 2]
    u = (np.sqrt((gx - a[0]) ** 2 + (gy - a[1]) ** 2 + a[2] ** 2) - params["r0"]) / dr
    off = int(u.min() + 0.25 * (u.max() - u.min()))
    keep = int(0.5 * (u.max() - u.min()))
    assert u.min() - off < 0 and u.max() - off > keep
    cut = dict(params, nr=keep, r0=params["r0"] + off * dr)
    e = np.ascontiguousarray(echo[:, off:off + keep])
    got = _gpu(cut, e, pos, "sinc8")
    ref = oracle.backproject(cut, e, pos, interp="sinc8")
    print(name, parity.assert_parity(got, ref, name + " cut range axis"))


@pytest.mark.parametrize("interp", ["linear", "sinc8", "nearest"])
@pytest.mark.parametrize("name", sorted(LONG_RANGE))
def test_long_slant_range(name, interp):
    """Every pixel against the oracle at 10-13 km slant range."""
    pos, fc, dr, spacing, centre = LONG_RANGE[name]
    params, echo, pos = _scene(pos, fc, dr, spacing, centre=centre, seed=5)
    rng_c = float(np.linalg.norm(pos[len(pos) // 2]))
    assert rng_c >= (12_000.0 if fc < 20e9 else 9_900.0), rng_c
    got = _gpu(params, echo, pos, interp)
    ref = oracle.backproject(params, echo, pos, interp=interp)
    m = parity.compare(got, ref)
    print(name, interp, f"slant range {rng_c:.0f} m", m)
    assert m["finite"] and m["rel_l2"] <= parity.REL_L2 and m["max_err"] <= parity.MAX_ERR, m
