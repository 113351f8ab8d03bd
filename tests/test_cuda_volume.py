"""Voxel-grid backprojection (sarbp_backproject_volume) against the FP64 oracle.

SARBP-GPU §3.3 (the page "基于GPU的SAR后向投影成像优化与CUDA加速实践") notes that
the pixel grid may leave the ground plane. A voxel grid is a stack of planes
z0 + iz dz; each plane must equal the planar call bit for bit, and the volume
must match the oracle's stack under the usual tolerances (tests/parity.py).
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from domain_backprojection_sarbp_gb300 import Plan, SarbpError, _native  # noqa: E402
from synth import scenes  # noqa: E402
from tests import parity  # noqa: E402
from tests.test_oracle_volume_pins import pin_focus  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def _dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=dtype)).to(DEV)


def gpu_volume(params, echo, pos, nz, dz, interp="linear", init=None, accumulate=False):
    vol = torch.full((nz, params["ny"], params["nx"]), complex(3.0, 1.0), dtype=torch.complex64,
                     device=DEV)
    if init is not None:
        vol.copy_(torch.from_numpy(init.astype(np.complex64)))
    with Plan(params) as plan:
        plan.backproject_volume(vol, _dev(echo, np.complex64), _dev(pos, np.float64), dz,
                                params=params, interp=interp, accumulate=accumulate)
        torch.cuda.synchronize()
    return vol.cpu().numpy()


def multipass_scene(nx, ny, passes=6, na_pass=96, targets=((20, 30, 1), (60, 400, 3))):
    spacing, dz = 0.25, 0.5
    pos = scenes.multipass_track(na_pass, passes, 1.0, 40.0)
    geo = scenes.image_geometry(nx, ny, spacing)
    geo["z0"] = -1.0
    vox = np.array(targets)
    txyz = np.stack([geo["x0"] + vox[:, 0] * spacing, geo["y0"] + vox[:, 1] * spacing,
                     geo["z0"] + vox[:, 2] * dz], axis=1).astype(np.float64)
    nr = 4096
    r0 = float(np.linalg.norm(pos[len(pos) // 2])) - (nr // 2) * scenes.DR
    echo = scenes.simulate_echoes(pos, txyz, np.ones(len(vox)), r0, scenes.DR, nr)
    echo += 0.05 * (np.random.default_rng(5).standard_normal(echo.shape) + 0j)
    params = dict(nx=nx, ny=ny, na=len(pos), nr=nr, r0=r0, dr=scenes.DR,
                  wavelength=scenes.WAVELENGTH, **geo)
    return params, echo.astype(np.complex64), pos, dz


def test_volume_matches_the_oracle():
    # 100 x 600: ragged tiles in both directions; 5 planes
    params, echo, pos, dz = multipass_scene(100, 600)
    got = gpu_volume(params, echo, pos, 5, dz)
    ref = oracle.backproject_volume(params, echo, pos, 5, dz)
    print(parity.assert_parity(got, ref, "volume"))


@pytest.mark.parametrize("interp", ["linear", "sinc8", "nearest"])
def test_each_plane_is_the_planar_call(interp):
    params, echo, pos, dz = multipass_scene(64, 70, passes=2, na_pass=64, targets=((10, 10, 0),))
    vol = gpu_volume(params, echo, pos, 3, dz, interp=interp)
    e, a = _dev(echo, np.complex64), _dev(pos, np.float64)
    with Plan(params) as plan:
        for iz in range(3):
            p = dict(params, z0=params["z0"] + iz * dz)
            img = torch.zeros((params["ny"], params["nx"]), dtype=torch.complex64, device=DEV)
            plan.backproject(img, e, a, params=p, interp=interp)
            torch.cuda.synchronize()
            assert np.array_equal(vol[iz], img.cpu().numpy()), (interp, iz)


def test_focusing_pin_on_the_gpu():
    def bpv(params, echo, pos, nz, dz):
        return gpu_volume(params, echo, pos, nz, dz)
    ok, bad = pin_focus(bpv)
    assert ok, bad


def test_volume_accumulate_and_arguments():
    params, echo, pos, dz = multipass_scene(40, 30, passes=2, na_pass=32, targets=((10, 10, 0),))
    rng = np.random.default_rng(2)
    init = (rng.standard_normal((2, 30, 40)) + 1j * rng.standard_normal((2, 30, 40))).astype(np.complex64)
    once = gpu_volume(params, echo, pos, 2, dz)
    acc = gpu_volume(params, echo, pos, 2, dz, init=init, accumulate=True)
    assert np.abs(acc - (init + once)).max() <= 1e-5 * np.abs(once).max()
    lib = _native.lib()
    prm = _native.Params.from_dict(params)
    vol = torch.zeros((2, 30, 40), dtype=torch.complex64, device=DEV)
    e, a = _dev(echo, np.complex64), _dev(pos, np.float64)
    args = (ctypes.c_void_p(vol.data_ptr()), ctypes.c_void_p(e.data_ptr()),
            ctypes.c_void_p(a.data_ptr()), ctypes.byref(prm))
    with Plan(params) as plan:
        assert lib.sarbp_backproject_volume(plan.handle, *args, 0, 1.0, None) == _native.SARBP_OK
        for nz, dzv in ((-1, 1.0), (2, float("nan")), (2, float("inf"))):
            assert lib.sarbp_backproject_volume(plan.handle, *args, nz, dzv, None) == \
                _native.SARBP_ERR_INVALID_ARG
    with Plan(params, height_range=(0.0, 1.0)) as hp:
        with pytest.raises(SarbpError) as ex:
            hp.backproject_volume(vol, e, a, dz)
        assert ex.value.status == _native.SARBP_ERR_PLAN_MISMATCH
