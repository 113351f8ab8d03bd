"""Failure handling, with the failure made on the host: a device allocation the
library makes is told to fail (sarbp_debug_fail_alloc) as if cudaMalloc had
run out of memory. Nothing faults, traps or hangs the GPU. Every call that
meets the failure must return SARBP_ERR_OOM, free what it had allocated and
leave the library usable: the next call succeeds and computes the right image.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from domain_backprojection_sarbp_gb300 import Plan, RangeCompressor, SarbpError, _native  # noqa: E402
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


@pytest.fixture(autouse=True)
def _reset():
    yield
    _native.lib().sarbp_debug_fail_alloc(0)


@pytest.fixture(scope="module")
def scene():
    return scenes.make_scene(scenes.shrink(scenes.CONFIGS[1], na=256, nx=128, ny=96, n_targets=2))


def _free_bytes():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


@pytest.mark.parametrize("which", [1, 2, 3, 4])
def test_plan_creation_fails_cleanly(scene, which):
    lib = _native.lib()
    prm = _native.Params.from_dict(scene.params)
    h = ctypes.c_void_p()
    Plan(scene.params).close()                     # warm the context and the library
    before = _free_bytes()
    lib.sarbp_debug_fail_alloc(which)              # plan_create makes four allocations
    st = lib.sarbp_plan(ctypes.byref(h), ctypes.byref(prm))
    assert st == _native.SARBP_ERR_OOM
    assert not h.value
    assert abs(_free_bytes() - before) <= 8 << 20  # freed (the stream-K partials alone are 40 MB)
    with Plan(scene.params) as plan:               # the next plan works
        img = torch.zeros((96, 128), dtype=torch.complex64, device=DEV)
        plan.backproject(img, torch.from_numpy(scene.echoes).to(DEV),
                         torch.from_numpy(scene.antenna_pos).to(DEV))
        torch.cuda.synchronize()
    ref = oracle.backproject(scene.params, scene.echoes, scene.antenna_pos)
    parity.assert_parity(img.cpu().numpy(), ref, "after a failed plan")


def test_heights_plan_fails_cleanly(scene):
    lib = _native.lib()
    prm = _native.Params.from_dict(scene.params)
    h = ctypes.c_void_p()
    lib.sarbp_debug_fail_alloc(2)
    assert lib.sarbp_plan_heights(ctypes.byref(h), ctypes.byref(prm), 0.0, 10.0) == \
        _native.SARBP_ERR_OOM
    assert not h.value


@pytest.mark.parametrize("which", [1, 2, 3])
def test_host_call_staging_fails_then_recovers(scene, which):
    lib = _native.lib()
    p = scene.params
    ref = oracle.backproject(p, scene.echoes, scene.antenna_pos)
    with Plan(p) as plan:
        img = np.zeros((p["ny"], p["nx"]), dtype=np.complex64)
        lib.sarbp_debug_fail_alloc(which)          # image, positions, echo band
        with pytest.raises(SarbpError) as ex:
            plan.backproject_host(img, scene.echoes, scene.antenna_pos)
        assert ex.value.status == _native.SARBP_ERR_OOM
        assert "cudaMalloc" in lib.sarbp_last_error(plan.handle).decode()
        lib.sarbp_debug_fail_alloc(0)
        plan.backproject_host(img, scene.echoes, scene.antenna_pos)
    parity.assert_parity(img, ref, "host call after a failed staging allocation")


@pytest.mark.parametrize("which", [1, 2, 3, 4])
def test_streamed_staging_fails_then_recovers(scene, which):
    lib = _native.lib()
    p = scene.params
    ref = oracle.backproject(p, scene.echoes, scene.antenna_pos)
    with Plan(p) as plan:
        img = np.zeros((p["ny"], p["nx"]), dtype=np.complex64)
        lib.sarbp_debug_fail_alloc(which)          # image, positions, two staging buffers
        with pytest.raises(SarbpError) as ex:
            plan.backproject_streamed(img, scene.echoes, scene.antenna_pos, chunk_pulses=64)
        assert ex.value.status == _native.SARBP_ERR_OOM
        lib.sarbp_debug_fail_alloc(0)
        plan.backproject_streamed(img, scene.echoes, scene.antenna_pos, chunk_pulses=64)
    parity.assert_parity(img, ref, "streamed call after a failed staging allocation")


def test_range_compression_plan_fails_cleanly():
    """The range-compression plan makes one device allocation, the filter
    spectrum; when it fails the plan is not made, and the next one works."""
    lib = _native.lib()
    ref = torch.ones(64, dtype=torch.complex64, device=DEV)
    lib.sarbp_debug_fail_alloc(1)                  # the filter spectrum
    with pytest.raises(SarbpError) as ex:
        RangeCompressor(ref, 4, 1000)
    assert ex.value.status == _native.SARBP_ERR_OOM
    lib.sarbp_debug_fail_alloc(2)                  # armed past the plan's one allocation
    RangeCompressor(ref, 4, 1000).close()
    lib.sarbp_debug_fail_alloc(0)
    raw = torch.randn(4, 1000, dtype=torch.complex64, device=DEV)
    out = torch.empty_like(raw)
    with RangeCompressor(ref, 4, 1000) as rc:
        rc(out, raw)
        torch.cuda.synchronize()
    from oracle import range_compression as rco
    want = rco.range_compress(raw.cpu().numpy(), ref.cpu().numpy())
    assert parity.compare(out.cpu().numpy(), want)["rel_l2"] < 1e-5


def test_sinc_plan_creation_fails_cleanly(scene):
    """A plan made for sinc allocates its coefficient rows fifth; when that
    fails the plan is not made and its other scratch is freed."""
    lib = _native.lib()
    prm = _native.Params.from_dict(scene.params)
    prm.flags |= _native.SARBP_SINC8
    h = ctypes.c_void_p()
    Plan(scene.params).close()
    before = _free_bytes()
    lib.sarbp_debug_fail_alloc(5)
    assert lib.sarbp_plan(ctypes.byref(h), ctypes.byref(prm)) == _native.SARBP_ERR_OOM
    assert not h.value
    assert abs(_free_bytes() - before) <= 8 << 20


def test_first_sinc_call_allocation_fails_then_recovers(scene):
    """On a plan made without sinc, the first sinc call allocates the
    coefficient rows; when that fails the call returns SARBP_ERR_OOM having
    queued nothing (the image is untouched), and the next call works."""
    lib = _native.lib()
    p = scene.params
    e = torch.from_numpy(scene.echoes).to(DEV)
    a = torch.from_numpy(scene.antenna_pos).to(DEV)
    with Plan(p) as plan:
        img = torch.full((p["ny"], p["nx"]), complex(3.0, 4.0), dtype=torch.complex64, device=DEV)
        lib.sarbp_debug_fail_alloc(1)
        with pytest.raises(SarbpError) as ex:
            plan.backproject(img, e, a, interp="sinc8")
        assert ex.value.status == _native.SARBP_ERR_OOM
        assert "sinc" in lib.sarbp_last_error(plan.handle).decode()
        torch.cuda.synchronize()
        assert bool(torch.all(img == complex(3.0, 4.0)))
        lib.sarbp_debug_fail_alloc(0)
        plan.backproject(img, e, a, interp="sinc8")
        torch.cuda.synchronize()
    ref = oracle.backproject(p, scene.echoes, scene.antenna_pos, interp="sinc8")
    parity.assert_parity(img.cpu().numpy(), ref, "sinc call after a failed coefficient-row allocation")
