"""Pulse-chunked host entry point (sarbp_backproject_streamed) and huge scenes.

SARBP-GPU §3.3 (the page "基于GPU的SAR后向投影成像优化与CUDA加速实践")
processes pulses in batches with copies overlapped on streams, and §4.1
images an 8192 x 8192 scene. Acceptance as for the other paths
(tests/parity.py) against the FP64 oracle; the single-chunk call must equal
sarbp_backproject_host bit for bit.
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


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(scope="module")
def small_spotlight():
    return scenes.make_scene(scenes.CONFIGS[1])


def streamed(plan, sc, chunk, init=None, accumulate=False):
    p = sc.params
    img = np.full((p["ny"], p["nx"]), 7 - 3j, dtype=np.complex64) if init is None else init.copy()
    plan.backproject_streamed(img, sc.echoes, sc.antenna_pos, chunk_pulses=chunk,
                              accumulate=accumulate)
    return img


@pytest.mark.parametrize("chunk", [100, 512])
def test_streamed_matches_oracle(small_spotlight, chunk):
    sc = small_spotlight                       # 1024 pulses: chunks of 100 leave a ragged 24
    with Plan(sc.params) as plan:
        got = streamed(plan, sc, chunk)
        h2d, d2h = plan.host_transfer_bytes()
    ref = oracle.backproject(sc.params, sc.echoes, sc.antenna_pos)
    parity.assert_parity(got, ref, f"streamed, chunk {chunk}")
    assert not parity.argmax_mismatches(got, ref, sc.targets)
    assert d2h == got.nbytes
    assert 0 < h2d <= sc.echoes.nbytes + sc.antenna_pos.nbytes


@pytest.mark.parametrize("interp", ["sinc8", "nearest"])
def test_streamed_interpolation_variants(small_spotlight, interp):
    sc = small_spotlight
    p = sc.params
    img = np.zeros((p["ny"], p["nx"]), dtype=np.complex64)
    with Plan(p) as plan:
        plan.backproject_streamed(img, sc.echoes, sc.antenna_pos, chunk_pulses=300, interp=interp)
    ref = oracle.backproject(p, sc.echoes, sc.antenna_pos, interp=interp)
    m = parity.compare(img, ref)
    # nearest: samples chosen at a half-bin knife edge may differ (both valid);
    # the image-wide error stays within the tolerance
    assert m["rel_l2"] <= parity.REL_L2 and m["max_err"] <= parity.MAX_ERR, m


def test_one_chunk_is_the_host_path(small_spotlight):
    sc = small_spotlight
    p = sc.params
    with Plan(p) as plan:
        one = streamed(plan, sc, 1 << 20)
        host = np.zeros((p["ny"], p["nx"]), dtype=np.complex64)
        plan.backproject_host(host, sc.echoes, sc.antenna_pos)
    assert np.array_equal(one, host)


def test_chunks_agree_with_the_host_path(small_spotlight):
    sc = small_spotlight
    p = sc.params
    with Plan(p) as plan:
        host = np.zeros((p["ny"], p["nx"]), dtype=np.complex64)
        plan.backproject_host(host, sc.echoes, sc.antenna_pos)
        for chunk in (1, 7, 128, 1023):
            got = streamed(plan, sc, chunk)
            err = np.abs(got - host).max() / np.abs(host).max()
            assert err <= 2e-5, (chunk, err)


def test_streamed_accumulate(small_spotlight):
    sc = small_spotlight
    p = sc.params
    rng = np.random.default_rng(11)
    init = (rng.standard_normal((p["ny"], p["nx"])) +
            1j * rng.standard_normal((p["ny"], p["nx"]))).astype(np.complex64)
    with Plan(p) as plan:
        once = streamed(plan, sc, 256)
        acc = streamed(plan, sc, 256, init=init, accumulate=True)
    assert np.abs(acc - (init + once)).max() <= 1e-5 * np.abs(once).max()


def test_long_track_chunks_copy_less():
    """A 1.6 km aperture: each chunk of pulses reaches a narrower band of range
    bins than the whole track, so the streamed call copies fewer bytes."""
    cfg = scenes.shrink(scenes.CONFIGS[3], na=4096, nr=8192, nx=512, ny=512,
                        pulse_step=0.4, n_targets=16)
    sc = scenes.make_scene(cfg)
    p = sc.params
    with Plan(p) as plan:
        got = streamed(plan, sc, 512)
        h2d_streamed, _ = plan.host_transfer_bytes()
        host = np.zeros((p["ny"], p["nx"]), dtype=np.complex64)
        plan.backproject_host(host, sc.echoes, sc.antenna_pos)
        h2d_host, _ = plan.host_transfer_bytes()
    assert h2d_streamed < h2d_host
    pix = scenes.compared_pixels(sc)
    ref = oracle.backproject(p, sc.echoes, sc.antenna_pos, pix)
    parity.assert_parity(got.reshape(-1)[pix], ref, "long track, streamed")


def test_streamed_arguments(small_spotlight):
    sc = small_spotlight
    p = sc.params
    lib = _native.lib()
    prm = _native.Params.from_dict(p)
    img = np.zeros((p["ny"], p["nx"]), dtype=np.complex64)
    with Plan(p) as plan:
        for chunk in (0, -5):
            st = lib.sarbp_backproject_streamed(
                plan.handle, ctypes.c_void_p(img.ctypes.data), ctypes.c_void_p(sc.echoes.ctypes.data),
                ctypes.c_void_p(sc.antenna_pos.ctypes.data), ctypes.byref(prm), chunk, None)
            assert st == _native.SARBP_ERR_INVALID_ARG
    with Plan(p, height_range=(0.0, 1.0)) as hp:
        with pytest.raises(SarbpError) as ex:
            hp.backproject_streamed(img, sc.echoes, sc.antenna_pos)
        assert ex.value.status == _native.SARBP_ERR_PLAN_MISMATCH


def test_no_pulses_and_no_bins():
    sc = scenes.make_scene(scenes.CONFIGS[0])
    for change in (dict(na=0), dict(nr=1)):
        p = dict(sc.params, **change)
        ech = np.ones((p["na"], p["nr"]), dtype=np.complex64)
        pos = sc.antenna_pos[:p["na"]].copy()
        img = np.full((p["ny"], p["nx"]), 1 + 1j, dtype=np.complex64)
        with Plan(p) as plan:
            plan.backproject_streamed(img, ech, pos, chunk_pulses=16)
        assert not img.any(), change


# ----------------------------------------------------------- huge scene
@pytest.mark.slow
def test_scene_8192_squared():
    """The page's large scene size, 8192 x 8192 pixels, in one call (tiles are
    the kernel's own; no seams), streamed in chunks; sampled against the oracle."""
    cfg = scenes.shrink(scenes.CONFIGS[3], na=256, nr=8192, nx=8192, ny=8192, n_targets=64,
                        pulse_step=1.6)
    sc = scenes.make_scene(cfg)
    with Plan(sc.params) as plan:
        got = streamed(plan, sc, 64)
    pix = scenes.compared_pixels(sc)
    ref = oracle.backproject(sc.params, sc.echoes, sc.antenna_pos, pix)
    parity.assert_parity(got.reshape(-1)[pix], ref, "8192 x 8192")
    full = np.zeros(cfg.nx * cfg.ny, dtype=np.complex128)
    full[pix] = ref
    assert not parity.argmax_mismatches(got, full.reshape(cfg.ny, cfg.nx), sc.targets)
