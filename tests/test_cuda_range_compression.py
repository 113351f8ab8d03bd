"""Range compression on the GPU (sarbp_range_compress) against the FP64 oracle.

SARBP-GPU §3.1 (the page "基于GPU的SAR后向投影成像优化与CUDA加速实践"): batched
range FFT, matched-filter multiply with an optional Hamming window, inverse FFT.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from domain_backprojection_sarbp_gb300 import Plan, RangeCompressor, SarbpError, _native  # noqa: E402
from oracle import range_compression as rco  # noqa: E402
from synth import chirp, scenes  # noqa: E402
from tests import parity  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def gpu_compress(raw, ref, window="none", band=1.0):
    r = torch.from_numpy(np.ascontiguousarray(raw, dtype=np.complex64)).to(DEV)
    f = torch.from_numpy(np.ascontiguousarray(ref, dtype=np.complex64)).to(DEV)
    out = torch.full_like(r, complex(9.0, 9.0))
    with RangeCompressor(f, raw.shape[0], raw.shape[1], window, band) as rc:
        rc(out, r)
        torch.cuda.synchronize()
    return out.cpu().numpy()


# FFT sizes 2 .. 16384: every first-pass radix (2, 4, 8, 16) and one to four passes
@pytest.mark.parametrize("ns,nref", [(1, 1), (3, 2), (5, 3), (10, 5), (20, 9), (50, 10), (100, 7),
                                     (200, 40), (400, 100), (1000, 25), (1500, 300), (3000, 500),
                                     (4096, 359), (16384 - 358, 359)])
def test_random_rows(ns, nref):
    rng = np.random.default_rng(ns)
    raw = (rng.standard_normal((5, ns)) + 1j * rng.standard_normal((5, ns))).astype(np.complex64)
    ref = (rng.standard_normal(nref) + 1j * rng.standard_normal(nref)).astype(np.complex64)
    got = gpu_compress(raw, ref)
    want = rco.range_compress(raw, ref)
    m = parity.compare(got, want)
    assert m["rel_l2"] < 1e-5 and m["max_err"] < 1e-5, m


@pytest.mark.parametrize("window", ["hamming", "taylor"])
def test_chirp_windowed_page_size(window):
    sc = scenes.make_scene(scenes.shrink(scenes.CONFIGS[2], na=64, nx=64, ny=64, n_targets=1))
    ref = chirp.chirp()
    band = chirp.BANDWIDTH / (chirp.C_LIGHT / (2 * chirp.DR))
    tgt = np.array([[0.0, 0.0, 0.0]])
    raw = chirp.raw_echoes(sc.antenna_pos, tgt, np.array([1.0]), sc.params["r0"], 4096)
    raw += 0.1 * (np.random.default_rng(3).standard_normal(raw.shape) + 0j)
    got = gpu_compress(raw, ref, window, band)
    want = rco.range_compress(raw.astype(np.complex64), ref.astype(np.complex64), window, band)
    m = parity.compare(got, want)
    assert m["rel_l2"] < 1e-5 and m["max_err"] < 1e-5, m


def test_limits_and_errors():
    ref = torch.zeros(359, dtype=torch.complex64, device=DEV)
    with pytest.raises(SarbpError):
        RangeCompressor(ref, 4, 16384 - 357)                 # N would be 32768
    with pytest.raises(SarbpError):
        RangeCompressor(ref, 4, 1000, "hamming", 0.0)
    p = _native.RcParams(4, 100, 359, 7, 1.0)
    h = ctypes.c_void_p()
    assert _native.lib().sarbp_rc_plan(ctypes.byref(h), ctypes.byref(p),
                                       ctypes.c_void_p(ref.data_ptr()), None) == \
        _native.SARBP_ERR_INVALID_ARG


def test_raw_to_image_pipeline():
    """raw chirps -> range compression -> backprojection, against the same two
    steps in the oracle."""
    cfg = scenes.shrink(scenes.CONFIGS[0], na=64, nr=512, nx=64, ny=64, n_targets=3,
                        pulse_step=0.5)
    sc = scenes.make_scene(cfg, noise=False)
    p = sc.params
    txyz = np.zeros((len(sc.targets), 3))
    txyz[:, 0] = p["x0"] + sc.targets[:, 0] * p["dx"]
    txyz[:, 1] = p["y0"] + sc.targets[:, 1] * p["dy"]
    raw = chirp.raw_echoes(sc.antenna_pos, txyz, sc.amps, p["r0"], p["nr"]).astype(np.complex64)
    ref = chirp.chirp().astype(np.complex64)
    band = chirp.BANDWIDTH / (chirp.C_LIGHT / (2 * chirp.DR))

    rc_gpu = torch.from_numpy(gpu_compress(raw, ref, "hamming", band)).to(DEV)
    pos = torch.from_numpy(sc.antenna_pos).to(DEV)
    img = torch.zeros((p["ny"], p["nx"]), dtype=torch.complex64, device=DEV)
    with Plan(p) as plan:
        plan.backproject(img, rc_gpu, pos)
        torch.cuda.synchronize()
    got = img.cpu().numpy()

    rc_ref = rco.range_compress(raw, ref, "hamming", band).astype(np.complex64)
    want = oracle.backproject(p, rc_ref, sc.antenna_pos)
    parity.assert_parity(got, want, "raw -> image")
    assert not parity.argmax_mismatches(got, want, sc.targets)


def _raw_scene(nr, na=64, nx=64, ny=64):
    cfg = scenes.shrink(scenes.CONFIGS[0], na=na, nr=nr, nx=nx, ny=ny, n_targets=3,
                        pulse_step=0.5)
    sc = scenes.make_scene(cfg, noise=False)
    p = sc.params
    txyz = np.zeros((len(sc.targets), 3))
    txyz[:, 0] = p["x0"] + sc.targets[:, 0] * p["dx"]
    txyz[:, 1] = p["y0"] + sc.targets[:, 1] * p["dy"]
    raw = chirp.raw_echoes(sc.antenna_pos, txyz, sc.amps, p["r0"], p["nr"])
    g = np.random.default_rng(nr).standard_normal((na, nr, 2))
    raw += 0.05 * (g[..., 0] + 1j * g[..., 1])
    return sc, raw.astype(np.complex64)


# FFT sizes 512 (radix-32 first pass, one pass of radix 16), 1024 (first pass of
# radix 4) and 8192 (radix 32, 16, 16); up to 512 bins the table rows of this
# 64 x 64 image (one 512-row tile) span the whole range axis, so the band kept
# in shared memory is the whole row; at 4096 it is a window of it
@pytest.mark.parametrize("nr", [128, 256, 512, 4096])
def test_raw_entry_point(nr):
    """sarbp_backproject_raw (range compression fused with the echo table)
    against the oracle's range compression followed by its backprojection,
    and bit for bit against the two library calls it fuses. One pulse has a
    non-finite antenna position and contributes nothing."""
    sc, raw = _raw_scene(nr)
    p = sc.params
    with Plan(p) as probe:
        full = probe.describe()["full_window"]
    assert full == (1 if nr <= 512 else 0), (nr, full)
    pos_np = sc.antenna_pos.copy()
    pos_np[7] = np.nan
    ref = chirp.chirp().astype(np.complex64)
    band = chirp.BANDWIDTH / (chirp.C_LIGHT / (2 * chirp.DR))
    r = torch.from_numpy(raw).to(DEV)
    pos = torch.from_numpy(pos_np).to(DEV)
    f = torch.from_numpy(ref).to(DEV)
    img = torch.full((p["ny"], p["nx"]), complex(3.0, 3.0), dtype=torch.complex64, device=DEV)
    two = torch.full_like(img, complex(3.0, 3.0))
    comp = torch.empty_like(r)
    with RangeCompressor(f, p["na"], p["nr"], "hamming", band) as rc, Plan(p) as plan:
        plan.backproject_raw(img, r, pos, rc)
        rc(comp, r)
        plan.backproject(two, comp, pos)
        torch.cuda.synchronize()
    got = img.cpu().numpy()
    assert np.array_equal(got.view(np.uint64), two.cpu().numpy().view(np.uint64))

    rc_ref = rco.range_compress(raw, ref, "hamming", band).astype(np.complex64)
    want = oracle.backproject(p, rc_ref, pos_np)
    print(parity.assert_parity(got, want, f"raw -> image, nr={nr}"))
    assert not parity.argmax_mismatches(got, want, sc.targets)


def test_raw_entry_point_accumulates_and_checks_plans():
    sc, raw = _raw_scene(512, na=48)
    p = sc.params
    ref = torch.from_numpy(chirp.chirp().astype(np.complex64)).to(DEV)
    r = torch.from_numpy(raw).to(DEV)
    pos = torch.from_numpy(sc.antenna_pos).to(DEV)
    img = torch.zeros((p["ny"], p["nx"]), dtype=torch.complex64, device=DEV)
    with RangeCompressor(ref, p["na"], p["nr"]) as rc, Plan(p) as plan:
        plan.backproject_raw(img, r, pos, rc)
        once = img.clone()
        plan.backproject_raw(img, r, pos, rc, accumulate=True)
        torch.cuda.synchronize()
        assert torch.allclose(img, 2 * once, rtol=1e-6, atol=1e-6 * once.abs().max().item())
        with pytest.raises(SarbpError) as err:
            plan.backproject_raw(img, r, pos, rc, params=dict(p, flags=_native.SARBP_SINC8))
        assert err.value.status == _native.SARBP_ERR_INVALID_ARG
    # a compression plan of another shape
    with RangeCompressor(ref, p["na"], p["nr"] - 1) as rc_other, Plan(p) as plan:
        with pytest.raises(SarbpError) as err:
            plan.backproject_raw(img, r, pos, rc_other)
        assert err.value.status == _native.SARBP_ERR_PLAN_MISMATCH
    # a height-map plan
    with RangeCompressor(ref, p["na"], p["nr"]) as rc, Plan(p, height_range=(0.0, 5.0)) as hplan:
        with pytest.raises(SarbpError) as err:
            hplan.backproject_raw(img, r, pos, rc)
        assert err.value.status == _native.SARBP_ERR_PLAN_MISMATCH
