"""The no-allocation entry point against the plan-based one, through the C-ABI.

sarbp_backproject_noalloc serves callers that cannot allocate device memory
(a plug-in handed only buffers, a framework whose pool owns the GPU, a
real-time loop that forbids cudaMalloc once running). It keeps its scratch in
a fixed device array shared by all calls, so the calls here follow one
another with different sizes: the page-sized scene (two chunks of pulses, the
second one short, 368 table entries per pulse), then the tiny scene (one
chunk, a narrower row), then the page-sized scene again. Each result must
match the plan-based entry point, so nothing one call leaves in the array
may leak into the next. It groups the pulse sum by chunks, so it is compared
with sarbp_backproject within the parity tolerance, not bitwise. A call is
also made with the library's next device allocation armed to fail: it must
succeed and leave that failure unused. This file is named to run last.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

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


def _device(sc):
    e = torch.from_numpy(sc.echoes).to(DEV)
    a = torch.from_numpy(sc.antenna_pos).to(DEV)
    return e, a


def _with_plan(sc, e, a):
    img = torch.empty((sc.params["ny"], sc.params["nx"]), dtype=torch.complex64, device=DEV)
    with Plan(sc.params) as plan:
        plan.backproject(img, e, a)
        torch.cuda.synchronize()
    return img.cpu().numpy()


def _call(img, sc, e, a, flags=0):
    p = _native.Params.from_dict(sc.params, flags=flags)
    stream = torch.cuda.current_stream().cuda_stream
    return _native.lib().sarbp_backproject_noalloc(
        ctypes.c_void_p(img.data_ptr()), ctypes.c_void_p(e.data_ptr()),
        ctypes.c_void_p(a.data_ptr()), ctypes.byref(p), ctypes.c_void_p(stream))


def _no_alloc(sc, e, a, flags=0, init=None):
    img = torch.full((sc.params["ny"], sc.params["nx"]), complex(5.0, 5.0),
                     dtype=torch.complex64, device=DEV)
    if init is not None:
        img.copy_(torch.from_numpy(init))
    st = _call(img, sc, e, a, flags)
    assert st == _native.SARBP_OK, _native.lib().sarbp_status_string(st)
    torch.cuda.synchronize()
    return img.cpu().numpy()


def test_matches_plan_entry_point_across_sizes():
    small = scenes.make_scene(scenes.CONFIGS[0])
    # the page-sized scene needs two chunks of pulses in the 16 MiB scratch
    page = scenes.make_scene(scenes.CONFIGS[2])
    refs, dev = {}, {}
    for sc in (small, page):
        dev[sc.cfg.name] = _device(sc)
        refs[sc.cfg.name] = _with_plan(sc, *dev[sc.cfg.name])
    out = []
    for sc in (page, small, page):
        got = _no_alloc(sc, *dev[sc.cfg.name])
        parity.assert_parity(got, refs[sc.cfg.name], f"{sc.cfg.name} call {len(out) + 1}")
        out.append(got)
    # the same inputs give the same image, whatever ran in between
    assert np.array_equal(out[0].view(np.uint64), out[2].view(np.uint64))


def test_allocates_nothing():
    sc = scenes.make_scene(scenes.CONFIGS[1])
    e, a = _device(sc)
    ref = _with_plan(sc, e, a)
    _no_alloc(sc, e, a)                            # the array is loaded in this context
    lib = _native.lib()
    img = torch.full((sc.params["ny"], sc.params["nx"]), complex(5.0, 5.0),
                     dtype=torch.complex64, device=DEV)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    lib.sarbp_debug_fail_alloc(1)                  # the next device allocation would fail
    try:
        assert _call(img, sc, e, a) == _native.SARBP_OK
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free_before
        # the armed failure is still there: the next plan meets it
        h = ctypes.c_void_p()
        prm = _native.Params.from_dict(sc.params)
        assert lib.sarbp_plan(ctypes.byref(h), ctypes.byref(prm)) == _native.SARBP_ERR_OOM
        assert not h.value
    finally:
        lib.sarbp_debug_fail_alloc(0)
    parity.assert_parity(img.cpu().numpy(), ref, "no-alloc call with allocations armed to fail")


def test_accumulate_and_rejection():
    sc = scenes.make_scene(scenes.CONFIGS[0])
    e, a = _device(sc)
    ref = _with_plan(sc, e, a)
    once = _no_alloc(sc, e, a)
    twice = _no_alloc(sc, e, a, flags=_native.SARBP_ACCUMULATE, init=once)
    parity.assert_parity(twice, 2 * ref.astype(np.complex128), "accumulate")

    # a range axis so long that one pulse's table row cannot fit in the scratch
    big = dict(sc.params, nx=32, ny=32, dr=1e-4, nr=4_000_000, na=1)
    p = _native.Params.from_dict(big)
    img = torch.zeros((32, 32), dtype=torch.complex64, device=DEV)
    st = _native.lib().sarbp_backproject_noalloc(
        ctypes.c_void_p(img.data_ptr()), ctypes.c_void_p(e.data_ptr()),
        ctypes.c_void_p(a.data_ptr()), ctypes.byref(p), None)
    assert st == _native.SARBP_ERR_SCRATCH_TOO_SMALL
    assert b"scratch" in _native.lib().sarbp_status_string(st)
