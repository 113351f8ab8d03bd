"""Host entry point with pinned buffers the device can address directly.

sarbp_backproject_host reads the echo band and writes the image in place when
the caller's buffers are pinned and mapped (no staging copies); pageable
buffers are staged through device memory. Only the transport differs, so
both must give the same image bit for bit, and the pinned path must match
the FP64 oracle under the usual tolerances (tests/parity.py).
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from domain_backprojection_sarbp_gb300 import Plan  # noqa: E402
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
def scene():
    return scenes.make_scene(scenes.CONFIGS[1])


def pinned(a):
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def run(plan, img, echoes, pos, accumulate=False):
    plan.backproject_host(img, echoes, pos, accumulate=accumulate)
    return img.numpy() if hasattr(img, "numpy") else img


@pytest.mark.parametrize("which", ["both", "echoes", "image"])
def test_pinned_equals_pageable(scene, which):
    p = scene.params
    shape = (p["ny"], p["nx"])
    with Plan(p) as plan:
        ref = run(plan, np.zeros(shape, np.complex64), scene.echoes, scene.antenna_pos)
        ref_bytes = plan.host_transfer_bytes()
        img = pinned(np.full(shape, 3 + 1j, np.complex64)) if which in ("both", "image") else \
            np.full(shape, 3 + 1j, np.complex64)
        ech = pinned(scene.echoes) if which in ("both", "echoes") else scene.echoes
        got = run(plan, img, ech, pinned(scene.antenna_pos))
        assert plan.host_transfer_bytes() == ref_bytes
    assert np.array_equal(got, ref), which


@pytest.mark.parametrize("interp", ["sinc8", "nearest"])
def test_pinned_equals_pageable_other_interpolations(scene, interp):
    p = scene.params
    shape = (p["ny"], p["nx"])
    with Plan(p) as plan:
        ref = np.zeros(shape, np.complex64)
        plan.backproject_host(ref, scene.echoes, scene.antenna_pos, interp=interp)
        got = pinned(np.zeros(shape, np.complex64))
        plan.backproject_host(got, pinned(scene.echoes), pinned(scene.antenna_pos), interp=interp)
    assert np.array_equal(got.numpy(), ref), interp


def test_pinned_accumulate(scene):
    p = scene.params
    rng = np.random.default_rng(4)
    init = (rng.standard_normal((p["ny"], p["nx"])) +
            1j * rng.standard_normal((p["ny"], p["nx"]))).astype(np.complex64)
    with Plan(p) as plan:
        ref = run(plan, init.copy(), scene.echoes, scene.antenna_pos, accumulate=True)
        got = run(plan, pinned(init), pinned(scene.echoes), pinned(scene.antenna_pos),
                  accumulate=True)
    assert np.array_equal(got, ref)


def test_pinned_matches_the_oracle(scene):
    p = scene.params
    with Plan(p) as plan:
        got = run(plan, pinned(np.zeros((p["ny"], p["nx"]), np.complex64)), pinned(scene.echoes),
                  pinned(scene.antenna_pos))
    ref = oracle.backproject(p, scene.echoes, scene.antenna_pos)
    print(parity.assert_parity(got, ref, "pinned host buffers"))
    assert not parity.argmax_mismatches(got, ref, scene.targets)


def test_pinned_no_pulse_reaches_the_image(scene):
    """Antennas beyond the range axis: nothing runs, the image is zeroed."""
    p = scene.params
    pos = scene.antenna_pos.copy()
    pos[:, 2] += 1.0e6
    img = pinned(np.full((p["ny"], p["nx"]), 5 - 2j, np.complex64))
    with Plan(p) as plan:
        got = run(plan, img, pinned(scene.echoes), pinned(pos))
    assert not got.any()


def test_wrong_host_dtype_is_rejected(scene):
    p = scene.params
    with Plan(p) as plan:
        with pytest.raises(ValueError):
            plan.backproject_host(torch.zeros((p["ny"], p["nx"]), dtype=torch.complex128),
                                  scene.echoes, scene.antenna_pos)
