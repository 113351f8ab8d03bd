"""The oracle's pins (tests/pins.py), run on the CUDA path.

The pins hold for the method itself, whatever computes it: the closed form at
an isolated target (SARBP-GPU §1.1, §4.2), a zero image from zero echoes,
linearity in the echoes, independence from the pulse order, focusing at the
true pixel (§3.2, §4.2), mirror symmetry of a centred target under a
symmetric track, and the textbook point-response widths. Here they are
checked on the library's float32 output, with tolerances set by float32
rounding (relative 1e-4 for the closed form, 1e-5 for the identities) instead
of the oracle's float64 ones.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from domain_backprojection_sarbp_gb300 import Plan  # noqa: E402
from tests import pins  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


def gpu_bp(interp):
    def bp(params, echo, pos, pixels):
        img = torch.zeros((params["ny"], params["nx"]), dtype=torch.complex64, device=DEV)
        with Plan(params) as plan:
            plan.backproject(img, torch.from_numpy(np.ascontiguousarray(echo, dtype=np.complex64)).to(DEV),
                             torch.from_numpy(np.ascontiguousarray(pos, dtype=np.float64)).to(DEV),
                             interp=interp)
            torch.cuda.synchronize()
        out = img.cpu().numpy().astype(np.complex128)
        return out if pixels is None else out.reshape(-1)[pixels]
    return bp


CASES = [
    ("closed_form", lambda bp: pins.pin_closed_form(bp, tol=1e-4)),
    ("zero_echo", pins.pin_zero_echo),
    ("linearity", lambda bp: pins.pin_linearity(bp, tol=1e-5)),
    ("pulse_permutation", lambda bp: pins.pin_pulse_permutation(bp, tol=1e-5)),
    ("focusing", pins.pin_focusing),
    ("mirror_symmetry", lambda bp: pins.pin_mirror_symmetry(bp, tol=1e-5)),
    ("resolution", pins.pin_resolution),
]


@pytest.mark.parametrize("name,pin", CASES, ids=[c[0] for c in CASES])
def test_pin_on_the_linear_path(name, pin):
    ok, detail = pin(gpu_bp("linear"))
    print(name, detail)
    assert ok, f"{name}: {detail}"


@pytest.mark.parametrize("name,pin", [c for c in CASES if c[0] in
                                      ("zero_echo", "linearity", "pulse_permutation",
                                       "mirror_symmetry")], ids=lambda c: c if isinstance(c, str) else "")
@pytest.mark.parametrize("interp", ["sinc8", "nearest"])
def test_identities_on_the_other_interpolations(name, pin, interp):
    ok, detail = pin(gpu_bp(interp))
    print(name, interp, detail)
    assert ok, f"{name} ({interp}): {detail}"
