"""Acceptance of a GPU image against the FP64 oracle.

Tolerances: relative L2 <= 1e-3 over the compared pixels, max |error| <=
1e-3 of the oracle's peak, and the same argmax pixel in every target's 9 x 9
neighbourhood. The argmax is compared where it is unique: when the oracle's
two largest values in a window differ by less than ARGMAX_TIE of the peak,
either of them is accepted.
"""

from __future__ import annotations

import numpy as np

REL_L2 = 1e-3
MAX_ERR = 1e-3
ARGMAX_TIE = 2e-4


def compare(got: np.ndarray, ref: np.ndarray) -> dict:
    got = np.asarray(got, dtype=np.complex128).reshape(-1)
    ref = np.asarray(ref, dtype=np.complex128).reshape(-1)
    err = np.abs(got - ref)
    nref = np.linalg.norm(ref)
    peak = np.abs(ref).max() if ref.size else 0.0
    return dict(rel_l2=float(np.linalg.norm(got - ref) / nref) if nref > 0 else float(err.max(initial=0)),
                max_err=float(err.max(initial=0) / peak) if peak > 0 else float(err.max(initial=0)),
                finite=bool(np.all(np.isfinite(got))))


def argmax_mismatches(got_img, ref_img, targets, halo=4):
    """Targets whose GPU argmax differs from the oracle's (beyond ties)."""
    bad = []
    for ix, iy in targets:
        g = np.abs(got_img[iy - halo:iy + halo + 1, ix - halo:ix + halo + 1]).reshape(-1)
        r = np.abs(ref_img[iy - halo:iy + halo + 1, ix - halo:ix + halo + 1]).reshape(-1)
        gi = int(np.argmax(g))
        order = np.argsort(r)[::-1]
        best = r[order[0]]
        tied = [int(i) for i in order if best - r[i] <= ARGMAX_TIE * best]
        if gi not in tied:
            bad.append((int(ix), int(iy), gi, int(order[0])))
    return bad


def assert_parity(got, ref, label=""):
    m = compare(got, ref)
    assert m["finite"], f"{label}: non-finite values"
    assert m["rel_l2"] <= REL_L2, f"{label}: relative L2 {m['rel_l2']:.3e} > {REL_L2}"
    assert m["max_err"] <= MAX_ERR, f"{label}: max error/peak {m['max_err']:.3e} > {MAX_ERR}"
    return m
