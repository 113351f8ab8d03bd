"""The error figure behind the windowed-sinc kernel's per-bin polynomials.

The CUDA table stores, for each range bin, the interpolant G on that bin as a
degree-7 polynomial: each of the eight tap weights h(1/2 + s - d), d = -3..4,
h(t) = sinc(t) (1 + cos(pi t / 4)) / 2, is replaced by its interpolant at the
eight Chebyshev nodes of the bin. Here, in float64 and independently of the
library, the summed error of the eight interpolants (the bound on |dG| per
unit sample magnitude) is checked to be the 5.2e-6 the kernel's comments
state, and the next lower degree is shown not to meet the 4e-5 budget the
thread-level polynomial modes use.
"""

import numpy as np


def _h(t):
    return np.sinc(t) * 0.5 * (1.0 + np.cos(np.pi * t / 4.0))


def _summed_error(degree):
    s = np.linspace(-0.5, 0.5, 20001)
    i = np.arange(degree + 1)
    nodes = 0.5 * np.cos((2 * i + 1) * np.pi / (2 * degree + 2))
    total = 0.0
    for d in range(-3, 5):
        coef = np.linalg.solve(np.vander(nodes, increasing=True), _h(0.5 + nodes - d))
        fit = np.polynomial.polynomial.polyval(s, coef)
        total += np.max(np.abs(fit - _h(0.5 + s - d)))
    return total


def test_degree_seven_error_bound():
    err = _summed_error(7)
    assert 4.5e-6 < err < 6.0e-6, err


def test_degree_six_would_not_meet_the_budget():
    assert _summed_error(6) > 4e-5
