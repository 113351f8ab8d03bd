"""The error figures behind the windowed-sinc kernel's polynomials.

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


def _tap_derivative_sum(n):
    """max over f of sum_d |h^(n)(f - d)|, d = -3..4: bounds |G^(n)| / max|e|."""
    # the symbolic derivative cancels badly near t = 0 in float64: 30 digits
    sympy = __import__("pytest").importorskip("sympy")
    import mpmath
    mpmath.mp.dps = 30
    t = sympy.symbols("t", real=True)
    h = sympy.sin(sympy.pi * t) / (sympy.pi * t) * (1 + sympy.cos(sympy.pi * t / 4)) / 2
    d = sympy.lambdify(t, sympy.diff(h, t, n), "mpmath")
    f = np.linspace(0.0005, 0.9995, 300)
    return float(max(sum(abs(d(mpmath.mpf(float(x)) - k)) for k in range(-3, 5)) for x in f))


def test_thread_polynomial_bounds_at_the_kernel_spans():
    """The thread-level interpolants the kernel uses: degree 4 on spans up to
    0.34 bin, degree 3 up to 0.17 bin and degree 2 up to 0.05 bin. With the
    window's own derivative sums (31 for n = 3, 98 for n = 4, 312 for n = 5)
    the Chebyshev bounds stay under the 4e-5 budget; the bare 8 pi^n bound
    would not allow these spans."""
    s3, s4, s5 = _tap_derivative_sum(3), _tap_derivative_sum(4), _tap_derivative_sum(5)
    assert 30 < s3 < 32.5 and 95 < s4 < 101 and 305 < s5 < 318, (s3, s4, s5)
    quartic = s5 * 0.17 ** 5 / (2 ** 4 * 120)
    cubic = s4 * 0.085 ** 4 / (2 ** 3 * 24)
    quadratic = s3 * 0.025 ** 3 / (2 ** 2 * 6)       # spans up to 0.05 bin
    assert quartic < 2.5e-5 and cubic < 2.8e-5 and quadratic < 2.1e-5, (quartic, cubic, quadratic)
    assert 8 * np.pi ** 5 * 0.17 ** 5 / (2 ** 4 * 120) > 4e-5


def test_wide_kernel_polynomial_bounds():
    """The wide-geometry kernel's higher degrees: degree 5 on six nodes up to
    0.56 bin and degree 6 on seven nodes up to 0.80 bin. The window's
    derivative sums (1007 for n = 6, 3199 for n = 7) keep the Chebyshev bounds
    within one bin under 2.2e-5, the budget of the lower degrees."""
    s6, s7 = _tap_derivative_sum(6), _tap_derivative_sum(7)
    assert 990 < s6 < 1025 and 3140 < s7 < 3260, (s6, s7)
    quintic = s6 * 0.28 ** 6 / (2 ** 5 * 720)
    sextic = s7 * 0.40 ** 7 / (2 ** 6 * 5040)
    assert quintic < 2.2e-5 and sextic < 1.7e-5, (quintic, sextic)


def _window_g(u, e):
    k = np.floor(u).astype(int)
    out = np.zeros(u.shape, complex)
    for d in range(-3, 5):
        t = u - (k + d)
        out += e[k + d] * _h(t)
    return out


def test_thread_polynomial_across_a_bin_boundary():
    """Where the interval crosses a bin boundary G is only C^2 (a tap enters
    the stencil, another leaves), so the derivative bound does not apply;
    measured on random samples (|e| <= 1) the interpolants of every degree the
    kernels use, at their widest spans, stay under 4e-5."""
    rng = np.random.default_rng(7)
    worst = {}
    for nn, span in ((4, 0.17), (5, 0.34), (6, 0.56), (7, 0.80)):
        i = np.arange(nn)
        x = np.cos((2 * i + 1) * np.pi / (2 * nn))
        w = 0.0
        for _ in range(400):
            e = np.exp(2j * np.pi * rng.random(64)) * rng.random(64) ** 0.2
            base = 20 + rng.integers(0, 20)
            mid = base + (rng.random() - 0.5) * span          # straddles bin `base`
            nodes = mid + 0.5 * span * x
            g = _window_g(nodes, e)
            v = np.vander(x, nn, increasing=True)
            cr, ci = np.linalg.solve(v, g.real), np.linalg.solve(v, g.imag)
            uu = np.linspace(mid - 0.5 * span, mid + 0.5 * span, 101)
            tt = (uu - mid) / (0.5 * span)
            p = (np.polynomial.polynomial.polyval(tt, cr)
                 + 1j * np.polynomial.polynomial.polyval(tt, ci))
            w = max(w, np.abs(p - _window_g(uu, e)).max())
        worst[nn] = w
    assert all(w < 4e-5 for w in worst.values()), worst


def test_library_tap_polynomials():
    """The coefficients the CUDA library builds its sinc table from
    (sarbp_debug_sinc_taps, host code, no GPU needed) reproduce each tap weight
    h(1/2 + s - d) on a fine grid: the eight errors sum to under 5.5e-6 (the
    figure the kernel's comments and the design state), and they match a
    float64 fit at the same nodes to float32 rounding."""
    import ctypes
    from domain_backprojection_sarbp_gb300 import _native, build
    build.build()                      # the library builds and loads without a GPU
    lib = _native.lib()
    out = (ctypes.c_float * 64)()
    assert lib.sarbp_debug_sinc_taps(out) == _native.SARBP_OK
    assert lib.sarbp_debug_sinc_taps(None) == _native.SARBP_ERR_INVALID_ARG
    c = np.frombuffer(out, dtype=np.float32).reshape(8, 8).astype(np.float64)
    s = np.linspace(-0.5, 0.5, 20001)
    total = 0.0
    i = np.arange(8)
    nodes = 0.5 * np.cos((2 * i + 1) * np.pi / 16)
    for row, d in enumerate(range(-3, 5)):
        fit = np.polynomial.polynomial.polyval(s, c[row])
        total += np.max(np.abs(fit - _h(0.5 + s - d)))
        ref = np.linalg.solve(np.vander(nodes, increasing=True), _h(0.5 + nodes - d))
        assert np.allclose(c[row], ref, rtol=1e-6, atol=1e-6), (d, c[row], ref)
    assert total < 5.5e-6, total
