"""The FP64 range-compression oracle against facts fixed outside itself."""

import numpy as np
import pytest

from oracle import range_compression as rc
from synth import chirp


def test_equals_direct_correlation_on_small_sizes():
    rng = np.random.default_rng(0)
    raw = rng.standard_normal((3, 40)) + 1j * rng.standard_normal((3, 40))
    ref = rng.standard_normal(9) + 1j * rng.standard_normal(9)
    got = rc.range_compress(raw, ref)
    want = rc.direct_correlation(raw, ref)
    assert np.abs(got - want).max() < 1e-12 * np.abs(want).max()


def test_integer_delay_peak_closed_form():
    ref = chirp.chirp()
    ns, delay, amp = 2048, 700, 0.8 - 0.3j
    raw = np.zeros((1, ns), dtype=np.complex128)
    raw[0, delay:delay + ref.size] = amp * ref
    out = rc.range_compress(raw, ref)[0]
    assert int(np.argmax(np.abs(out))) == delay
    want = amp * np.sum(np.abs(ref) ** 2)
    assert abs(out[delay] - want) < 1e-9 * abs(want)


def test_shift_equivariance_and_linearity():
    rng = np.random.default_rng(1)
    ref = chirp.chirp()[:64]
    a = rng.standard_normal((2, 300)) + 1j * rng.standard_normal((2, 300))
    b = rng.standard_normal((2, 300)) + 1j * rng.standard_normal((2, 300))
    lin = rc.range_compress(2 * a - 1j * b, ref, "hamming", 0.8)
    assert np.allclose(lin, 2 * rc.range_compress(a, ref, "hamming", 0.8)
                       - 1j * rc.range_compress(b, ref, "hamming", 0.8), atol=1e-10)
    shifted = np.zeros_like(a)
    shifted[:, 5:] = a[:, :-5]
    x = rc.range_compress(a, ref)
    y = rc.range_compress(shifted, ref)
    # the first ns - 5 - L outputs see no boundary and are shifted copies
    assert np.allclose(y[:, 5:300 - 64], x[:, :300 - 5 - 64], atol=1e-10)


def _profile(window, over=8):
    """Compressed point response, band-limited-interpolated 8x (the samples alone,
    1.2 per resolution cell, do not resolve the sidelobes)."""
    ref = chirp.chirp()
    ns, delay = 4096, 1500
    raw = np.zeros((1, ns), dtype=np.complex128)
    raw[0, delay:delay + ref.size] = ref
    band = chirp.BANDWIDTH / (chirp.C_LIGHT / (2 * chirp.DR))
    out = rc.range_compress(raw, ref, window, band)[0]
    spec = np.fft.fft(out)
    half = ns // 2
    padded = np.concatenate([spec[:half], np.zeros((over - 1) * ns), spec[half:]])
    fine = np.abs(np.fft.ifft(padded)) * over
    return fine, delay * over


def _mainlobe_and_sidelobe(prof, peak_at):
    p = prof / prof[peak_at]
    # first nulls (local minima) around the peak
    left = peak_at
    while p[left - 1] < p[left]:
        left -= 1
    right = peak_at
    while p[right + 1] < p[right]:
        right += 1
    side = max(p[:left].max(), p[right + 1:].max())
    # -3 dB width by linear interpolation of the power profile
    thr = 1 / np.sqrt(2)
    def cross(i, step):
        while p[i] >= thr:
            i += step
        j = i - step
        return j + step * (p[j] - thr) / (p[j] - p[i])
    width = cross(peak_at, 1) - cross(peak_at, -1)
    return 20 * np.log10(side), width


def test_sidelobes_and_mainlobe_match_the_page():
    # SARBP-GPU §3.1: plain matched filtering leaves sidelobes near -13 dB; a
    # Hamming window lowers them and widens the mainlobe by about 1.3-1.5x
    rect, d = _profile("none")
    ham, _ = _profile("hamming")
    psl_rect, w_rect = _mainlobe_and_sidelobe(rect, d)
    psl_ham, w_ham = _mainlobe_and_sidelobe(ham, d)
    assert -14.5 < psl_rect < -12.0, psl_rect
    assert psl_ham < -30.0, psl_ham
    assert 1.3 <= w_ham / w_rect <= 1.55, w_ham / w_rect
    # -3 dB width without a window: 0.886 of the resolution cell c / 2B, in samples
    cell = (chirp.C_LIGHT / (2 * chirp.BANDWIDTH)) / chirp.DR
    assert abs(w_rect / 8 / (0.886 * cell) - 1) < 0.05


def _taylor_pattern(u, coeffs):
    """Far-field pattern of w(x) = 1 + 2 sum F_m cos(2 pi m x) over |x| <= 1/2:
    sinc(u) + sum F_m (sinc(u - m) + sinc(u + m)), closed form."""
    out = np.sinc(u).astype(float)
    for m, f in enumerate(coeffs, start=1):
        out += f * (np.sinc(u - m) + np.sinc(u + m))
    return out


def pin_taylor(coeffs):
    """Taylor's construction puts the first nbar - 1 pattern zeros at
    u_n = sigma sqrt(A^2 + (n - 1/2)^2) and the sidelobes near the design level."""
    nbar, sll = rc.TAYLOR_NBAR, rc.TAYLOR_SLL_DB
    a = np.arccosh(10 ** (sll / 20)) / np.pi
    sigma2 = nbar ** 2 / (a ** 2 + (nbar - 0.5) ** 2)
    zeros = [np.sqrt(sigma2 * (a ** 2 + (n - 0.5) ** 2)) for n in range(1, nbar)]
    p0 = _taylor_pattern(np.array([0.0]), coeffs)[0]
    at_zeros = np.abs(_taylor_pattern(np.array(zeros), coeffs)) / p0
    u = np.linspace(zeros[0], 12.0, 100001)
    psl = 20 * np.log10(np.abs(_taylor_pattern(u, coeffs)).max() / p0)
    return bool(at_zeros.max() < 1e-9 and -35.5 < psl < -34.5), (at_zeros.max(), psl)


def test_taylor_window_meets_its_design():
    # SARBP-GPU §3.1 names Taylor beside Hamming. Taylor's weighting, nbar = 5,
    # 35 dB: exact pattern zeros and sidelobes at the design level; on the
    # compressed chirp (time-bandwidth 300, whose spectrum ripples) the peak
    # sidelobe stays below -32 dB and the mainlobe widens less than with Hamming.
    ok, detail = pin_taylor(rc.taylor_coefficients())
    assert ok, detail
    tay, d = _profile("taylor")
    rect, _ = _profile("none")
    ham, _ = _profile("hamming")
    psl_t, w_t = _mainlobe_and_sidelobe(tay, d)
    _, w_r = _mainlobe_and_sidelobe(rect, d)
    _, w_h = _mainlobe_and_sidelobe(ham, d)
    assert psl_t < -32.0, psl_t
    assert w_r < w_t < w_h, (w_r, w_t, w_h)
    x = (np.arange(100000) + 0.5) / 100000 - 0.5
    fm = rc.taylor_coefficients()
    w = 1 + 2 * sum(f * np.cos(2 * np.pi * (m + 1) * x) for m, f in enumerate(fm))
    assert abs(w.mean() - 1.0) < 1e-9
    assert np.allclose(w, w[::-1])


@pytest.mark.parametrize("slip", ["sign", "sigma_dropped", "half_factor"])
def test_taylor_pin_rejects_plausible_slips(slip):
    good = rc.taylor_coefficients()
    if slip == "sign":                     # (-1)^m for (-1)^(m+1)
        bad = -good
    elif slip == "sigma_dropped":          # the stretch sigma^2 left out
        nbar, a = rc.TAYLOR_NBAR, np.arccosh(10 ** (rc.TAYLOR_SLL_DB / 20)) / np.pi
        bad = np.array([(-1.0) ** (m + 1) * np.prod([1 - m ** 2 / (a ** 2 + (i - 0.5) ** 2)
                                                      for i in range(1, nbar)])
                        / (2 * np.prod([1 - m ** 2 / i ** 2 for i in range(1, nbar) if i != m]))
                        for m in range(1, nbar)])
    else:                                  # the 1/2 of the denominator left out
        bad = 2 * good
    assert not pin_taylor(bad)[0], slip


def test_raw_generator_compresses_to_target_range():
    pos = np.array([[0.0, -7000.0, 5000.0]])
    tgt = np.array([[0.0, 0.0, 0.0]])
    r = np.linalg.norm(pos[0] - tgt[0])
    r0 = r - 1000 * chirp.DR
    raw = chirp.raw_echoes(pos, tgt, np.array([1.0]), r0, 2048)
    out = rc.range_compress(raw, chirp.chirp())[0]
    k = int(np.argmax(np.abs(out)))
    assert abs(k - 1000) <= 1
    # at the peak the carrier phase -4 pi R / lambda survives compression
    # (within the chirp's residual phase at a fractional delay)
    assert abs(np.angle(out[1000] * np.exp(1j * 4 * np.pi * r / chirp.WAVELENGTH))) < 0.2
