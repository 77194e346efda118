"""The kernels' softcap polynomial (tanh(y)/y as a cubic in y^2 on |y| <= Y0, used where all
of a warp's scores lie in range) against float64 tanh.  The constants are read from the
kernels' shared header; the evaluation repeats the kernels' float32 Horner order, both in y
and in the folded form in the raw score.  CPU only."""
import math
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "flexible_mask_attention_range_gb300", "csrc", "ffa_internal.h")
LOG2E = 1.4426950408889634


def _constants():
    s = open(SRC).read()
    y0 = float(re.search(r"constexpr double kTanhPolyY = ([0-9.eE+-]+);", s).group(1))
    body = re.search(r"constexpr double kTanhPoly\[4\] = \{([^}]*)\};", s).group(1)
    c = [float(x) for x in body.split(",")]
    assert len(c) == 4
    return y0, c


def _horner32(coef, t):
    w = np.full_like(t, np.float32(coef[3]))
    for ci in (coef[2], coef[1], coef[0]):
        w = (w * t + np.float32(ci)).astype(np.float32)
    return w


def test_polynomial_matches_tanh_on_its_interval():
    y0, c = _constants()
    y = np.linspace(-y0, y0, 400001).astype(np.float32)
    t = (y * y).astype(np.float32)
    r = (y * _horner32(c, t)).astype(np.float64)
    ref = np.tanh(y.astype(np.float64))
    nz = ref != 0
    rel = np.abs(r[nz] - ref[nz]) / np.abs(ref[nz])
    assert rel.max() < 1.6e-7
    assert np.all(r[y == 0] == 0)
    # odd and increasing (the row max is taken at the raw maximum)
    assert np.array_equal(r[::-1], -r)
    assert np.all(np.diff(r) >= -2 * np.spacing(np.abs(r[1:]).astype(np.float32)))


def test_polynomial_differs_from_a_truncated_taylor_series():
    # a fitted (not truncated) series: the Taylor cubic in y^2 is ~1e-5 off at the interval end
    y0, c = _constants()
    taylor = [1.0, -1.0 / 3.0, 2.0 / 15.0, -17.0 / 315.0]
    e_fit = abs(y0 * sum(ci * y0 ** (2 * i) for i, ci in enumerate(c)) - math.tanh(y0))
    e_tay = abs(y0 * sum(ci * y0 ** (2 * i) for i, ci in enumerate(taylor)) - math.tanh(y0))
    assert e_fit < 1e-7 < e_tay


def test_folded_form_in_the_raw_score():
    """x(s) = s * sum_i q_i s^(2i), q_i = C c_i a^(2i+1): the capped logit in the log2 domain,
    C = softcap * log2(e), a = scale / softcap, for |s| <= Y0 / a."""
    y0, c = _constants()
    for scale, cap in ((1 / math.sqrt(128), 30.0), (1 / 8.0, 50.0), (0.05, 50.0), (0.02, 2.0)):
        a = scale / cap
        C = cap * LOG2E
        q = [np.float32(C * ci * a ** (2 * i + 1)) for i, ci in enumerate(c)]
        slim = np.float32(y0 / a * (1 - 1e-6))
        s = np.linspace(-slim, slim, 200001).astype(np.float32)
        t = (s * s).astype(np.float32)
        w = np.full_like(t, q[3])
        for qi in (q[2], q[1], q[0]):
            w = (w * t + qi).astype(np.float32)
        x = (s * w).astype(np.float64)
        ref = C * np.tanh(a * s.astype(np.float64))
        # absolute error of the log2-domain logit: a relative error of p of about 1e-6
        assert np.abs(x - ref).max() < 1e-6 * max(1.0, C * math.tanh(y0))


def test_header_coefficients_are_the_generator_output():
    """The constants in the header are what the committed fitting script produces."""
    from flexible_mask_attention_range_gb300 import fit_tanh_poly as F
    y0, c = _constants()
    assert y0 == F.Y
    fitted = F.fit()
    assert [f"{x:.9e}" for x in fitted] == [f"{x:.9e}" for x in c]


def _constants5():
    s = open(SRC).read()
    body = re.search(r"constexpr double kTanhPoly5\[3\] = \{([^}]*)\};", s).group(1)
    c = [float(x) for x in body.split(",")]
    assert len(c) == 3
    return c


def test_degree5_polynomial_matches_tanh_on_its_interval():
    """kTanhPoly5 (the bounded-softcap forward kernel's form) against float64 tanh, evaluated
    in the kernels' float32 Horner order: within 4.5e-6 relative, odd and increasing."""
    y0, _ = _constants()
    c = _constants5()
    y = np.linspace(-y0, y0, 400001).astype(np.float32)
    t = (y * y).astype(np.float32)
    w = np.full_like(t, np.float32(c[2]))
    for ci in (c[1], c[0]):
        w = (w * t + np.float32(ci)).astype(np.float32)
    r = (y * w).astype(np.float64)
    ref = np.tanh(y.astype(np.float64))
    nz = ref != 0
    rel = np.abs(r[nz] - ref[nz]) / np.abs(ref[nz])
    assert rel.max() < 4.5e-6
    # a fitted, not truncated, series: the Taylor quadratic in y^2 is ~6e-5 off at the end
    taylor = [1.0, -1.0 / 3.0, 2.0 / 15.0]
    e_tay = abs(y0 * sum(ci * y0 ** (2 * i) for i, ci in enumerate(taylor)) - math.tanh(y0)) / math.tanh(y0)
    assert rel.max() < e_tay / 5
    assert np.array_equal(r[::-1], -r)
    assert np.all(np.diff(r) >= -2 * np.spacing(np.abs(r[1:]).astype(np.float32)))


def test_degree5_folded_form_where_the_bounded_softcap_kernel_uses_it():
    """The bounded-softcap kernel runs for softcap * log2(e) <= 60; there the folded degree-5
    form stays within 1e-4 of the exact capped logit (log2 domain), a relative error of p
    below 7e-5 (bf16 P carries 2^-9)."""
    y0, _ = _constants()
    c = _constants5()
    for scale, cap in ((1 / math.sqrt(128), 30.0), (1 / 8.0, 41.0), (0.05, 10.0), (0.02, 2.0)):
        a = scale / cap
        C = cap * LOG2E
        assert 2 * C <= 120
        q = [np.float32(C * ci * a ** (2 * i + 1)) for i, ci in enumerate(c)]
        slim = np.float32(y0 / a * (1 - 1e-6))
        s = np.linspace(-slim, slim, 200001).astype(np.float32)
        t = (s * s).astype(np.float32)
        w = np.full_like(t, q[2])
        for qi in (q[1], q[0]):
            w = (w * t + qi).astype(np.float32)
        x = (s * w).astype(np.float64)
        ref = C * np.tanh(a * s.astype(np.float64))
        assert np.abs(x - ref).max() < 1e-4


def test_degree5_coefficients_are_the_generator_output():
    from flexible_mask_attention_range_gb300 import fit_tanh_poly as F
    c = _constants5()
    fitted = F.fit(degree=3)
    assert [f"{x:.9e}" for x in fitted] == [f"{x:.9e}" for x in c]
