"""CPU checks of the softcap's tanh polynomial (the constants the bf16 forward
kernel evaluates on the FMA pipes when every score of a tile is in range)."""
import math
import os
import re

import numpy as np

from softmax_attention_attn_gb300 import tanh_fit

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KERNEL = os.path.join(ROOT, "softmax_attention_attn_gb300", "csrc", "attn_fwd_bf16.cu")


def _source_constants():
    src = open(KERNEL).read()
    body = re.search(r"kTanhPoly\[6\]\s*=\s*\{([^}]*)\}", src).group(1)
    ymax = float(re.search(r"kTanhPolyYMax\s*=\s*([0-9.eE+-]+);", src).group(1))
    return np.array([float(x) for x in body.split(",")]), ymax


def test_kernel_constants_are_the_remez_fit():
    coef, ymax = _source_constants()
    fit, err = tanh_fit.remez()
    assert ymax == tanh_fit.Y_MAX and coef.size == tanh_fit.DEGREE + 1
    np.testing.assert_allclose(coef, fit, rtol=1e-12, atol=1e-15)
    assert err < 6e-7


def test_fp32_evaluation_meets_the_stated_bound():
    coef, ymax = _source_constants()
    assert tanh_fit.fp32_horner_rel_err(coef, ymax) <= tanh_fit.MAX_REL_ERR


def test_polynomial_against_math_tanh_at_chosen_points():
    """Independent spot checks (math.tanh in double): zero, tiny, mid-range, the range end."""
    coef, _ = _source_constants()
    for y in (0.0, 1e-6, 0.01, 0.25, 0.5, 0.75, 0.999, 1.0, -0.3, -1.0):
        approx = y * sum(c * (y * y) ** k for k, c in enumerate(coef))
        exact = math.tanh(y)
        assert abs(approx - exact) <= 6e-7 * max(abs(exact), 1e-300), (y, approx, exact)


def test_the_fit_equioscillates():
    """A minimax fit's error reaches its maximum, with alternating signs, at DEGREE + 2 points."""
    coef, _ = tanh_fit.remez()
    z = np.linspace(0, tanh_fit.Y_MAX ** 2, 200001)
    t = tanh_fit.tanh_over_y(z)
    err = (np.polyval(coef[::-1], z) - t) / t
    E = np.abs(err).max()
    cuts = np.flatnonzero(np.diff(np.sign(err)) != 0) + 1
    peaks = [np.abs(err[seg]).max() for seg in np.split(np.arange(z.size), cuts)]
    assert sum(p > 0.99 * E for p in peaks) >= tanh_fit.DEGREE + 2
