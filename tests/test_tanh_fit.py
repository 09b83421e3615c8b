"""CPU checks of the softcap's tanh polynomials (the constants the bf16 forward
kernel evaluates on the FMA pipes when every score of a tile is in range)."""
import math
import os
import re

import numpy as np
import pytest

from softmax_attention_attn_gb300 import tanh_fit

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KERNEL = os.path.join(ROOT, "softmax_attention_attn_gb300", "csrc", "attn_fwd_bf16.cu")


def _source_constants(name):
    src = open(KERNEL).read()
    tag = name.capitalize()
    body = re.search(r"kTanhPoly%s\[\d+\]\s*=\s*\{([^}]*)\}" % tag, src).group(1)
    ymax = float(re.search(r"kTanhPoly%sYMax\s*=\s*([0-9.eE+-]+);" % tag, src).group(1))
    return np.array([float(x) for x in body.split(",")]), ymax


@pytest.mark.parametrize("name", sorted(tanh_fit.FITS))
def test_kernel_constants_are_the_remez_fit(name):
    coef, ymax = _source_constants(name)
    deg, fit_ymax = tanh_fit.FITS[name]
    fit, err = tanh_fit.remez(deg, fit_ymax)
    assert ymax == fit_ymax and coef.size == deg + 1
    np.testing.assert_allclose(coef, fit, rtol=1e-12, atol=1e-15)
    assert err < 6e-7


@pytest.mark.parametrize("name", sorted(tanh_fit.FITS))
def test_fp32_evaluation_meets_the_stated_bound(name):
    coef, ymax = _source_constants(name)
    assert tanh_fit.fp32_horner_rel_err(coef, ymax) <= tanh_fit.MAX_REL_ERR


@pytest.mark.parametrize("name", sorted(tanh_fit.FITS))
def test_polynomial_against_math_tanh_at_chosen_points(name):
    """Independent spot checks (math.tanh in double): zero, tiny, mid-range, the range ends."""
    coef, ymax = _source_constants(name)
    for f in (0.0, 1e-6, 0.01, 0.25, 0.5, 0.9, 0.999, 1.0, -0.3, -1.0):
        y = f * ymax
        approx = y * sum(c * (y * y) ** k for k, c in enumerate(coef))
        exact = math.tanh(y)
        assert abs(approx - exact) <= 6e-7 * max(abs(exact), 1e-300), (y, approx, exact)


@pytest.mark.parametrize("name", sorted(tanh_fit.FITS))
def test_the_fit_equioscillates(name):
    """A minimax fit's error reaches its maximum, with alternating signs, at degree + 2 points."""
    deg, ymax = tanh_fit.FITS[name]
    coef, _ = tanh_fit.remez(deg, ymax)
    z = np.linspace(0, ymax ** 2, 200001)
    t = tanh_fit.tanh_over_y(z)
    err = (np.polyval(coef[::-1], z) - t) / t
    E = np.abs(err).max()
    cuts = np.flatnonzero(np.diff(np.sign(err)) != 0) + 1
    peaks = [np.abs(err[seg]).max() for seg in np.split(np.arange(z.size), cuts)]
    assert sum(p > 0.99 * E for p in peaks) >= deg + 2
