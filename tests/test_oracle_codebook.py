"""Pins for the Lloyd-Max codebook of the rotated-coordinate (Beta) distribution."""
import json
import os

import numpy as np
import pytest
from scipy import integrate, special

from oracle import beta_marginal_pdf, lloyd_max_codebook
from oracle.codebook import mse_distortion

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _quad(f, a, b):
    v, _ = integrate.quad(f, a, b, epsabs=1e-14, epsrel=1e-13, limit=500)
    return v


@pytest.mark.parametrize("d", [64, 128, 256])
def test_density_is_the_unit_sphere_marginal(d):
    pdf = lambda x: beta_marginal_pdf(np.array([x]), d)[0]
    assert abs(_quad(pdf, -1, 1) - 1.0) < 1e-12
    # a coordinate of a uniform unit vector in R^d has E[x^2] = 1/d exactly
    assert abs(_quad(lambda x: x * x * pdf(x), -1, 1) - 1.0 / d) < 1e-13
    # Monte Carlo against uniform points on the sphere
    g = np.random.default_rng(d).standard_normal((20000, d))
    x = (g / np.linalg.norm(g, axis=1, keepdims=True))[:, 0]
    assert abs(np.mean(x ** 4) - _quad(lambda t: t ** 4 * pdf(t), -1, 1)) < 5 * np.std(x ** 4) / np.sqrt(len(x))


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_lloyd_max_fixed_point(d, bits):
    c, t = lloyd_max_codebook(d, bits)
    assert len(c) == 1 << bits and len(t) == (1 << bits) - 1
    assert np.all(np.diff(c) > 0)
    assert np.allclose(c, -c[::-1], atol=1e-15)
    # each boundary is the midpoint of its neighbouring centroids
    assert np.max(np.abs(t - 0.5 * (c[:-1] + c[1:]))) < 1e-13
    # each centroid is the conditional mean of its cell (independent quadrature of the raw density)
    pdf = lambda x: beta_marginal_pdf(np.array([x]), d)[0]
    edges = np.concatenate([[-1.0], t, [1.0]])
    for i in range(len(c)):
        m = _quad(pdf, edges[i], edges[i + 1])
        mean = _quad(lambda x: x * pdf(x), edges[i], edges[i + 1]) / m
        assert abs(mean - c[i]) < 1e-12 * max(1.0, abs(c[i]) * np.sqrt(d))


@pytest.mark.parametrize("d", [64, 128, 256, 1000])
def test_one_bit_closed_form(d):
    c, t = lloyd_max_codebook(d, 1)
    e_abs = np.exp(special.gammaln(d / 2) - special.gammaln((d + 1) / 2)) / np.sqrt(np.pi)
    assert np.allclose(c, [-e_abs, e_abs], rtol=1e-13)
    assert t[0] == 0.0 or abs(t[0]) < 1e-16


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_large_d_limit_is_gaussian_lloyd_max(bits):
    table = np.array(json.load(open(os.path.join(GOLDEN, "gaussian_lloyd_max.json")))["levels"][str(bits)])
    gaps = []
    for d in (512, 2048):
        c, _ = lloyd_max_codebook(d, bits)
        pos = c[len(c) // 2:] * np.sqrt(d)
        gap = np.abs(pos - table)
        # table printed to 4 significant digits; the Beta-vs-Gaussian gap is O(level^2 / d)
        assert np.all(gap < 1e-4 + 3.0 * table ** 2 / d)
        gaps.append(gap.max())
    assert gaps[1] < gaps[0] / 2.5  # the gap shrinks like 1/d


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_distortion_matches_monte_carlo(bits):
    d = 128
    c, t = lloyd_max_codebook(d, bits)
    D = mse_distortion(d, c, t)
    g = np.random.default_rng(bits).standard_normal((4000, d))
    x = (g / np.linalg.norm(g, axis=1, keepdims=True)).ravel()
    idx = np.searchsorted(t, x)
    err = (x - c[idx]) ** 2
    assert abs(err.mean() - D) < 5 * err.std() / np.sqrt(err.size)
    # unit-vector distortion d * D falls as the bit width grows
    assert d * D < {1: 0.37, 2: 0.12, 3: 0.035, 4: 0.0095}[bits]
