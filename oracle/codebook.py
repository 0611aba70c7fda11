"""Lloyd-Max codebook for one coordinate of a rotated unit vector.

[Guide] §二 step 2 gives "Lloyd-Max optimal quantisation with a codebook optimal for the Beta
distribution", with codebook files per dimension (64/128/576) and bit width (1..4). After a random
rotation, one coordinate x of a unit vector in R^d has density

    f_d(x) = C_d (1 - x^2)^((d-3)/2)  on [-1, 1],   C_d = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2)),

which is equivalent to x^2 ~ Beta(1/2, (d-1)/2). The codebook with 2^b levels is the fixed point of
Lloyd's two conditions:
* every centroid is the conditional mean of its cell;
* every boundary is the midpoint of its two neighbours.

This module iterates those two conditions with the cell integrals in closed form:
* mass(a, b) = F(b) - F(a), where F is written with the regularised incomplete beta function;
* first moment: int_a^b x f_d(x) dx = C_d [(1-a^2)^((d-1)/2) - (1-b^2)^((d-1)/2)] / (d-1).
"""

import numpy as np
from scipy import special


def _log_norm_const(d):
    return special.gammaln(d / 2.0) - 0.5 * np.log(np.pi) - special.gammaln((d - 1) / 2.0)


def beta_marginal_pdf(x, d):
    """f_d(x) = C_d (1 - x^2)^((d-3)/2) for |x| < 1, else 0."""
    x = np.asarray(x, dtype=np.float64)
    inside = np.abs(x) < 1.0
    out = np.zeros_like(x)
    out[inside] = np.exp(_log_norm_const(d) + (d - 3) / 2.0 * np.log1p(-x[inside] ** 2))
    return out


def _cdf(x, d):
    """P(X <= x) for X ~ f_d: 1/2 + sign(x)/2 * I_{x^2}(1/2, (d-1)/2)."""
    x = np.clip(np.asarray(x, dtype=np.float64), -1.0, 1.0)
    return 0.5 + 0.5 * np.sign(x) * special.betainc(0.5, (d - 1) / 2.0, x * x)


def _first_moment(a, b, d):
    """int_a^b x f_d(x) dx in closed form."""
    e = (d - 1) / 2.0
    c = np.exp(_log_norm_const(d))
    return c * ((1.0 - a * a) ** e - (1.0 - b * b) ** e) / (d - 1)


def lloyd_max_codebook(d, bits, tol=1e-15, max_iter=200000):
    """Return (centroids[2^bits], boundaries[2^bits - 1]), ascending, fp64."""
    levels = 1 << bits
    # start from equal-mass cells of the Gaussian approximation N(0, 1/d)
    from scipy.stats import norm
    edges = norm.ppf(np.linspace(0.0, 1.0, levels + 1)[1:-1]) / np.sqrt(d)
    bounds = np.clip(edges, -0.999, 0.999)
    cent = None
    for _ in range(max_iter):
        lo = np.concatenate([[-1.0], bounds])
        hi = np.concatenate([bounds, [1.0]])
        mass = _cdf(hi, d) - _cdf(lo, d)
        cent = _first_moment(lo, hi, d) / mass
        new_bounds = 0.5 * (cent[:-1] + cent[1:])
        if np.max(np.abs(new_bounds - bounds)) < tol:
            bounds = new_bounds
            break
        bounds = new_bounds
    lo = np.concatenate([[-1.0], bounds])
    hi = np.concatenate([bounds, [1.0]])
    cent = _first_moment(lo, hi, d) / (_cdf(hi, d) - _cdf(lo, d))
    # f_d is even, so the optimal codebook is odd-symmetric; remove the rounding asymmetry so that
    # the middle boundary is exactly 0
    cent = 0.5 * (cent - cent[::-1])
    bounds = 0.5 * (bounds - bounds[::-1])
    return cent, bounds


def mse_distortion(d, centroids, boundaries):
    """E[(X - Q(X))^2] for X ~ f_d under the given quantiser (numerical quadrature)."""
    from scipy import integrate
    lo = np.concatenate([[-1.0], boundaries])
    hi = np.concatenate([boundaries, [1.0]])
    total = 0.0
    for a, b, c in zip(lo, hi, centroids):
        val, _ = integrate.quad(lambda x: (x - c) ** 2 * beta_marginal_pdf(np.array([x]), d)[0], a, b,
                                epsabs=1e-14, epsrel=1e-12, limit=400)
        total += val
    return total
