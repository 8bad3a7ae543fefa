"""Beta sphere-marginal density and its Lloyd-Max scalar codebook (float64).

[TQ-KV] "Marco Teórico": a coordinate u_1 of a vector drawn uniformly on the
sphere S^{d-1} has (u_1 + 1) / 2 ~ Beta((d-1)/2, (d-1)/2), tending to a
Gaussian as d grows.  [ABL] "Configuração Experimental" (TurboQuant item):
the rotated coordinates are quantized with a data-oblivious Beta Lloyd-Max
codebook.  [TQ-KV] "Esquemas de Cuantización" item 1 names the scalar quantizer
"MSE (Lloyd-Max)".

Reading: the Beta law is taken on [0, 1] for t = (x + 1) / 2, i.e. the density
of x on [-1, 1] is f(x) = (1 - x^2)^((d-3)/2) / B(1/2, (d-1)/2).  This is the
only support under which the statement about a unit vector's coordinate holds.
"""

import numpy as np
from scipy import special


def _a(d):
    return (d - 1) / 2.0


def density(x, d):
    """f(x) on [-1, 1] for a coordinate of a uniform unit vector ([TQ-KV] "Marco Teórico")."""
    x = np.asarray(x, dtype=np.float64)
    return (1.0 - x * x) ** ((d - 3) / 2.0) / special.beta(0.5, _a(d))


def cdf(x, d):
    """P(u_1 <= x) = I_{(x+1)/2}(a, a), a = (d-1)/2 (regularized incomplete beta)."""
    a = _a(d)
    return special.betainc(a, a, (np.asarray(x, dtype=np.float64) + 1.0) / 2.0)


def survival(x, d):
    """P(u_1 > x), computed from the mirror image so that upper tails keep precision."""
    a = _a(d)
    return special.betainc(a, a, (1.0 - np.asarray(x, dtype=np.float64)) / 2.0)


def cell_mass(lo, hi, d):
    """Integral of f over [lo, hi] (vectorized); upper cells use the survival function."""
    lo = np.asarray(lo, dtype=np.float64)
    hi = np.asarray(hi, dtype=np.float64)
    upper = survival(lo, d) - survival(hi, d)
    lower = cdf(hi, d) - cdf(lo, d)
    middle = 1.0 - cdf(lo, d) - survival(hi, d)
    return np.where(lo >= 0.0, upper, np.where(hi <= 0.0, lower, middle))


def cell_first_moment(lo, hi, d):
    """Integral of x f(x) over [lo, hi] in closed form.

    d/dx [-(1 - x^2)^((d-1)/2) / (d - 1)] = x (1 - x^2)^((d-3)/2).
    """
    lo = np.asarray(lo, dtype=np.float64)
    hi = np.asarray(hi, dtype=np.float64)
    p = (d - 1) / 2.0
    # (1 - lo^2)^p - (1 - hi^2)^p, written as A * (1 - exp(p * (log(1 - hi^2) - log(1 - lo^2))))
    # so that narrow cells do not lose digits to cancellation.
    with np.errstate(divide="ignore"):
        log_lo = np.log1p(-lo * lo)
        log_hi = np.log1p(-hi * hi)
    a_lo = np.exp(p * log_lo)
    a_hi = np.exp(p * log_hi)
    lead = np.where(np.abs(lo) <= np.abs(hi), a_lo, a_hi)
    sign = np.where(np.abs(lo) <= np.abs(hi), 1.0, -1.0)
    with np.errstate(invalid="ignore"):
        diff = np.where(np.abs(lo) <= np.abs(hi), log_hi - log_lo, log_lo - log_hi)
        num = sign * lead * -np.expm1(p * diff)
    num = np.where(np.isfinite(num), num, a_lo - a_hi)
    return num / ((d - 1) * special.beta(0.5, _a(d)))


def lloyd_max(d, bits, tol=1e-13, max_iter=100000):
    """Lloyd-Max codebook for the sphere-coordinate density ([ABL] "Configuração Experimental").

    Steps, in the order of the Lloyd-Max conditions:
      1. start from the density's quantiles at (k + 1/2) / L, L = 2**bits;
      2. thresholds are the midpoints of neighbouring centroids;
      3. each centroid is the conditional mean of its cell;
      4. repeat 2-3 until no centroid moves by tol (1e-13: float64 evaluation
         of the cell moments jitters at about 5e-15 for d = 1024, so a tighter
         stop is never reached); finally make the codebook exactly odd-symmetric
         (the density is even).
    Returns (centroids, thresholds), float64, ascending; len L and L - 1.
    """
    L = 1 << bits
    a = _a(d)
    c = 2.0 * special.betaincinv(a, a, (np.arange(L) + 0.5) / L) - 1.0
    for _ in range(max_iter):
        t = 0.5 * (c[:-1] + c[1:])
        edges = np.concatenate([[-1.0], t, [1.0]])
        new = cell_first_moment(edges[:-1], edges[1:], d) / cell_mass(edges[:-1], edges[1:], d)
        moved = np.max(np.abs(new - c))
        c = new
        if moved < tol:
            break
    c = 0.5 * (c - c[::-1])
    t = 0.5 * (c[:-1] + c[1:])
    return c, t


def mse(centroids, thresholds, d):
    """Mean squared error E[(x - Q(x))^2] of a codebook under f (closed-form moments + mass)."""
    c = np.asarray(centroids, dtype=np.float64)
    edges = np.concatenate([[-1.0], np.asarray(thresholds, dtype=np.float64), [1.0]])
    lo, hi = edges[:-1], edges[1:]
    m0 = cell_mass(lo, hi, d)
    m1 = cell_first_moment(lo, hi, d)
    # E[x^2] over the whole sphere coordinate is 1/d; subtract what the centroids explain.
    return 1.0 / d - np.sum(2.0 * c * m1 - c * c * m0)


def fp32_tables(d, bits):
    """The codebook as the decoder stores it: fp32 (round-to-nearest-even) centroids and thresholds.

    The thresholds are the fp32 roundings of the float64 midpoints, and a code
    decision compares an fp32 coordinate against them.
    """
    c, t = lloyd_max(d, bits)
    return c.astype(np.float32), t.astype(np.float32)
