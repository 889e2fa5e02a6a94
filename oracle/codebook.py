"""Lloyd-Max scalar codebooks for one coordinate of a randomly rotated unit vector.

[Hub] "Technical principle" step 2: after the rotation each coordinate follows
a Beta distribution, and TurboQuant quantises it with a precomputed Lloyd-Max
codebook for head_dim 128 and 256 at 2, 3 and 4 bits.  Written out: one
coordinate t of a uniform unit vector in R^d has density on [-1, 1]

    f_d(t) = C_d (1 - t^2)^((d-3)/2),   C_d = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2)),

i.e. (t + 1)/2 ~ Beta((d-1)/2, (d-1)/2).  A Lloyd-Max quantiser with L = 2^b
levels alternates two conditions until neither moves (Lloyd 1957/1982,
Max 1960):
  * each decision boundary is the midpoint of its two neighbouring centroids;
  * each centroid is the conditional mean of t over its cell.

[Roadmap] §4.3 describes a second, "uniform" dequantisation mode (SGLang's
tq4u): the centroids lie on a linear grid, so a code dequantises as
idx * step + c0 with no table.  The pages do not say how the grid is chosen;
the reading taken here is the distortion-optimal symmetric uniform quantiser
for the same density (Max 1960, Table II gives it for a Gaussian source).
"""

import numpy as np
from scipy import special


class SphereCoordinate:
    """Cell masses, first moments and quantiles of f_d."""

    def __init__(self, d):
        self.d = d
        self.alpha = (d - 1) / 2.0
        self.const = np.exp(special.gammaln(d / 2.0) - special.gammaln((d - 1) / 2.0)) / np.sqrt(np.pi)
        self.lo, self.hi = -1.0, 1.0

    def density(self, t):
        return self.const * (1.0 - t * t) ** ((self.d - 3) / 2.0)

    def _lower_cdf(self, t):
        # P(T <= t) via the regularised incomplete beta function.
        return special.betainc(self.alpha, self.alpha, (np.asarray(t) + 1.0) / 2.0)

    def mass(self, a, b):
        """P(a < T <= b), evaluated in the lower tail to avoid cancellation."""
        a, b = np.asarray(a, float), np.asarray(b, float)
        upper = a >= 0
        lo_a = np.where(upper, -b, a)
        lo_b = np.where(upper, -a, b)
        return self._lower_cdf(lo_b) - self._lower_cdf(lo_a)

    def moment(self, a, b):
        """Integral of t f_d(t) over (a, b], closed form:
        C_d/(d-1) [(1-a^2)^((d-1)/2) - (1-b^2)^((d-1)/2)]."""
        p = (self.d - 1) / 2.0
        a, b = np.asarray(a, float), np.asarray(b, float)
        return self.const / (self.d - 1) * ((1.0 - a * a) ** p - (1.0 - b * b) ** p)

    def quantile(self, u):
        return 2.0 * special.betaincinv(self.alpha, self.alpha, u) - 1.0


class StandardNormal:
    """The same three functions for N(0, 1); used only to check the Lloyd
    iteration against the published Gaussian Lloyd-Max tables (Max 1960)."""

    lo, hi = -np.inf, np.inf

    def density(self, t):
        return np.exp(-0.5 * t * t) / np.sqrt(2.0 * np.pi)

    def mass(self, a, b):
        a, b = np.asarray(a, float), np.asarray(b, float)
        upper = a >= 0
        return np.where(upper, special.ndtr(-a) - special.ndtr(-b), special.ndtr(b) - special.ndtr(a))

    def moment(self, a, b):
        return self.density(np.asarray(a, float)) - self.density(np.asarray(b, float))

    def quantile(self, u):
        return special.ndtri(u)


def lloyd_max(dist, levels, tol=1e-14, max_iter=10000):
    """Lloyd-Max fixed point for a symmetric density.

    Returns (centroids ascending, boundaries = midpoints, iterations).  Starts
    from the density's quantiles at (i + 1/2)/L; keeps c_{L-1-i} = -c_i by
    averaging each new codebook with its mirror (the density is even); stops
    when no centroid moves by more than ``tol``.
    """
    c = dist.quantile((np.arange(levels) + 0.5) / levels)
    for it in range(1, max_iter + 1):
        b = 0.5 * (c[:-1] + c[1:])
        edges = np.concatenate([[dist.lo], b, [dist.hi]])
        new = dist.moment(edges[:-1], edges[1:]) / dist.mass(edges[:-1], edges[1:])
        new = 0.5 * (new - new[::-1])
        moved = np.max(np.abs(new - c))
        c = new
        if moved < tol:
            break
    return c, 0.5 * (c[:-1] + c[1:]), it


def sphere_codebook(d, bits):
    """Centroids (2^bits, ascending) and boundaries (2^bits - 1) for f_d."""
    c, b, _ = lloyd_max(SphereCoordinate(d), 2 ** bits)
    return c, b


def per_vector_mse(d, centroids):
    """Expected ||x - R^T c[idx]||^2 for a unit vector x: at a Lloyd fixed point
    each coordinate contributes E[t^2] - sum_i P_i c_i^2 = 1/d - sum_i P_i c_i^2,
    so D = 1 - d sum_i P_i c_i^2."""
    dist = SphereCoordinate(d)
    b = 0.5 * (centroids[:-1] + centroids[1:])
    edges = np.concatenate([[-1.0], b, [1.0]])
    p = dist.mass(edges[:-1], edges[1:])
    return 1.0 - d * np.sum(p * centroids**2)


def uniform_quantiser(dist, levels, tol=1e-14, max_iter=10000):
    """Distortion-optimal symmetric uniform quantiser for a symmetric density.

    Centroids c_i = step * k_i with k_i = i - (L-1)/2 (so c0 = -step*(L-1)/2),
    decision boundaries at the midpoints.  Two conditions alternate, as in the
    Lloyd iteration but with one free parameter:
      * for a fixed step the nearest-neighbour cells (midpoints) are best;
      * for fixed cells the distortion sum_i int_cell (t - step k_i)^2 f is a
        quadratic in step, least at step = sum_i k_i M_i / sum_i k_i^2 P_i
        (P_i the cell's mass, M_i its first moment).
    Starts from the step whose outer centroid is the (L - 1/2)/L quantile and
    stops when the step moves by less than ``tol`` relative.  The iteration
    converges linearly; at very large d the incomplete-beta masses carry
    ~1e-13 relative noise, so it can end at ``max_iter`` with the step settled
    to that level (the d = 8192 Gaussian-limit pins do).  Returns
    (centroids ascending, boundaries, step, iterations).
    """
    k = np.arange(levels) - (levels - 1) / 2.0
    step = 2.0 * dist.quantile((levels - 0.5) / levels) / (levels - 1)
    for it in range(1, max_iter + 1):
        c = step * k
        edges = np.concatenate([[dist.lo], 0.5 * (c[:-1] + c[1:]), [dist.hi]])
        p = dist.mass(edges[:-1], edges[1:])
        m = dist.moment(edges[:-1], edges[1:])
        new = np.sum(k * m) / np.sum(k * k * p)
        moved = abs(new - step)
        step = new
        if moved < tol * step:
            break
    c = step * k
    return c, 0.5 * (c[:-1] + c[1:]), step, it


def sphere_uniform_codebook(d, bits):
    """Uniform-grid centroids (2^bits, ascending) and boundaries for f_d."""
    c, b, _, _ = uniform_quantiser(SphereCoordinate(d), 2**bits)
    return c, b


def sphere_codebook_of_kind(d, bits, kind):
    """kind "lloyd" (Lloyd-Max, [Hub] step 2) or "uniform" ([Roadmap] §4.3)."""
    if kind == "lloyd":
        return sphere_codebook(d, bits)
    if kind == "uniform":
        return sphere_uniform_codebook(d, bits)
    raise ValueError(f"unknown codebook kind {kind!r}")


def nearest_neighbour_mse(dist, second_moment, centroids):
    """E[(t - Q(t))^2] of the nearest-neighbour quantiser with these sorted
    centroids, for any codebook (not only a Lloyd fixed point):
    E[t^2] - sum_i (2 c_i M_i - c_i^2 P_i) over the midpoint cells."""
    edges = np.concatenate([[dist.lo], 0.5 * (centroids[:-1] + centroids[1:]), [dist.hi]])
    p = dist.mass(edges[:-1], edges[1:])
    m = dist.moment(edges[:-1], edges[1:])
    return second_moment - np.sum(2.0 * centroids * m - centroids**2 * p)
