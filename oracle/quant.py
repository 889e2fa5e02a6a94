"""Per-vector TurboQuant quantisers (store side) and the key-score estimator
(decode side), in fp64, vectorised over rows only.

Every function takes a batch of head vectors X of shape [N, d] (the values of
the bf16/fp32 inputs, held exactly in fp64) and applies the published steps to
each row independently.

Precision of decisions.  The pages fix no arithmetic precision, so where a
floating-point pre-image decides an integer (a centroid index, a half-up
rounding, an fp16 rounding) the decision is taken on the fp32 rounding of the
exact fp64 pre-image -- the precision the GPU kernels compute in.  The
fp64 pre-images are returned too, so that callers can count the cases that lie
within 1e-6 of a decision boundary (those may legitimately differ between two
correct implementations).
"""

import numpy as np


def to_f32(x):
    return np.asarray(x, np.float64).astype(np.float32).astype(np.float64)


def to_f16(x):
    """fp16 value of the fp32 rounding of x (float16 array)."""
    return np.asarray(x, np.float64).astype(np.float32).astype(np.float16)


def nearest_centroid(y, boundaries):
    """Index of the nearest centroid of a sorted Lloyd-Max codebook
    ([Hub] "Technical principle" step 2): the number of decision boundaries
    (midpoints between neighbouring centroids) strictly below y.  A y exactly on
    a boundary takes the lower index."""
    b32 = np.asarray(boundaries, np.float64).astype(np.float32)
    return np.searchsorted(b32, np.asarray(y).astype(np.float32), side="left")


def mse_quantise(X, R, boundaries):
    """TurboQuant-MSE of each row ([Explainer] steps 1-2, [Roadmap] §1,
    [Paged] "core idea"):

      n   = ||x||_2, stored as n16 = fp16(n)   (the norm/direction split)
      u   = x / n  (0 when n = 0)
      y   = R u                                (randomised Hadamard rotation)
      idx = nearest centroid of each coordinate of y

    Returns (n16 [N] float16, idx [N, d] int, pre-images {'n': n, 'y': y})."""
    n = np.sqrt(np.sum(X * X, axis=1))
    n16 = to_f16(n)
    u = np.divide(X, n[:, None], out=np.zeros_like(X), where=n[:, None] > 0)
    y = u @ R.T
    idx = nearest_centroid(y, boundaries)
    return n16, idx, {"n": n, "y": y}


def mse_reconstruct(n16, idx, R, centroids):
    """x_hat = n16 * R^T c[idx] (one row per vector)."""
    return n16.astype(np.float64)[:, None] * (np.asarray(centroids)[idx] @ R)


def qjl_residual(X, n16, idx, R, centroids, S):
    """Residual QJL for keys ([Explainer] step 3, [Hub] step 3, [Roadmap] §1):

      r     = x - n16 R^T c[idx]          (what the MSE stage missed)
      rho16 = fp16(||r||)
      bit_j = 1  iff  (S r)_j >= 0        (1-bit sign sketch; a zero maps to +1)

    Returns (rho16 [N] float16, bits [N, d] bool, pre-images {'rho', 'z'})."""
    r = X - mse_reconstruct(n16, idx, R, centroids)
    rho = np.sqrt(np.sum(r * r, axis=1))
    z = r @ np.asarray(S).T
    return to_f16(rho), z >= 0, {"rho": rho, "z": z}


def group32_quantise(V, bits):
    """Uniform group-32 value quantisation ([Hub] step 4): per group of 32
    consecutive coordinates (original, unrotated space) store an fp16 zero point
    and scale and a b-bit code per coordinate.  The page calls the scheme
    "symmetric" yet stores a zero point; the reading taken is asymmetric
    min/max, consistent with the idx*step + c0 dequant of [Roadmap] §4.3:

      z16 = fp16(min g),  s16 = fp16((max g - min g) / (2^b - 1))
      q   = clamp(floor((v - z16) / s16 + 1/2), 0, 2^b - 1)   (round half up)
      q   = 0 for the whole group when s16 = 0.

    Returns (s16 [N, d/32] float16, z16 [N, d/32] float16, q [N, d] int,
    pre-images {'scale', 'zero', 't'})."""
    N, d = V.shape
    g = V.reshape(N, d // 32, 32)
    lo, hi = g.min(axis=2), g.max(axis=2)
    top = 2**bits - 1
    scale = (hi - lo) / top
    z16, s16 = to_f16(lo), to_f16(scale)
    z, s = z16.astype(np.float64), s16.astype(np.float64)
    t = np.divide(g - z[..., None], s[..., None], out=np.zeros_like(g), where=s[..., None] > 0)
    q = np.clip(np.floor(to_f32(t) + 0.5), 0, top)
    q[np.broadcast_to((s == 0)[..., None], q.shape)] = 0
    return s16, z16, q.reshape(N, d).astype(np.int64), {"scale": scale, "zero": lo, "t": t}


def group32_reconstruct(s16, z16, q):
    N, d = q.shape
    s = np.repeat(s16.astype(np.float64), 32, axis=1)
    z = np.repeat(z16.astype(np.float64), 32, axis=1)
    return q * s + z


QJL_CONST = np.sqrt(np.pi / 2.0)


def key_scores(q, n16, idx, rho16, bits, R, centroids, S):
    """Estimated <q, k_t> for every stored key t ([Hub] "Technical principle",
    unbiased estimator; [Roadmap] §1):

      <R q, c[idx_t]> * n16_t  +  rho16_t * sqrt(pi/2)/d * <S q, 2 bit_t - 1>

    The first term is <q, n16 R^T c[idx_t]> written in the rotated basis; the
    second is the QJL estimate of <q, r_t>, unbiased over the draw of S because
    E[(s.q) sign(s.r)] = sqrt(2/pi) <q, r>/||r|| for a Gaussian row s.  With
    ``rho16``/``bits`` None (keys stored without QJL) only the first term."""
    d = len(q)
    rq = R @ q
    score = n16.astype(np.float64) * (np.asarray(centroids)[idx] @ rq)
    if bits is not None:
        sq = np.asarray(S) @ q
        score = score + rho16.astype(np.float64) * QJL_CONST / d * ((2.0 * bits - 1.0) @ sq)
    return score
