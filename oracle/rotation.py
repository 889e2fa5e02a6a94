"""The randomised Walsh-Hadamard rotation, built as a dense matrix.

[Roadmap] §1 and [Paged] "TurboQuant's core idea": each vector is first rotated
by a random orthogonal map realised with a Walsh-Hadamard transform; the
rotation keeps norms and inner products and spreads outlier energy over all
coordinates.  Reading taken (the pages name the transform, not its normalisation
or sign placement): R = H D / sqrt(d) with H the Sylvester-ordered Hadamard
matrix, H_ij = (-1)^popcount(i & j), and D = diag(+-1) from ``prng``.  The
inverse is R^T = D H / sqrt(d) (H is symmetric), applied to undo the rotation on
the value side ([Roadmap] §4.2).
"""

import numpy as np


def hadamard(d):
    """Sylvester Hadamard matrix of order d (a power of two), by its entry formula."""
    i = np.arange(d)
    parity = np.vectorize(lambda m: bin(m).count("1") & 1)(i[:, None] & i[None, :])
    return np.where(parity == 1, -1.0, 1.0)


def rotation_matrix(signs):
    """R = H diag(signs) / sqrt(d)."""
    d = len(signs)
    return hadamard(d) * np.asarray(signs, float)[None, :] / np.sqrt(d)
