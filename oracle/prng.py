"""Seeded random parameters of one TurboQuant cache: the rotation's sign diagonal
D and the QJL projection S.

The pages say the rotation is a randomised Walsh-Hadamard transform and the QJL
projection a d x d random (Gaussian) matrix S ([Roadmap] §1, [Hub] "Technical
principle" steps 1 and 3) but fix no generator.  Reading taken here (parity
unpinned): SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) as a counter-based stream, one stream per
seed; the i-th output (i = 0, 1, ...) is

    mix(seed + (i + 1) * 0x9E3779B97F4A7C15  mod 2^64)

with mix(z) = z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
z *= 0x94D049BB133111EB; z ^= z >> 31  (all mod 2^64).
"""

import numpy as np

GOLDEN_GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB


def splitmix64(seed, n):
    """First ``n`` outputs of the SplitMix64 stream for ``seed`` (uint64 array)."""
    counter = np.arange(1, n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + counter * np.uint64(GOLDEN_GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX2)
    return z ^ (z >> np.uint64(31))


def rotation_signs(d, seed):
    """The +-1 diagonal D of the randomised Hadamard rotation ([Roadmap] §1).

    D_i = -1 when the top bit of the i-th SplitMix64 output is set, else +1.
    """
    x = splitmix64(seed, d)
    return np.where((x >> np.uint64(63)) == 1, -1.0, 1.0)


def uniform01(x):
    """Map 64-bit outputs to doubles strictly inside (0, 1): ((x >> 11) + 1/2) * 2^-53."""
    return ((x >> np.uint64(11)).astype(np.float64) + 0.5) * 2.0**-53


def round_to_bf16(x):
    """Round fp64 values directly to the nearest bfloat16 value (8 significant
    bits, ties to even), returned as fp64.  Valid in bf16's normal range."""
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(np.rint(m * 256.0), e - 8)


def qjl_matrix(d, seed):
    """The d x d QJL projection S ([Hub] "Technical principle" step 3), row-major
    S[j, i], entries N(0, 1) by Box-Muller on consecutive output pairs:
    for pair p, u1 = U(x_2p), u2 = U(x_2p+1),
        S.flat[2p]   = sqrt(-2 ln u1) cos(2 pi u2)
        S.flat[2p+1] = sqrt(-2 ln u1) sin(2 pi u2),
    then rounded to bfloat16 (so that the matrix is exact in the tensor-core
    operand type; a reading, the pages fix no precision)."""
    u = uniform01(splitmix64(seed, d * d))
    u1, u2 = u[0::2], u[1::2]
    radius = np.sqrt(-2.0 * np.log(u1))
    g = np.empty(d * d)
    g[0::2] = radius * np.cos(2.0 * np.pi * u2)
    g[1::2] = radius * np.sin(2.0 * np.pi * u2)
    return round_to_bf16(g).reshape(d, d)
