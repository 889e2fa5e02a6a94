"""Pins of the fp64 oracle against values and facts fixed outside itself: the
pages' printed numbers, published tables, closed forms, invariants and brute
force.  CPU only."""

import os

import numpy as np
import pytest
from scipy import special, stats

from oracle import codebook, paged, prng, quant, rotation

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [line.split() for line in f if line.strip() and not line.startswith("#")]


# --------------------------------------------------------------------- PRNG
def test_splitmix64_known_answers():
    for row in _rows("splitmix64_known_answers.txt"):
        seed, expect = int(row[0]), [int(x) for x in row[1:]]
        got = [int(x) for x in prng.splitmix64(seed, len(expect))]
        assert got == expect


def test_qjl_matrix_is_gaussian_and_bf16_exact():
    S = prng.qjl_matrix(128, 1)
    flat = S.ravel()
    # bf16-exact: every entry has at most 8 significant bits.
    m, _ = np.frexp(flat)
    assert np.all(m * 256 == np.rint(m * 256))
    assert abs(flat.mean()) < 4 / np.sqrt(flat.size)
    assert abs(flat.var() - 1.0) < 4 * np.sqrt(2.0 / flat.size)
    assert stats.kstest(flat, "norm").pvalue > 1e-3
    # cos and sin halves of Box-Muller are uncorrelated
    assert abs(np.corrcoef(flat[0::2], flat[1::2])[0, 1]) < 4 / np.sqrt(flat.size / 2)


def test_round_to_bf16_matches_nearest_even():
    x = np.array([1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-8 + 2**-40, -3.0 - 2**-7])
    # halfway -> even mantissa; above halfway -> up
    assert list(prng.round_to_bf16(x)) == [1.0, 1.0 + 4 * 2**-8, 1.0 + 2**-7, -3.0]


def test_rotation_signs_are_pm1_and_balanced():
    s = prng.rotation_signs(4096, 2)
    assert set(np.unique(s)) == {-1.0, 1.0}
    assert abs(s.sum()) < 4 * np.sqrt(4096)


# ----------------------------------------------------------------- rotation
def _sylvester(d):
    h = np.ones((1, 1))
    while len(h) < d:
        h = np.block([[h, h], [h, -h]])
    return h


@pytest.mark.parametrize("d", [2, 4, 8, 16, 128])
def test_hadamard_entry_formula_equals_sylvester_recursion(d):
    assert np.array_equal(rotation.hadamard(d), _sylvester(d))


def test_rotation_orthogonal_and_preserves_geometry():
    R = rotation.rotation_matrix(prng.rotation_signs(128, 2))
    assert np.max(np.abs(R.T @ R - np.eye(128))) < 1e-14
    rng = np.random.default_rng(3)
    a, b = rng.standard_normal((2, 128))
    assert abs(np.linalg.norm(R @ a) - np.linalg.norm(a)) < 1e-12
    assert abs((R @ a) @ (R @ b) - a @ b) < 1e-11


def test_rotation_spreads_an_outlier():
    # [Paged] "core idea": the rotation spreads a large coordinate over all.
    R = rotation.rotation_matrix(prng.rotation_signs(128, 2))
    e = np.zeros(128)
    e[5] = 20.0
    assert np.allclose(np.abs(R @ e), 20.0 / np.sqrt(128))


# ----------------------------------------------------------------- codebook
def test_gaussian_lloyd_max_matches_max_1960():
    for row in _rows("max1960_gaussian_lloyd_max.txt"):
        L, mse = int(row[0]), float(row[1])
        pos = np.array([float(x) for x in row[2:]])
        c, b, _ = codebook.lloyd_max(codebook.StandardNormal(), L)
        assert np.allclose(c[L // 2:], pos, atol=6e-4)
        edges = np.concatenate([[-np.inf], b, [np.inf]])
        got = 1.0 - np.sum(codebook.StandardNormal().mass(edges[:-1], edges[1:]) * c**2)
        assert abs(got - mse) / mse < 1e-3


@pytest.mark.parametrize("d", [16, 128, 256])
def test_one_bit_centroid_closed_form(d):
    c, b = codebook.sphere_codebook(d, 1)
    expect = np.exp(special.gammaln(d / 2) - special.gammaln((d + 1) / 2)) / np.sqrt(np.pi)
    assert b[0] == 0.0
    assert abs(c[1] - expect) < 1e-14 and abs(c[0] + expect) < 1e-14


def _gauss_legendre_cell(f, a, b, n=400):
    x, w = np.polynomial.legendre.leggauss(n)
    t = 0.5 * (b - a) * x + 0.5 * (b + a)
    return 0.5 * (b - a) * np.sum(w * f(t))


@pytest.mark.parametrize("d,bits", [(128, 2), (128, 3), (128, 4), (256, 2), (256, 3), (256, 4)])
def test_codebook_centroid_condition_and_mse_by_quadrature(d, bits):
    c, b = codebook.sphere_codebook(d, bits)
    dist = codebook.SphereCoordinate(d)
    # the density integrates to one (pins the normalising constant)
    assert abs(_gauss_legendre_cell(dist.density, -1.0, 1.0, 2000) - 1.0) < 1e-12
    edges = np.concatenate([[-1.0], b, [1.0]])
    mse_quad = 0.0
    for i in range(len(c)):
        lo, hi = edges[i], edges[i + 1]
        mass = _gauss_legendre_cell(dist.density, lo, hi)
        mom = _gauss_legendre_cell(lambda t: t * dist.density(t), lo, hi)
        assert abs(mom / mass - c[i]) < 1e-12
        mse_quad += _gauss_legendre_cell(lambda t: (t - c[i]) ** 2 * dist.density(t), lo, hi)
    assert abs(d * mse_quad - codebook.per_vector_mse(d, c)) < 1e-10


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_codebook_mse_within_published_bound(bits):
    # [Roadmap] §6.3: distortion within a constant factor (~2.7) of the
    # information-theoretic lower bound, which is 4^-b per unit vector.
    D = codebook.per_vector_mse(128, codebook.sphere_codebook(128, bits)[0])
    assert 4.0**-bits <= D <= 2.7 * 4.0**-bits


def test_sphere_codebook_tends_to_gaussian_table():
    # sqrt(d) t -> N(0,1) as d grows, so sqrt(d) c -> the Gaussian quantiser.
    rows = {int(r[0]): np.array([float(x) for x in r[2:]]) for r in _rows("max1960_gaussian_lloyd_max.txt")}
    for bits in (2, 3):
        c, _ = codebook.sphere_codebook(8192, bits)
        assert np.allclose(np.sqrt(8192) * c[2 ** (bits - 1):], rows[2**bits], atol=2e-3)


@pytest.mark.parametrize("bits", [2, 3])
def test_codebook_mse_monte_carlo(bits):
    d = 128
    c, b = codebook.sphere_codebook(d, bits)
    R = rotation.rotation_matrix(prng.rotation_signs(d, 2))
    rng = np.random.default_rng(11)
    X = rng.standard_normal((20000, d))
    n16, idx, _ = quant.mse_quantise(X, R, b)
    Xn = X / np.linalg.norm(X, axis=1, keepdims=True)
    err = np.sum((Xn - c[idx] @ R) ** 2, axis=1)
    D = codebook.per_vector_mse(d, c)
    assert abs(err.mean() - D) < 3 * err.std() / np.sqrt(len(err))


def test_mse_cosine_consistent_with_hub_quality_table():
    # cos(x, x_hat) = sqrt(1 - D) for a Lloyd-Max quantiser; the hub prints
    # 0.940 for 2-bit values.
    table = {r[0]: float(r[1]) for r in _rows("hub_quality_table.txt")}
    D2 = codebook.per_vector_mse(128, codebook.sphere_codebook(128, 2)[0])
    assert abs(np.sqrt(1 - D2) - table["value2"]) < 0.005


def test_gaussian_uniform_quantiser_matches_max_1960():
    for row in _rows("max1960_gaussian_uniform.txt"):
        L, step, mse = int(row[0]), float(row[1]), float(row[2])
        c, b, got_step, _ = codebook.uniform_quantiser(codebook.StandardNormal(), L)
        assert abs(got_step - step) < 6e-4
        assert np.allclose(np.diff(c), got_step, rtol=1e-12) and abs(c[0] + c[-1]) < 1e-12
        got = codebook.nearest_neighbour_mse(codebook.StandardNormal(), 1.0, c)
        assert abs(got - mse) / mse < 1e-3


@pytest.mark.parametrize("d", [16, 128, 256])
def test_one_bit_uniform_is_the_lloyd_quantiser(d):
    # two levels are always equally spaced: the uniform quantiser is then the
    # Lloyd-Max one, +-E|t| in closed form
    c, b = codebook.sphere_uniform_codebook(d, 1)
    expect = np.exp(special.gammaln(d / 2) - special.gammaln((d + 1) / 2)) / np.sqrt(np.pi)
    assert abs(c[1] - expect) < 1e-13 and abs(c[0] + expect) < 1e-13 and b[0] == 0.0


def _distortion_by_quadrature(dist, c):
    """int (t - Q(t))^2 f over [-1, 1], cell by cell with Gauss-Legendre
    (independent of the closed-form masses and moments)."""
    x, w = _LEGGAUSS_400
    edges = np.concatenate([[-1.0], 0.5 * (c[:-1] + c[1:]), [1.0]])
    lo, hi = edges[:-1, None], edges[1:, None]
    t = 0.5 * (hi - lo) * x + 0.5 * (hi + lo)
    return float(np.sum(0.5 * (hi - lo)[:, 0] * np.sum(w * (t - c[:, None]) ** 2 * dist.density(t), axis=1)))


_LEGGAUSS_400 = np.polynomial.legendre.leggauss(400)


@pytest.mark.parametrize("d,bits", [(128, 2), (128, 3), (128, 4), (256, 4)])
def test_uniform_step_is_the_brute_force_minimum(d, bits):
    dist = codebook.SphereCoordinate(d)
    c, b, step, _ = codebook.uniform_quantiser(dist, 2**bits)
    k = np.arange(2**bits) - (2**bits - 1) / 2.0
    best = _distortion_by_quadrature(dist, c)
    # the generic distortion formula agrees with direct integration
    assert abs(codebook.nearest_neighbour_mse(dist, 1.0 / d, c) - best) < 1e-12
    # a grid search over steps finds nothing lower, and its minimum sits next to step
    grid = step * np.linspace(0.5, 1.5, 201)
    vals = np.array([_distortion_by_quadrature(dist, s * k) for s in grid])
    assert vals.min() >= best - 1e-15
    assert abs(grid[np.argmin(vals)] - step) <= step * 0.005 + 1e-15
    # and it is a strict local minimum
    for f in (1 - 1e-3, 1 + 1e-3):
        assert _distortion_by_quadrature(dist, f * step * k) > best


def test_uniform_sphere_quantiser_tends_to_gaussian_table():
    rows = {int(r[0]): float(r[1]) for r in _rows("max1960_gaussian_uniform.txt")}
    for bits in (2, 3, 4):
        _, _, step, _ = codebook.uniform_quantiser(codebook.SphereCoordinate(8192), 2**bits)
        assert abs(np.sqrt(8192) * step - rows[2**bits]) < 2e-3


@pytest.mark.parametrize("bits", [3, 4])
def test_uniform_codebook_mse_monte_carlo(bits):
    # random unit vectors through the rotation and the uniform codebook: the
    # mean squared error matches d * E[(t - Q(t))^2] within 3 standard errors
    d = 128
    c, b = codebook.sphere_uniform_codebook(d, bits)
    R = rotation.rotation_matrix(prng.rotation_signs(d, 2))
    X = np.random.default_rng(12).standard_normal((20000, d))
    n16, idx, _ = quant.mse_quantise(X, R, b)
    Xn = X / np.linalg.norm(X, axis=1, keepdims=True)
    err = np.sum((Xn - c[idx] @ R) ** 2, axis=1)
    D = d * codebook.nearest_neighbour_mse(codebook.SphereCoordinate(d), 1.0 / d, c)
    assert abs(err.mean() - D) < 3 * err.std() / np.sqrt(len(err))


def test_uniform_costs_little_distortion_at_four_bits():
    # [Roadmap] §4.3: at 4 bits the uniform grid costs almost nothing in
    # accuracy against the Lloyd codebook; in distortion it is above Lloyd-Max
    # (which is optimal among all 16-level quantisers) but close to it
    d = 128
    dist = codebook.SphereCoordinate(d)
    lloyd = codebook.per_vector_mse(d, codebook.sphere_codebook(d, 4)[0])
    unif = d * codebook.nearest_neighbour_mse(dist, 1.0 / d, codebook.sphere_uniform_codebook(d, 4)[0])
    assert lloyd < unif < 1.3 * lloyd
    assert np.sqrt(1 - unif) > 0.99


def test_nearest_centroid_is_brute_force_argmin():
    rng = np.random.default_rng(5)
    for d, bits, kind in [(4, 2, "lloyd"), (8, 3, "lloyd"), (16, 4, "lloyd"), (128, 3, "lloyd"), (8, 3, "uniform"),
                          (128, 4, "uniform")]:
        c, b = codebook.sphere_codebook_of_kind(d, bits, kind)
        y = rng.uniform(-1.2 * c[-1], 1.2 * c[-1], size=(200, d))
        idx = quant.nearest_centroid(y, b)
        brute = np.argmin(np.abs(y[..., None] - c), axis=-1)
        assert np.array_equal(idx, brute)
    # a point exactly on a boundary takes the lower index
    c, b = codebook.sphere_codebook(128, 2)
    on = np.float32(b[1]).astype(np.float64)
    assert quant.nearest_centroid(np.array([on]), b)[0] == 1


# ------------------------------------------------------------------ packing
def test_pack_golden_examples():
    for row in _rows("pack_examples.txt"):
        bits = int(row[0])
        nbytes = {2: 1, 4: 1, 3: 3, 1: 2}[bits]
        codes = np.array([int(x) for x in row[1:-nbytes]])
        expect = [int(x, 16) for x in row[-nbytes:]]
        if bits == 1:
            got = paged.pack_bits(codes[None].astype(bool))[0]
        else:
            got = paged.pack_codes(codes[None], bits)[0]
        assert list(got) == expect


def test_bit_plane_golden_examples():
    # the bit-sliced layout of key codes and MSE value codes, worked by hand
    with open(os.path.join(GOLDEN, "bit_plane_examples.txt")) as f:
        rows = [line.split("|") for line in f if line.strip() and not line.startswith("#")]
    for bits_s, codes_s, planes_s in rows:
        bits = int(bits_s)
        codes = np.array([int(x) for x in codes_s.split()])[None]
        expect = [bytes.fromhex(p.replace(" ", "")) for p in planes_s.split("/")]
        got = paged.pack_bit_planes(codes, bits)
        assert [bytes(p[0]) for p in got] == expect
        # same bytes per row as the page's stated density (b bits per code)
        assert sum(len(e) for e in expect) == codes.shape[1] * bits // 8
        assert np.array_equal(paged.unpack_bit_planes(got, codes.shape[1]), codes)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_pack_unpack_round_trip(bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 2**bits, size=(64, 128))
    rows = paged.pack_codes(codes, bits)
    assert rows.shape == (64, 128 * bits // 8)
    assert np.array_equal(paged.unpack_codes(rows, 128, bits), codes)
    flags = rng.integers(0, 2, size=(64, 256)).astype(bool)
    assert np.array_equal(paged.unpack_bits(paged.pack_bits(flags), 256), flags)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_bit_planes_round_trip_and_hand_example(bits):
    rng = np.random.default_rng(10 + bits)
    codes = rng.integers(0, 2**bits, size=(16, 128))
    planes = paged.pack_bit_planes(codes, bits)
    assert len(planes) == bits and all(p.shape == (16, 16) for p in planes)
    assert np.array_equal(paged.unpack_bit_planes(planes, 128), codes)
    # codes 5, 3, 6, 0, ...: bit-0 plane byte 0 = 1,1,0 -> 0x03; bit 1: 0,1,1 -> 0x06; bit 2: 1,0,1 -> 0x05
    ex = np.zeros((1, 8), np.int64)
    ex[0, :3] = [5, 3, 6]
    pl = paged.pack_bit_planes(ex, 3)
    assert [pl[0][0, 0], pl[1][0, 0], pl[2][0, 0]] == [0x03, 0x06, 0x05]


@pytest.mark.parametrize("d", [128, 256])
def test_group32_slot_permutation(d):
    tau = paged.group32_slot_coordinates(d)
    assert np.array_equal(np.sort(tau), np.arange(d))          # a bijection
    if d == 128:
        # hand-computed from slot k = 16 g + 2 m + e -> 32 (m//2) + 4 g + 2 (m%2) + e
        assert list(tau[:8]) == [0, 1, 2, 3, 32, 33, 34, 35] and list(tau[16:20]) == [4, 5, 6, 7]
    w = d // 8
    for k in range(0, d, 2):  # the two slots of a pair are adjacent coordinates of one group
        assert tau[k + 1] == tau[k] + 1 and tau[k] // 32 == tau[k + 1] // 32
    for m in range(d // 16):  # slot pair m of every g lies in group m // 2
        assert {tau[w * g + 2 * m] // 32 for g in range(8)} == {m // 2}


def test_group32_slot_round_trip_through_a_page():
    P = paged.CacheParams(128, 2, True, "g32", 4, 2, 1)
    rng = np.random.default_rng(4)
    V = rng.standard_normal((16, 1, 128))
    K = rng.standard_normal((16, 1, 128))
    cache = np.zeros((1, 1, P.layout.page_bytes), np.uint8)
    pre = paged.store(cache, P, K, V, np.arange(16))
    f = paged.read_tokens(cache, P, np.array([0]), 16, 0)
    assert np.array_equal(f["v_codes"], pre["v_q"])
    assert np.array_equal(f["k_idx"], pre["k_idx"])


def test_page_layout_sizes():
    # bytes per token-head: codes + signs + 2 fp16 norms, plus value codes and
    # metadata (these totals follow from the layout reading, e.g. 68 + 80 for
    # 3-bit keys with QJL and 4-bit group-32 values at d = 128)
    assert paged.PageLayout(128, 3, True, "g32", 4).page_bytes == 16 * (68 + 80)
    assert paged.PageLayout(256, 2, True, "mse", 2).page_bytes == 16 * (100 + 66)
    assert paged.PageLayout(128, 2, True, "mse", 2).page_bytes == 16 * (52 + 34)
    assert paged.PageLayout(128, 3, True, "mse", 2).page_bytes == 16 * (68 + 34)


# ---------------------------------------------------------------- group-32
def test_group32_is_nearest_level_brute_force():
    rng = np.random.default_rng(9)
    V = rng.standard_normal((300, 128)) * 3
    for bits in (2, 3, 4):
        s16, z16, q, pre = quant.group32_quantise(V, bits)
        s = np.repeat(s16.astype(float), 32, 1)
        z = np.repeat(z16.astype(float), 32, 1)
        levels = np.arange(2**bits)
        dist = np.abs(V[..., None] - (levels * s[..., None] + z[..., None]))
        brute = np.argmin(dist - 1e-12 * levels, axis=-1)  # ties -> upper (half up)
        near_half = np.abs(pre["t"].reshape(V.shape) - np.floor(pre["t"].reshape(V.shape)) - 0.5) < 1e-6
        assert np.array_equal(q[~near_half], brute[~near_half])


def test_group32_constant_group_and_range():
    V = np.zeros((2, 128))
    V[0, :32] = 1.5
    V[1] = np.linspace(-4, 4, 128)
    s16, z16, q, _ = quant.group32_quantise(V, 4)
    assert s16[0, 0] == 0 and z16[0, 0] == np.float16(1.5) and np.all(q[0, :32] == 0)
    # the group minimum maps to 0 and the maximum to 2^b - 1
    assert q[1, 0] == 0 and q[1, 31] == 15


def test_group32_cosine_consistent_with_hub_quality_table():
    table = {r[0]: float(r[1]) for r in _rows("hub_quality_table.txt")}
    rng = np.random.default_rng(12)
    V = rng.standard_normal((5000, 128))
    s16, z16, q, _ = quant.group32_quantise(V, 4)
    Vh = quant.group32_reconstruct(s16, z16, q)
    cos = np.sum(V * Vh, 1) / np.linalg.norm(V, axis=1) / np.linalg.norm(Vh, axis=1)
    assert abs(cos.mean() - table["value4"]) < 0.002


# -------------------------------------------------------------- QJL / keys
def test_qjl_sign_identity_closed_form():
    # E[(s.q) sign(s.r)] = sqrt(2/pi) <q,r>/||r|| for s ~ N(0, I)
    rng = np.random.default_rng(21)
    q, r = rng.standard_normal((2, 32))
    s = rng.standard_normal((400000, 32))
    x = (s @ q) * np.sign(s @ r)
    expect = np.sqrt(2 / np.pi) * (q @ r) / np.linalg.norm(r)
    assert abs(x.mean() - expect) < 3 * x.std() / np.sqrt(len(x))


def test_key_estimator_unbiased_over_qjl_seeds():
    # [Hub] "Technical principle": the compressed score is an unbiased
    # estimate of <q, k>; the expectation is over the draw of S.
    d = 32
    c, b = codebook.sphere_codebook(d, 2)
    R = rotation.rotation_matrix(prng.rotation_signs(d, 2))
    rng = np.random.default_rng(4)
    k = rng.standard_normal((1, d))
    q = rng.standard_normal(d)
    n16, idx, _ = quant.mse_quantise(k, R, b)
    est = []
    for seed in range(3000):
        S = prng.qjl_matrix(d, 1000 + seed)
        rho16, bits, _ = quant.qjl_residual(k, n16, idx, R, c, S)
        est.append(quant.key_scores(q, n16, idx, rho16, bits, R, c, S)[0])
    est = np.array(est)
    true = k[0] @ q
    assert abs(est.mean() - true) < 3 * est.std() / np.sqrt(len(est))
    # without the QJL term the MSE-only estimate is off by <q, r>
    mse_only = quant.key_scores(q, n16, idx, None, None, R, c, None)[0]
    r = k[0] - quant.mse_reconstruct(n16, idx, R, c)[0]
    assert abs(mse_only + q @ r - true) < 1e-9


def test_key_inner_product_cosine_at_3_bits():
    # [Hub] "Quality cost": key 3-bit cosine 1.000000.  Reading: cosine between
    # true and estimated <q, k> over random pairs of outlier-heavy vectors
    # (N(0,1) with 2% of channels x10, the decode workloads' recipe).
    d = 128
    P = paged.CacheParams(d, 3, True, "mse", 2, 2, 1)
    rng = np.random.default_rng(8)
    K = rng.standard_normal((4000, d))
    Q = rng.standard_normal((4000, d))
    K[:, :3] *= 10
    Q[:, :3] *= 10
    n16, idx, _ = quant.mse_quantise(K, P.R, P.k_boundaries)
    rho16, bits, _ = quant.qjl_residual(K, n16, idx, P.R, P.k_centroids, P.S)
    est = np.array([quant.key_scores(Q[i], n16[i:i + 1], idx[i:i + 1], rho16[i:i + 1], bits[i:i + 1],
                                     P.R, P.k_centroids, P.S)[0] for i in range(len(K))])
    true = np.sum(Q * K, axis=1)
    cos = est @ true / np.linalg.norm(est) / np.linalg.norm(true)
    assert cos > 0.998


# ------------------------------------------------------------------ decode
def _small_cache(v_mode, seed=0, T=40, H=2, d=128, k_bits=3, v_bits=4):
    P = paged.CacheParams(d, k_bits, True, v_mode, v_bits, 2, 1)
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((T, H, d))
    V = rng.standard_normal((T, H, d))
    K[..., :3] *= 10
    nblk = 8
    cache = np.zeros((nblk, H, P.layout.page_bytes), np.uint8)
    table = rng.permutation(nblk)[None, :]
    slots = table[0, np.arange(T) // 16] * 16 + np.arange(T) % 16
    paged.store(cache, P, K, V, slots)
    return P, cache, table, K, V


@pytest.mark.parametrize("v_mode", ["mse", "g32"])
def test_decode_equals_textbook_attention_on_reconstructed_keys(v_mode):
    # Special-case reduction: the rotated-basis score equals <q, k_hat> with
    # k_hat = n16 R^T c[idx] + rho16 sqrt(pi/2)/d S^T (2 bits - 1); decode is
    # then plain softmax attention over (k_hat, v_hat).
    P, cache, table, K, V = _small_cache(v_mode)
    T, H, d = K.shape
    rng = np.random.default_rng(1)
    Q = rng.standard_normal((1, 2 * H, d))
    out = paged.decode_attention(cache, P, Q, table, [T])
    for g in range(H):
        f = paged.read_tokens(cache, P, table[0], T, g)
        k_hat = quant.mse_reconstruct(f["k_n16"], f["k_idx"], P.R, P.k_centroids)
        k_hat += f["k_rho16"].astype(float)[:, None] * np.sqrt(np.pi / 2) / d * ((2.0 * f["k_bits"] - 1) @ P.S)
        if v_mode == "mse":
            v_hat = quant.mse_reconstruct(f["v_n16"], f["v_codes"], P.R, P.v_centroids)
        else:
            v_hat = quant.group32_reconstruct(f["v_s16"], f["v_z16"], f["v_codes"])
        for h in (2 * g, 2 * g + 1):
            p = special.softmax(k_hat @ Q[0, h] / np.sqrt(d))
            assert np.max(np.abs(p @ v_hat - out[0, h])) < 1e-10


def test_decode_one_token_returns_its_value():
    P, cache, table, K, V = _small_cache("mse")
    Q = np.random.default_rng(2).standard_normal((1, 4, 128)) * 30
    out = paged.decode_attention(cache, P, Q, table, [1])
    f = paged.read_tokens(cache, P, table[0], 1, 0)
    v0 = quant.mse_reconstruct(f["v_n16"], f["v_codes"], P.R, P.v_centroids)[0]
    assert np.max(np.abs(out[0, 0] - v0)) < 1e-12


def test_decode_empty_sequence_is_zero_and_tail_only_is_exact_attention():
    P, cache, table, K, V = _small_cache("g32")
    rng = np.random.default_rng(3)
    Q = rng.standard_normal((1, 4, 128))
    assert np.all(paged.decode_attention(cache, P, Q, table, [0]) == 0)
    tk = rng.standard_normal((1, 2, 8, 128))
    tv = rng.standard_normal((1, 2, 8, 128))
    out = paged.decode_attention(cache, P, Q, table, [0], tail_k=tk, tail_v=tv, tail_lens=[5])
    p = special.softmax(tk[0, 1, :5] @ Q[0, 3] / np.sqrt(128))
    assert np.max(np.abs(out[0, 3] - p @ tv[0, 1, :5])) < 1e-12


def test_store_skips_negative_slots_and_block_table_is_respected():
    P = paged.CacheParams(128, 2, True, "mse", 2, 2, 1)
    rng = np.random.default_rng(6)
    K = rng.standard_normal((20, 1, 128))
    V = rng.standard_normal((20, 1, 128))
    a = np.zeros((4, 1, P.layout.page_bytes), np.uint8)
    b = np.zeros_like(a)
    slots = np.arange(20)
    skip = slots.copy()
    skip[3] = -1
    paged.store(a, P, K, V, slots)
    paged.store(b, P, K, V, skip)
    row3 = paged.gather_rows(b, P, np.array([0]), np.array([3]), 0, "k_code0")
    assert np.all(row3 == 0)
    # the same tokens placed in other physical blocks decode identically
    c = np.zeros_like(a)
    perm = np.array([2, 0])
    paged.store(c, P, K, V, perm[np.arange(20) // 16] * 16 + np.arange(20) % 16)
    Q = rng.standard_normal((1, 1, 128))
    o1 = paged.decode_attention(a, P, Q, np.array([[0, 1]]), [20])
    o2 = paged.decode_attention(c, P, Q, perm[None], [20])
    assert np.array_equal(o1, o2)


def test_decode_extreme_logits_reach_the_one_hot_limit():
    # Logit spreads of thousands (queries x1e3) must not overflow: softmax
    # tends to the one-hot at the best-scoring key, and out to its value.
    P, cache, table, K, V = _small_cache("g32")
    T = K.shape[0]
    Q = np.random.default_rng(7).standard_normal((1, 4, 128)) * 1e3
    out = paged.decode_attention(cache, P, Q, table, [T])
    assert np.all(np.isfinite(out))
    f = paged.read_tokens(cache, P, table[0], T, 0)
    s = quant.key_scores(Q[0, 0], f["k_n16"], f["k_idx"], f["k_rho16"], f["k_bits"], P.R, P.k_centroids, P.S)
    v_hat = quant.group32_reconstruct(f["v_s16"], f["v_z16"], f["v_codes"])
    assert np.max(np.abs(out[0, 0] - v_hat[np.argmax(s)])) < 1e-9


def test_store_with_no_tokens_is_a_noop():
    P = paged.CacheParams(128, 3, True, "g32", 4, 2, 1)
    cache = np.zeros((2, 8, P.layout.page_bytes), np.uint8)
    empty = np.zeros((0, 8, 128))
    paged.store(cache, P, empty, empty, np.zeros(0, np.int64))
    paged.store(cache, P, np.ones((3, 8, 128)), np.ones((3, 8, 128)), np.full(3, -1))
    assert not cache.any()


# ------------------------------------------------------------------ extend
def _extend_problem(v_mode, prefix, chunks, seed=4):
    """Two sequences sharing nothing: sequence b has prefix[b] tokens in the
    cache and chunks[b] new exact tokens."""
    P = paged.CacheParams(128, 3, True, v_mode, 4, 2, 1)
    H, Hq, d = 2, 4, 128
    rng = np.random.default_rng(seed)
    nblk = sum((n + 15) // 16 for n in prefix) + 2
    cache = np.zeros((nblk, H, P.layout.page_bytes), np.uint8)
    perm = rng.permutation(nblk)
    width = max(1, max((n + 15) // 16 for n in prefix))
    table = np.zeros((len(prefix), width), np.int64)
    at = 0
    for b, n in enumerate(prefix):
        k = (n + 15) // 16
        table[b, :k] = perm[at:at + k]
        at += k
        K = rng.standard_normal((n, H, d))
        K[..., :3] *= 10
        V = rng.standard_normal((n, H, d))
        t = np.arange(n)
        paged.store(cache, P, K, V, table[b, t // 16] * 16 + t % 16)
    cu = np.concatenate([[0], np.cumsum(chunks)])
    T = int(cu[-1])
    Q = rng.standard_normal((T, Hq, d))
    ck = rng.standard_normal((T, H, d))
    cv = rng.standard_normal((T, H, d))
    return P, cache, table, cu, Q, ck, cv


def test_extend_without_prefix_is_textbook_causal_attention():
    # Special-case reduction: no cached prefix leaves plain causal softmax
    # attention over the new tokens, written here as one masked matrix product.
    P, cache, table, cu, Q, ck, cv = _extend_problem("g32", [0, 0], [5, 9])
    out = paged.extend_attention(cache, P, Q, table, [0, 0], cu, ck, cv)
    for b in range(2):
        lo, hi = cu[b], cu[b + 1]
        for h in range(4):
            g = h // 2
            s = Q[lo:hi, h] @ ck[lo:hi, g].T / np.sqrt(128)
            s[np.triu_indices(hi - lo, 1)] = -np.inf
            assert np.max(np.abs(special.softmax(s, axis=1) @ cv[lo:hi, g] - out[lo:hi, h])) < 1e-12


@pytest.mark.parametrize("v_mode", ["mse", "g32"])
def test_extend_is_masked_attention_over_prefix_and_new_tokens(v_mode):
    # With a prefix: one softmax over [dequantised prefix keys; exact new keys]
    # with a causal mask on the new-token block, built as a single matrix.
    P, cache, table, cu, Q, ck, cv = _extend_problem(v_mode, [40, 17], [6, 3])
    prefix = [40, 17]
    out = paged.extend_attention(cache, P, Q, table, prefix, cu, ck, cv)
    d = 128
    for b in range(2):
        lo, hi = cu[b], cu[b + 1]
        n = hi - lo
        for g in range(2):
            f = paged.read_tokens(cache, P, table[b], prefix[b], g)
            k_hat = quant.mse_reconstruct(f["k_n16"], f["k_idx"], P.R, P.k_centroids)
            k_hat += f["k_rho16"].astype(float)[:, None] * np.sqrt(np.pi / 2) / d * ((2.0 * f["k_bits"] - 1) @ P.S)
            if v_mode == "mse":
                v_hat = quant.mse_reconstruct(f["v_n16"], f["v_codes"], P.R, P.v_centroids)
            else:
                v_hat = quant.group32_reconstruct(f["v_s16"], f["v_z16"], f["v_codes"])
            keys = np.concatenate([k_hat, ck[lo:hi, g]])
            vals = np.concatenate([v_hat, cv[lo:hi, g]])
            mask = np.zeros((n, prefix[b] + n), bool)
            mask[:, prefix[b]:] = np.triu(np.ones((n, n), bool), 1)
            for h in (2 * g, 2 * g + 1):
                s = Q[lo:hi, h] @ keys.T / np.sqrt(d)
                s[mask] = -np.inf
                ref = special.softmax(s, axis=1) @ vals
                assert np.max(np.abs(ref - out[lo:hi, h])) < 1e-10


def test_extend_last_token_of_a_chunk_sees_every_new_token():
    # the chunk's first token sees only itself among the new tokens: changing
    # a later new token leaves its output unchanged, and changes the last one
    P, cache, table, cu, Q, ck, cv = _extend_problem("g32", [20], [4])
    a = paged.extend_attention(cache, P, Q, table, [20], cu, ck, cv)
    ck2, cv2 = ck.copy(), cv.copy()
    ck2[3] += 5.0
    cv2[3] -= 3.0
    b = paged.extend_attention(cache, P, Q, table, [20], cu, ck2, cv2)
    assert np.array_equal(a[:3], b[:3])
    assert np.max(np.abs(a[3] - b[3])) > 1e-3
