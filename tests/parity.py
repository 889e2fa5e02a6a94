"""Test-side helpers: compare a cache written by the CUDA store with the one the
oracle wrote, byte by byte, excusing only the counted boundary cases -- codes
whose fp64 pre-image lies within 1e-6 of a decision boundary, QJL signs with
|(S r)_j| / ||k|| < 1e-6, and fp16 metadata whose pre-image lies within 1e-6
(relative) of an fp16 rounding midpoint (plus everything derived from such a
value in the same vector).  Expected bytes always come from the oracle.

Every comparison also counts the boundary cases of each class, checks that no
class is more frequent than its density allows (a regression that pushed codes
toward the decision points would show up here), and records the counts so that
the test session prints them (tests/conftest.py)."""

import numpy as np

from oracle import codebook, paged

EPS = 1e-6

# (case, counts) of every store comparison made in this process, printed at the
# end of the test session
RECORDED = []


def near_f16_midpoint(x, rel=EPS):
    """True where |x| is within rel*|x| of a midpoint between adjacent fp16 values."""
    x = np.abs(np.asarray(x, np.float64))
    h = x.astype(np.float16)
    lo = np.where(h.astype(np.float64) > x, np.nextafter(h, np.float16(0)), h).astype(np.float64)
    hi = np.nextafter(lo.astype(np.float16), np.float16(np.inf)).astype(np.float64)
    mid = 0.5 * (lo + hi)
    return np.abs(x - mid) <= rel * np.maximum(x, 1e-30)


def near_boundary(y, boundaries, eps=EPS):
    """[N, d] mask: y within eps of any decision boundary."""
    b = np.asarray(boundaries, np.float64)
    return np.min(np.abs(np.asarray(y)[..., None] - b), axis=-1) < eps


def _g32_near_half(pre, exact=None):
    """[N, d] mask: (v - z16)/s16 within 1e-6 of a half-integer (exact=None),
    exactly on one (exact=True) or near but not on one (exact=False)."""
    N, d = pre["v_q"].shape
    t = pre["v_t"].reshape(N, d)
    dist = np.abs(t - np.floor(t) - 0.5)
    if exact is None:
        return dist < EPS
    return dist == 0 if exact else (dist > 0) & (dist < EPS)


def boundary_masks(P, pre):
    """Per-vector / per-coordinate masks of legitimately uncertain fields."""
    L = P.layout
    m = {}
    kc = near_boundary(pre["k_y"], P.k_boundaries)
    kn = near_f16_midpoint(pre["k_n"])
    m["k_codes"] = kc
    m["k_norm"] = kn
    if L.k_qjl:
        n = np.maximum(pre["k_n"], 1e-30)[:, None]
        vec_bad = kc.any(axis=1) | kn
        m["k_signs"] = (np.abs(pre["k_z"]) / n < EPS) | vec_bad[:, None]
        m["k_rnorm"] = near_f16_midpoint(pre["k_rho"]) | vec_bad
    if L.v_mode == "mse":
        m["v_codes"] = near_boundary(pre["v_y"], P.v_boundaries)
        m["v_meta"] = near_f16_midpoint(pre["v_n"])
    else:
        N, d = pre["v_q"].shape
        sc = near_f16_midpoint(pre["v_scale"]) | near_f16_midpoint(pre["v_zero"])  # [N, d/32]
        m["v_codes"] = _g32_near_half(pre) | np.repeat(sc, 32, axis=1)
        m["v_meta"] = sc.any(axis=1)
    return m


def boundary_counts(P, pre):
    """How many decisions of each class lie within 1e-6 of their decision point
    (each counted once, before propagation to the fields derived from it):
      code_near_boundary   key (and MSE value) codes, |y - beta| < 1e-6
      sign_small_unit      QJL signs, |(S r)_j| / ||k|| < 1e-6
      sign_small_raw       the same at raw scale, |(S r)_j| < 1e-6
      f16_near_midpoint    norms, residual norms, group-32 scales and zero
                           points within 1e-6 (relative) of an fp16 midpoint
      g32_near_half        group-32 codes, (v - z16)/s16 within 1e-6 of k + 1/2
                           but not on it
      g32_exact_half       group-32 codes exactly on k + 1/2: bf16 inputs and
                           fp16 scales put t on a lattice, so exact ties occur
                           far more often than a density predicts; both sides
                           compute such a t exactly in fp32 and round it up
                           alike"""
    L = P.layout
    codes = int(near_boundary(pre["k_y"], P.k_boundaries).sum())
    f16 = int(near_f16_midpoint(pre["k_n"]).sum())
    c = {}
    if L.k_qjl:
        n = np.maximum(pre["k_n"], 1e-30)[:, None]
        c["sign_small_unit"] = int((np.abs(pre["k_z"]) / n < EPS).sum())
        c["sign_small_raw"] = int((np.abs(pre["k_z"]) < EPS).sum())
        f16 += int(near_f16_midpoint(pre["k_rho"]).sum())
    if L.v_mode == "mse":
        codes += int(near_boundary(pre["v_y"], P.v_boundaries).sum())
        f16 += int(near_f16_midpoint(pre["v_n"]).sum())
    else:
        c["g32_near_half"] = int(_g32_near_half(pre, exact=False).sum())
        c["g32_exact_half"] = int(_g32_near_half(pre, exact=True).sum())
        f16 += int(near_f16_midpoint(pre["v_scale"]).sum() + near_f16_midpoint(pre["v_zero"]).sum())
    c["code_near_boundary"] = codes
    c["f16_near_midpoint"] = f16
    return c


def _key_distortion(P):
    """Per-vector distortion D = d E[(t - Q(t))^2] of the key codebook: the
    expected fraction of ||k||^2 the residual keeps."""
    sc = codebook.SphereCoordinate(P.d)
    return P.d * codebook.nearest_neighbour_mse(sc, 1.0 / P.d, np.asarray(P.k_centroids, np.float64))


def expected_counts(P, n_vectors):
    """Expected number of boundary cases of each class among n_vectors random
    vectors, from the density f of the decision variable at its decision points
    (P(|X - x0| < eps) = 2 eps f(x0) to first order):
      codes   the rotated unit-vector coordinate has the density f_d of the
              codebook module, so a coordinate meets boundary beta_j with
              probability 2 eps f_d(beta_j);
      signs   for a Gaussian row s, (s.r)/||k|| ~ N(0, ||r||^2/||k||^2) and
              E||r||^2/||k||^2 is the codebook distortion D_b, so the density at
              0 is 1/sqrt(2 pi D_b);
      fp16    a value x in [2^e, 2^(e+1)) has fp16 midpoints 2^(e-10) apart, so
              |x - mid| < eps |x| has probability 2 eps |x| / 2^(e-10), at most
              2 eps 2^11 = 4.1e-3 per value;
      halves  (v - z)/s spreads over a range of 2^b - 1 code steps, so one
              coordinate comes within eps of a half-integer (without sitting
              exactly on it) with probability about 2 eps."""
    L = P.layout
    d = P.d
    f = codebook.SphereCoordinate(d).density
    per_code = 2 * EPS * float(np.sum(f(np.asarray(P.k_boundaries, np.float64))))
    e = {"code_near_boundary": n_vectors * d * per_code}
    n_f16 = 1 + (1 if L.k_qjl else 0)
    if L.v_mode == "mse":
        e["code_near_boundary"] += n_vectors * d * 2 * EPS * float(np.sum(f(np.asarray(P.v_boundaries))))
        n_f16 += 1
    else:
        n_f16 += 2 * (d // 32)
        e["g32_near_half"] = n_vectors * d * 2 * EPS
    e["f16_near_midpoint"] = n_vectors * n_f16 * 2 * EPS * 2**11
    if L.k_qjl:
        D = _key_distortion(P)
        e["sign_small_unit"] = n_vectors * d * 2 * EPS / np.sqrt(2 * np.pi * D)
    return e


def count_bound(expected):
    """An upper bound a Poisson count of mean `expected` exceeds with
    negligible probability (well beyond 5 standard deviations)."""
    return 4.0 * expected + 10.0


def _mask_key(name):
    if name.startswith("k_code"):
        return "k_codes"
    if name.startswith("v_code"):
        return "v_codes"
    return name


def _excused(mask, name, L, byte_in_row):
    """Whether a mismatching byte of a plane row touches an uncertain field."""
    if name == "v_codes" and L.v_mode == "g32":
        lo, hi = byte_in_row * 8 // L.v_bits, (byte_in_row * 8 + 7) // L.v_bits
        coords = paged.group32_slot_coordinates(L.d)[lo:hi + 1]
        return bool(mask[coords].any())
    if name.startswith(("k_code", "v_code", "k_signs")):
        return bool(mask[byte_in_row * 8: byte_in_row * 8 + 8].any())
    return bool(np.any(mask))


def _plane_list(L):
    return L.planes()


def gpu_rows(cache_pages, L, slots, heads, name, base, width):
    """Rows of plane `name` for every (slot, head), slot-major: [len(slots)*heads, width]."""
    slots = np.asarray(slots, np.int64)
    blk = np.repeat(slots // 16, heads)
    row = np.repeat(slots % 16, heads)
    head = np.tile(np.arange(heads), len(slots))
    cols = base + row[:, None] * width + np.arange(width)[None, :]
    return cache_pages[blk[:, None], head[:, None], cols]


def compare_store(cache_pages, P, K, V, slots, heads):
    """Compare the rows a GPU store wrote for tokens with slot >= 0 against the
    oracle's encoding of the same K/V rows.  cache_pages: uint8
    [num_blocks, heads, page_bytes] copied from the device.  Returns
    dict(vectors, checked_bytes, mismatched_bytes, excusable_bytes, unexplained,
    counts, expected, mismatches_by_plane)."""
    L = P.layout
    slots = np.asarray(slots, np.int64)
    keep = np.nonzero(slots >= 0)[0]
    d = K.shape[-1]
    fields, pre = paged.encode(P, np.asarray(K, np.float64)[keep].reshape(-1, d),
                               np.asarray(V, np.float64)[keep].reshape(-1, d))
    masks = boundary_masks(P, pre)
    unexplained, mismatched, checked, excusable = [], 0, 0, 0
    by_plane = {}
    for name, base, width in _plane_list(L):
        got = gpu_rows(cache_pages, L, slots[keep], heads, name, base, width)
        exp = fields[name]
        bad_vec, bad_byte = np.nonzero(got != exp)
        checked += exp.size
        mismatched += len(bad_vec)
        if len(bad_vec):
            by_plane[name] = int(len(bad_vec))
        mk = masks[_mask_key(name)]
        for vec in range(exp.shape[0]) if mk.any() else ():
            if mk[vec].any():
                excusable += sum(_excused(mk[vec], name, L, byte) for byte in range(width))
        for vec, byte in zip(bad_vec, bad_byte):
            if not _excused(mk[vec], name, L, int(byte)):
                unexplained.append((name, int(vec), int(byte), int(got[vec, byte]), int(exp[vec, byte])))
    n_vec = len(keep) * heads
    return dict(vectors=n_vec, checked_bytes=checked, mismatched_bytes=mismatched, excusable_bytes=excusable,
                unexplained=unexplained, counts=boundary_counts(P, pre), expected=expected_counts(P, n_vec),
                mismatches_by_plane=by_plane)


def check_store(r, case, density_bound=True):
    """The parity bar on a compare_store result: every mismatching byte touches
    a counted boundary case, and (for random inputs; density_bound=False for
    hand-made degenerate vectors such as an all-zero key, whose every
    coordinate sits on the middle boundary) every class of boundary case stays
    within the bound its density gives.  Records the counts under `case`."""
    RECORDED.append((case, r))
    assert not r["unexplained"], r["unexplained"][:10]
    assert r["mismatched_bytes"] <= r["excusable_bytes"]
    if density_bound:
        for k, mean in r["expected"].items():
            assert r["counts"].get(k, 0) <= count_bound(mean), (k, r["counts"], r["expected"])


def summary_line(case, r):
    c = r["counts"]
    parts = [f"{k}={c[k]}(exp {r['expected'].get(k, 0):.2g})" for k in sorted(c)]
    return (f"{case}: {r['vectors']} vectors, {r['checked_bytes']} bytes, mismatched {r['mismatched_bytes']} "
            f"(excusable {r['excusable_bytes']}); " + ", ".join(parts))


def output_errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    max_abs = float(np.max(np.abs(got - ref))) if got.size else 0.0
    den = float(np.linalg.norm(ref))
    rel_l2 = float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got - ref))
    return max_abs, rel_l2


MAX_ABS = 2e-3  # attention-output tolerance stated for the path (fp32 out)
REL_L2 = 1e-3
