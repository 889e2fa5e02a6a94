"""Test-side helpers: compare a cache written by the CUDA store with the one the
oracle wrote, byte by byte, excusing only the counted boundary cases -- codes
whose fp64 pre-image lies within 1e-6 of a decision boundary, QJL signs with
|(S r)_j| / ||k|| < 1e-6, and fp16 metadata whose pre-image lies within 1e-6
(relative) of an fp16 rounding midpoint (plus everything derived from such a
value in the same vector).  Expected bytes always come from the oracle."""

import numpy as np

from oracle import paged

EPS = 1e-6


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
        t = pre["v_t"].reshape(N, d)
        half = np.abs(t - np.floor(t) - 0.5) < EPS
        m["v_codes"] = half | np.repeat(sc, 32, axis=1)
        m["v_meta"] = sc.any(axis=1)
    return m


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
    dict(checked_bytes, mismatched_bytes, unexplained, boundary_fields)."""
    L = P.layout
    slots = np.asarray(slots, np.int64)
    keep = np.nonzero(slots >= 0)[0]
    d = K.shape[-1]
    fields, pre = paged.encode(P, np.asarray(K, np.float64)[keep].reshape(-1, d),
                               np.asarray(V, np.float64)[keep].reshape(-1, d))
    masks = boundary_masks(P, pre)
    unexplained, mismatched, checked = [], 0, 0
    for name, base, width in _plane_list(L):
        got = gpu_rows(cache_pages, L, slots[keep], heads, name, base, width)
        exp = fields[name]
        bad_vec, bad_byte = np.nonzero(got != exp)
        checked += exp.size
        mismatched += len(bad_vec)
        for vec, byte in zip(bad_vec, bad_byte):
            if not _excused(masks[_mask_key(name)][vec], name, L, int(byte)):
                unexplained.append((name, int(vec), int(byte), int(got[vec, byte]), int(exp[vec, byte])))
    counted = {k: int(np.sum(v)) for k, v in masks.items()}
    return dict(checked_bytes=checked, mismatched_bytes=mismatched, unexplained=unexplained,
                boundary_fields=counted)


def output_errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    max_abs = float(np.max(np.abs(got - ref))) if got.size else 0.0
    den = float(np.linalg.norm(ref))
    rel_l2 = float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got - ref))
    return max_abs, rel_l2


MAX_ABS = 2e-3  # attention-output tolerance stated for the path (fp32 out)
REL_L2 = 1e-3
