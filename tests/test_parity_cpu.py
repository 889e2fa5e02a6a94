"""CPU checks of the parity helpers themselves (tests/parity.py): the store
comparison finds no difference between two identical oracle encodings, flags a
planted byte error that no boundary case explains, and the density-derived
boundary-case expectations agree with counts measured on the oracle's own
pre-images (at a wider epsilon, where the counts are large enough to test)."""

import numpy as np
import pytest

import parity
from oracle import paged
from turboquant_bit_kv_tq_gb300 import workloads as wl


def _params(w):
    return paged.CacheParams(w.d, w.k_bits, w.k_qjl, w.v_mode, w.v_bits, w.seed_rot, w.seed_qjl,
                             w.k_codebook, w.v_codebook)


def _oracle_cache(w, K, V, slots, num_blocks):
    P = _params(w)
    cache = np.zeros((num_blocks, w.kv_heads, P.layout.page_bytes), np.uint8)
    paged.store(cache, P, K, V, slots)
    return P, cache


@pytest.mark.parametrize("name", ["store_64seq_65536tok", "llama8b_gqa4_b16_8k"])
def test_identical_caches_compare_clean(name):
    w = wl.config(name)
    K, V = wl.kv_tokens(w, 0, 0, 64)
    slots = np.arange(5, 69, dtype=np.int64)
    P, cache = _oracle_cache(w, K, V, slots, 5)
    r = parity.compare_store(cache, P, K, V, slots, w.kv_heads)
    assert r["mismatched_bytes"] == 0 and not r["unexplained"]
    assert r["vectors"] == 64 * w.kv_heads
    assert r["checked_bytes"] == 64 * w.kv_heads * (P.layout.page_bytes // 16)
    for k, mean in r["expected"].items():
        assert r["counts"].get(k, 0) <= parity.count_bound(mean)


def test_planted_byte_error_is_unexplained():
    w = wl.config("store_64seq_65536tok")
    K, V = wl.kv_tokens(w, 0, 0, 32)
    slots = np.arange(32, dtype=np.int64)
    P, cache = _oracle_cache(w, K, V, slots, 2)
    L = P.layout
    bad = cache.copy()
    bad[1, 3, L.k_signs + 5 * L.bit_row + 2] ^= 0x10  # one sign bit of token 21, head 3
    r = parity.compare_store(bad, P, K, V, slots, w.kv_heads)
    assert r["mismatched_bytes"] == 1
    assert r["unexplained"] and r["unexplained"][0][0] == "k_signs"
    with pytest.raises(AssertionError):
        parity.check_store(r, "planted")
    parity.RECORDED.pop()


def _poisson_ok(count, mean, lo_factor=1.0, hi_factor=1.0):
    """count within 5 sigma of [lo_factor*mean, hi_factor*mean]."""
    return lo_factor * mean - 5 * np.sqrt(mean) - 3 <= count <= hi_factor * mean + 5 * np.sqrt(mean) + 3


def test_density_expectations_match_oracle_counts():
    # the store workload's shape, 1,024 tokens x 8 heads: the boundary classes
    # counted at eps = 1e-3 / rel = 1e-4 (many hits) against the same formulas
    w = wl.config("store_64seq_65536tok")
    K, V = wl.kv_tokens(w, 0, 0, 1024)
    P = _params(w)
    d = w.d
    _, pre = paged.encode(P, np.asarray(K, np.float64).reshape(-1, d), np.asarray(V, np.float64).reshape(-1, d))
    n = pre["k_y"].shape[0]
    from oracle import codebook

    f = codebook.SphereCoordinate(d).density
    eps = 1e-3
    got = int(parity.near_boundary(pre["k_y"], P.k_boundaries, eps).sum())
    mean = n * d * 2 * eps * float(np.sum(f(np.asarray(P.k_boundaries))))
    assert _poisson_ok(got, mean, 0.9, 1.1), (got, mean)
    # QJL projections at unit-key scale
    zn = np.abs(pre["k_z"]) / pre["k_n"][:, None]
    got = int((zn < eps).sum())
    mean = n * d * 2 * eps / np.sqrt(2 * np.pi * parity._key_distortion(P))
    assert _poisson_ok(got, mean, 0.85, 1.15), (got, mean)
    # fp16 midpoints: between 2 rel 2^10 and 2 rel 2^11 per value
    rel = 1e-4
    vals = np.concatenate([pre["k_n"], pre["k_rho"], pre["v_n"]])
    got = int(parity.near_f16_midpoint(vals, rel).sum())
    assert _poisson_ok(got, len(vals) * 2 * rel * 2**11, 0.5, 1.0), (got, len(vals))
    # group-32 half-integers on the 8B-shaped workload's 4-bit values
    w2 = wl.config("llama8b_gqa4_b16_8k")
    K2, V2 = wl.kv_tokens(w2, 0, 0, 512)
    P2 = _params(w2)
    _, pre2 = paged.encode(P2, np.asarray(K2, np.float64).reshape(-1, d), np.asarray(V2, np.float64).reshape(-1, d))
    t = pre2["v_t"].reshape(pre2["v_q"].shape)
    dist = np.abs(t - np.floor(t) - 0.5)
    got = int(((dist > 0) & (dist < eps)).sum())
    mean = t.size * 2 * eps
    assert _poisson_ok(got, mean, 0.85, 1.15), (got, mean)
