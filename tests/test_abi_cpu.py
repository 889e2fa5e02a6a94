"""CPU checks of the C-ABI library: it loads, exports every function
include/tq_kv.h declares, and its host-side tables (codebooks, rotation signs,
QJL matrix, page sizes) equal the oracle's independently generated ones.  No
compute call needs a GPU here."""

import os
import re

import numpy as np
import pytest

import turboquant_bit_kv_tq_gb300 as tq
from oracle import codebook, paged, prng

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    if not os.path.exists(tq.library_path()):
        from turboquant_bit_kv_tq_gb300 import _build

        _build.build()
    tq.load_library()


def test_header_functions_all_exported():
    with open(os.path.join(ROOT, "include", "tq_kv.h")) as f:
        text = f.read()
    declared = sorted(set(re.findall(r"^\s*(?:tq_status|const char\*)\s+(tq_\w+)\s*\(", text, re.M)))
    assert declared == sorted(tq.EXPORTED)
    lib = tq.load_library()
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings():
    assert tq.tq_status_string(0) == "ok"
    for s in (-1, -2, -3, -4, -5):
        assert tq.tq_status_string(s) != "unknown status"


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_codebook_matches_oracle(d, bits):
    c, b, mse = tq.tq_make_codebook(d, bits)
    oc, ob = codebook.sphere_codebook(d, bits)
    assert np.max(np.abs(c - oc)) < 1e-11
    assert np.max(np.abs(b - ob)) < 1e-11
    # the fp32 tables the kernels use are then identical
    assert np.array_equal(c.astype(np.float32), oc.astype(np.float32))
    assert np.array_equal(b.astype(np.float32), ob.astype(np.float32))
    assert abs(mse - codebook.per_vector_mse(d, oc)) < 1e-10


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_uniform_codebook_matches_oracle(d, bits):
    c, b, mse = tq.tq_make_uniform_codebook(d, bits)
    oc, ob = codebook.sphere_uniform_codebook(d, bits)
    assert np.max(np.abs(c - oc)) < 1e-11
    assert np.max(np.abs(b - ob)) < 1e-11
    assert np.array_equal(c.astype(np.float32), oc.astype(np.float32))
    assert np.array_equal(b.astype(np.float32), ob.astype(np.float32))
    step = c[1] - c[0]
    assert np.allclose(np.diff(c), step, rtol=1e-12, atol=0)
    assert abs(mse - d * codebook.nearest_neighbour_mse(codebook.SphereCoordinate(d), 1.0 / d, oc)) < 1e-10


def test_uniform_codebook_high_bits_is_stationary():
    # 8 bits: the step the library finds makes the distortion stationary
    # (sum k M = step sum k^2 P over the midpoint cells), checked with the
    # oracle's density functions
    d, L = 128, 256
    c, b, _ = tq.tq_make_uniform_codebook(d, 8)
    dist = codebook.SphereCoordinate(d)
    k = np.arange(L) - (L - 1) / 2.0
    step = (c[-1] - c[0]) / (L - 1)
    edges = np.concatenate([[-1.0], b, [1.0]])
    g = np.sum(k * dist.moment(edges[:-1], edges[1:])) - step * np.sum(k * k * dist.mass(edges[:-1], edges[1:]))
    assert abs(g) < 1e-9 * step * np.sum(k * k * dist.mass(edges[:-1], edges[1:]))


def test_page_bytes_do_not_depend_on_the_codebook():
    base = dict(head_dim=128, num_kv_heads=1, num_q_heads=1, num_blocks=2, k_bits=4, v_mode=0, v_bits=3,
                max_blocks_per_seq=2)
    uni = tq.tq_cache_sizes(tq.tq_cache_config(**base, k_codebook=1, v_codebook=1))
    assert uni == tq.tq_cache_sizes(tq.tq_cache_config(**base))


@pytest.mark.parametrize("d,seed", [(128, 2), (256, 2), (128, 12345)])
def test_rotation_signs_match_oracle(d, seed):
    assert np.array_equal(tq.tq_make_rotation_signs(d, seed), prng.rotation_signs(d, seed).astype(np.float32))


@pytest.mark.parametrize("d,seed", [(128, 1), (256, 1), (128, 99)])
def test_qjl_matrix_matches_oracle(d, seed):
    bits = tq.tq_make_qjl_matrix(d, seed).astype(np.uint32) << 16
    lib_vals = bits.view(np.float32).astype(np.float64)
    assert np.array_equal(lib_vals, prng.qjl_matrix(d, seed))


@pytest.mark.parametrize("d,kb,vm,vb", [(128, 2, 0, 2), (128, 3, 1, 4), (256, 2, 0, 2), (128, 4, 1, 2),
                                        (256, 3, 0, 3), (256, 4, 1, 4)])
def test_page_bytes_match_oracle_layout(d, kb, vm, vb):
    cfg = tq.tq_cache_config(head_dim=d, num_kv_heads=8, num_q_heads=32, num_blocks=10, k_bits=kb, v_mode=vm,
                             v_bits=vb, max_blocks_per_seq=4)
    sizes = tq.tq_cache_sizes(cfg)
    lay = paged.PageLayout(d, kb, True, "mse" if vm == 0 else "g32", vb)
    assert sizes["page_bytes"] == lay.page_bytes
    assert sizes["cache_bytes"] == 10 * 8 * lay.page_bytes
    assert sizes["page_bytes"] % 16 == 0


def test_bad_configs_are_rejected_on_the_host():
    ok = dict(head_dim=128, num_kv_heads=8, num_q_heads=32, num_blocks=10, k_bits=3, v_mode=1, v_bits=4,
              max_blocks_per_seq=4)
    tq.tq_cache_sizes(tq.tq_cache_config(**ok))
    for bad, status in [(dict(head_dim=64), -2), (dict(k_bits=5), -2), (dict(v_bits=1), -2), (dict(block_size=32), -2),
                        (dict(num_q_heads=30), -1), (dict(num_blocks=0), -1), (dict(v_mode=7), -2),
                        (dict(split_blocks=0), -1), (dict(tail_cap=-1), -1), (dict(v_mode=1, v_bits=3), -2),
                        (dict(num_q_heads=48), -2), (dict(k_codebook=2), -1), (dict(v_codebook=-1), -1),
                        (dict(v_codebook=1), -1)]:
        with pytest.raises(tq.TQError) as e:
            tq.tq_cache_sizes(tq.tq_cache_config(**{**ok, **bad}))
        assert e.value.status == status, bad


def test_extend_binding_checks_shapes_before_any_call():
    torch = pytest.importorskip("torch")
    q = torch.zeros((5, 4, 128))
    table = torch.zeros((2, 3), dtype=torch.int32)
    pl = torch.zeros(2, dtype=torch.int32)
    cu = torch.tensor([0, 2, 5], dtype=torch.int32)
    kv = torch.zeros((5, 1, 128), dtype=torch.bfloat16)
    out = torch.zeros((5, 4, 128))
    with pytest.raises(ValueError):
        tq.tq_extend_attention(None, q, None, table, pl, cu, kv[:4], kv, out)
    with pytest.raises(ValueError):
        tq.tq_extend_attention(None, q, None, table, pl, cu[:2], kv, kv, out)
    with pytest.raises(ValueError):
        tq.tq_extend_attention(None, q, None, table[:1], pl, cu, kv, kv, out)
    with pytest.raises(ValueError):  # CPU tensors never reach the library
        tq.tq_extend_attention(None, q, torch.zeros(16, dtype=torch.uint8), table, pl, cu, kv, kv, out)


def test_store_decode_entry_checks_arguments_before_any_launch():
    torch = pytest.importorskip("torch")
    lib = tq.load_library()
    # a null cache handle is refused before anything reaches CUDA
    st = lib.tq_store_decode_attention(None, None, None, tq.TQ_DTYPE_BF16, 0, None, None, tq.TQ_DTYPE_BF16, None,
                                       None, None, None, None, None, 0.0, 1, None, tq.TQ_DTYPE_F32, None)
    assert st == -1  # TQ_ERR_INVALID_ARG
    # the binding checks shapes and devices first
    k = torch.zeros((2, 8, 128), dtype=torch.bfloat16)
    q = torch.zeros((2, 32, 128), dtype=torch.bfloat16)
    slots = torch.zeros(2, dtype=torch.int64)
    table = torch.zeros((2, 4), dtype=torch.int32)
    lens = torch.zeros(2, dtype=torch.int32)
    out = torch.zeros((2, 32, 128))
    with pytest.raises(ValueError):  # k and v differ
        tq.tq_store_decode_attention(None, k, k[:1], slots, q, None, table, lens, out)
    with pytest.raises(ValueError):  # CPU tensors never reach the library
        tq.tq_store_decode_attention(None, k, k, slots, q, torch.zeros(16, dtype=torch.uint8), table, lens, out)
