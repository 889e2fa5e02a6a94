"""GPU parity of tq_store against the oracle: every byte of every written row is
bit-exact except the counted boundary cases (tests/parity.py)."""

import numpy as np
import pytest

import parity
import turboquant_bit_kv_tq_gb300 as tq
from oracle import paged
from turboquant_bit_kv_tq_gb300 import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _cache_for(w, num_blocks):
    return tq.TQCache(**wl.cache_config_kwargs(w, num_blocks=num_blocks, max_blocks=4, max_batch=1))


def _oracle_params(w):
    return paged.CacheParams(w.d, w.k_bits, w.k_qjl, w.v_mode, w.v_bits, w.seed_rot, w.seed_qjl,
                             w.k_codebook, w.v_codebook)


def _to_dev(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to(device="cuda", dtype=torch.bfloat16 if dtype == "bf16" else torch.float32)


def _run(w, K, V, slots, num_blocks):
    c = _cache_for(w, num_blocks)
    c.store(_to_dev(K, w.dtype), _to_dev(V, w.dtype), torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    pages = c.pages().cpu().numpy()
    err = c.device_error()
    return pages, err


def _check(w, K, V, slots, num_blocks, case, expect_err=0, density_bound=True):
    pages, err = _run(w, K, V, slots, num_blocks)
    assert err == expect_err
    P = _oracle_params(w)
    r = parity.compare_store(pages, P, K, V, slots, w.kv_heads)
    parity.check_store(r, case, density_bound)
    # untouched rows stay zero: rebuild the set of written (block,row) pairs
    written = np.zeros((num_blocks, 16), bool)
    s = slots[slots >= 0]
    written[s // 16, s % 16] = True
    L = P.layout
    for name, base, width in parity._plane_list(L):
        rows = pages[:, :, base:base + 16 * width].reshape(num_blocks, w.kv_heads, 16, width)
        assert not rows.transpose(0, 2, 1, 3)[~written].any(), name
    return r


CASES = [
    # name, d, H, k_bits, v_mode, v_bits, dtype, qjl, n_out, scale[, codebook]
    ("c1_like_f32", 128, 1, 2, "mse", 2, "f32", True, 4, 20.0),
    ("c2_like", 128, 8, 3, "g32", 4, "bf16", True, 3, 10.0),
    ("c3_like_d256", 256, 4, 2, "mse", 2, "bf16", True, 5, 15.0),
    ("k4_v2g32", 128, 2, 4, "g32", 2, "bf16", True, 3, 10.0),
    ("d256_f32_k3_g32v2", 256, 2, 3, "g32", 2, "f32", True, 5, 15.0),
    ("no_qjl_v4mse", 128, 2, 3, "mse", 4, "bf16", False, 3, 10.0),
    ("k4_v3mse_d256", 256, 1, 4, "mse", 3, "bf16", True, 5, 15.0),
    ("uniform_k4_v4mse", 128, 2, 4, "mse", 4, "bf16", True, 3, 10.0, "uniform"),
    ("uniform_k3_v2mse_d256", 256, 1, 3, "mse", 2, "f32", True, 5, 15.0, "uniform"),
    ("k2_v3mse", 128, 4, 2, "mse", 3, "bf16", True, 3, 10.0),
    ("k2_v4g32", 128, 2, 2, "g32", 4, "bf16", True, 3, 10.0),
]


@pytest.fixture(params=["per_vector", "persistent"])
def store_path(request):
    """Run a store test through the one-CTA-per-vector kernel (the default for
    a few thousand vectors) or the persistent kernel (forced)."""
    tq.tq_set_store_small_max(-1 if request.param == "per_vector" else 0)
    yield request.param
    tq.tq_set_store_small_max(-1)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_store_parity_small(case, store_path):
    name, d, H, kb, vm, vb, dt, qjl, n_out, sc = case[:10]
    cb = case[10] if len(case) > 10 else "lloyd"
    w = wl.Workload(name, d, H, H, kb, vm, vb, dt, n_out, sc, seed=11, k_qjl=qjl, batch=1, seq_lens=[300],
                    k_codebook=cb, v_codebook=cb if vm == "mse" else "lloyd")
    T = 300
    K, V = wl.kv_tokens(w, 0, 0, T)
    num_blocks = 24  # 384 slots, 300 used + ragged
    rng = np.random.default_rng(5)
    slots = rng.permutation(num_blocks * 16)[:T].astype(np.int64)
    slots[rng.choice(T, 7, replace=False)] = -1
    r = _check(w, K, V, slots, num_blocks, f"{name}/{store_path}")
    assert r["checked_bytes"] > 0


def test_store_edge_vectors(store_path):
    # zero vectors, constant groups, identical keys, x1e3 outliers, ragged block
    w = wl.Workload("edges", 128, 2, 2, 3, "g32", 4, "bf16", 3, 10.0, seed=12, batch=1, seq_lens=[40])
    K, V = wl.kv_tokens(w, 0, 0, 40)
    K[0] = 0.0
    V[0] = 0.0
    V[1, :, :32] = 2.5
    K[2] = K[3]
    V[2] = V[3]
    K[4, :, 7] *= 1e3
    V[4, :, 7] *= 1e3
    K, V = wl.round_bf16(K), wl.round_bf16(V)
    slots = np.arange(3, 43, dtype=np.int64)  # starts mid-block, ends mid-block
    _check(w, K, V, slots, 4, f"edge_vectors/{store_path}", density_bound=False)


def test_store_skip_and_bad_slot_sets_device_error(store_path):
    w = wl.Workload("badslot", 128, 2, 2, 2, "mse", 2, "bf16", 3, 10.0, seed=13, batch=1, seq_lens=[20])
    K, V = wl.kv_tokens(w, 0, 0, 20)
    slots = np.arange(20, dtype=np.int64)
    slots[3] = -1          # skipped silently
    slots[5] = 2 * 16      # == num_slots for 2 blocks: out of range
    slots[6] = -7          # invalid negative
    pages, err = _run(w, K, V, slots, 2)
    assert err == tq.TQ_DEVERR_SLOT
    ok = slots.copy()
    ok[[5, 6]] = -1
    P = _oracle_params(w)
    r = parity.compare_store(pages, P, K, V, ok, w.kv_heads)
    parity.check_store(r, f"bad_slot/{store_path}")


@pytest.mark.parametrize("offset_elems", [0, 2], ids=["aligned_full_tiles", "rows_4B_aligned_only"])
def test_store_bulk_tile_edges(offset_elems):
    # 256 tokens x 2 KV heads = 512 vectors, exactly four 128-vector tiles,
    # through the bulk path.  With the K and V rows 4- but not 16-byte aligned
    # (a view two bf16 elements into its buffer) the tensor-core store cannot
    # use bulk-tensor copies and the eight-vectors-per-CTA kernel must take the
    # call; either way every byte matches the oracle up to counted cases.
    w = wl.Workload("tiles", 128, 2, 2, 3, "mse", 2, "bf16", 3, 10.0, seed=14, batch=1, seq_lens=[256])
    T = 256
    K, V = wl.kv_tokens(w, 0, 0, T)
    num_blocks = 20
    rng = np.random.default_rng(9)
    slots = rng.permutation(num_blocks * 16)[:T].astype(np.int64)
    c = _cache_for(w, num_blocks)

    def dev_view(x):
        flat = torch.zeros(x.size + offset_elems, dtype=torch.bfloat16, device="cuda")
        flat[offset_elems:] = torch.from_numpy(np.ascontiguousarray(x).reshape(-1)).cuda().to(torch.bfloat16)
        return flat[offset_elems:].view(x.shape)

    k, v = dev_view(K), dev_view(V)
    assert (k.data_ptr() % 16 == 0) == (offset_elems == 0)
    tq.tq_set_store_small_max(0)  # bulk path
    try:
        c.store(k, v, torch.from_numpy(slots).cuda())
        torch.cuda.synchronize()
    finally:
        tq.tq_set_store_small_max(-1)
    assert c.device_error() == 0
    r = parity.compare_store(c.pages().cpu().numpy(), _oracle_params(w), K, V, slots, w.kv_heads)
    parity.check_store(r, f"bulk_tiles/{offset_elems}")
    assert r["checked_bytes"] > 0


def test_store_zero_tokens_is_noop():
    w = wl.Workload("empty", 128, 1, 1, 2, "mse", 2, "bf16", 0, 1.0, seed=1, batch=1, seq_lens=[1])
    c = _cache_for(w, 2)
    k = torch.zeros((0, 1, 128), dtype=torch.bfloat16, device="cuda")
    c.store(k, k, torch.zeros(0, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert not c.cache.any().item()


def test_store_full_size_sampled():
    # The store workload at full size (65,536 tokens x 8 KV heads into a
    # 1M-token pool) in the launch configuration the benchmark times; the oracle
    # re-encodes a random sample of 1,024 tokens and their rows must match.
    w = wl.config("store_64seq_65536tok")
    lens, prior, table, slots = wl.store_layout(w)
    K, V = wl.store_tokens(w)
    c = _cache_for(w, w.pool_blocks)
    c.store(_to_dev(K, w.dtype), _to_dev(V, w.dtype), torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    assert c.device_error() == 0
    rng = np.random.default_rng(0)
    pick = np.sort(rng.choice(len(slots), 1024, replace=False))
    P = _oracle_params(w)
    L = P.layout
    # gather only the sampled slots' pages to the host
    blocks = torch.from_numpy(np.unique(slots[pick] // 16)).cuda()
    sub = c.pages()[blocks].cpu().numpy()
    remap = {int(b): i for i, b in enumerate(blocks.cpu().numpy())}
    sub_slots = np.array([remap[int(s) // 16] * 16 + int(s) % 16 for s in slots[pick]], np.int64)
    r = parity.compare_store(sub, P, K[pick], V[pick], sub_slots, w.kv_heads)
    parity.check_store(r, "store_64seq_65536tok/sampled1024")
    assert r["checked_bytes"] == 1024 * 8 * (L.page_bytes // 16)
