"""GPU parity of tq_extend_attention against the oracle's extend attention on
the same compressed cache (written by the oracle's store and uploaded): every
new token attends to its sequence's compressed prefix and, causally, to the
exact new tokens.  Same error bar as the decode: max-abs 2e-3, relative L2
1e-3 on an fp32 output."""

import numpy as np
import pytest

import parity
import turboquant_bit_kv_tq_gb300 as tq
from oracle import paged
from turboquant_bit_kv_tq_gb300 import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


class Extend:
    """Sequences with prefix[b] cached tokens (oracle-encoded) and chunk[b]
    new exact bf16 tokens; queries for every new token."""

    def __init__(self, w, prefix, chunk, spare_blocks=2):
        self.w, self.prefix, self.chunk = w, list(prefix), list(chunk)
        self.P = paged.CacheParams(w.d, w.k_bits, w.k_qjl, w.v_mode, w.v_bits, w.seed_rot, w.seed_qjl, w.k_codebook,
                                   w.v_codebook)
        B = len(prefix)
        need = [(n + 15) // 16 for n in prefix]
        self.max_blocks = max(1, max(need))
        self.num_blocks = sum(need) + spare_blocks
        rng = np.random.default_rng((w.seed, 91))
        perm = rng.permutation(self.num_blocks)
        self.table = np.zeros((B, self.max_blocks), np.int32)
        at = 0
        for b, n in enumerate(need):
            self.table[b, :n] = perm[at:at + n]
            at += n
        self.cache = np.zeros((self.num_blocks, w.kv_heads, self.P.layout.page_bytes), np.uint8)
        ks, vs = [], []
        for b in range(B):
            K, V = wl.kv_tokens(w, b, 0, prefix[b])
            t = np.arange(prefix[b])
            paged.store(self.cache, self.P, K, V, self.table[b, t // 16].astype(np.int64) * 16 + t % 16)
            K, V = wl.kv_tokens(w, b, prefix[b], chunk[b])
            ks.append(wl.round_bf16(K))
            vs.append(wl.round_bf16(V))
        self.cu = np.concatenate([[0], np.cumsum(chunk)]).astype(np.int32)
        self.T = int(self.cu[-1])
        self.ck = np.concatenate(ks) if self.T else np.zeros((0, w.kv_heads, w.d), np.float32)
        self.cv = np.concatenate(vs) if self.T else np.zeros((0, w.kv_heads, w.d), np.float32)
        self.Q = wl.queries(w, max(1, self.T))[: self.T]

    def oracle(self):
        return paged.extend_attention(self.cache, self.P, self.Q.astype(np.float64), self.table, self.prefix,
                                      self.cu, self.ck, self.cv)

    def make_cache(self, split_blocks, tail_cap=None, max_batch=None):
        kw = wl.cache_config_kwargs(self.w, num_blocks=self.num_blocks, max_blocks=self.max_blocks,
                                    max_batch=max_batch or max(1, self.T), split_blocks=split_blocks)
        kw["tail_cap"] = tail_cap or max(1, max(self.chunk))
        c = tq.TQCache(**kw)
        c.cache.copy_(torch.from_numpy(self.cache.reshape(-1)))
        return c

    def run(self, c, cu=None, out_dtype=torch.float32):
        dt = torch.bfloat16 if self.w.dtype == "bf16" else torch.float32
        q = torch.from_numpy(np.ascontiguousarray(self.Q)).to("cuda", dt)
        bf = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to("cuda", torch.bfloat16)  # noqa: E731
        cu = self.cu if cu is None else cu
        out = c.extend(q, torch.from_numpy(self.table).cuda(),
                       torch.tensor(self.prefix, dtype=torch.int32, device="cuda"),
                       torch.from_numpy(np.asarray(cu, np.int32)).cuda(), bf(self.ck), bf(self.cv),
                       out_dtype=out_dtype)
        torch.cuda.synchronize()
        return out.float().cpu().numpy()


def _assert_close(got, ref):
    max_abs, rel = parity.output_errors(got, ref)
    assert max_abs <= parity.MAX_ABS and rel <= parity.REL_L2, (max_abs, rel)


CASES = [
    # id, workload, changes, prefix lens, chunk lens, split blocks
    ("gqa4_g32", "llama8b_gqa4_b16_8k", {}, [300, 0, 17], [5, 9, 1], 4),
    ("gqa4_long_chunk", "llama8b_gqa4_b16_8k", {}, [129], [40], 2),
    ("d256_mse", "d256_gqa8_b8_32k", {}, [200, 33], [7, 3], 4),
    ("uniform_k4_gqa8", "llama70b_gqa8_b4_ragged131k_hybrid", dict(k_bits=4, k_codebook="uniform", tail=0),
     [64, 500], [12, 2], 8),
    ("f32_single_head", "single_head_d128_1k", {}, [1024], [8], 8),
    # fp32 queries in the prefix kernel's query blocks (32 virtual heads per
    # prep CTA: S q on tensor cores, the query in three bf16 parts)
    ("gqa4_f32_queries", "llama8b_gqa4_b16_8k", dict(dtype="f32"), [200, 70], [9, 12], 4),
    ("prefill_only", "llama8b_gqa4_b16_8k", {}, [0, 0], [16, 3], 4),
    ("prefill_long_chunks", "llama8b_gqa4_b16_8k", {}, [0, 5], [150, 77], 4),
    ("k4_lloyd_fallback_kernel", "llama8b_gqa4_b16_8k", dict(k_bits=4), [100, 7], [9, 4], 4),
    ("mse_values_chunk", "llama8b_gqa4_b16_8k", dict(v_mode="mse", v_bits=3), [64, 0], [20, 11], 4),
    ("empty_chunk_first", "llama8b_gqa4_b16_8k", {}, [50, 30, 9], [0, 5, 2], 4),
    # the prefix kernel's other instances: 2-bit keys with 2-bit group-32
    # values, 3-bit uniform keys with 4-bit MSE values, keys without QJL
    ("k2_g32v2", "llama8b_gqa4_b16_8k", dict(k_bits=2, v_bits=2), [200, 64], [11, 6], 4),
    ("uniform_k3_mse_v4", "llama8b_gqa4_b16_8k", dict(k_codebook="uniform", v_mode="mse", v_bits=4), [150], [13], 4),
    ("no_qjl_keys", "llama8b_gqa4_b16_8k", dict(k_qjl=False), [90, 33], [9, 17], 2),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_extend_parity(case):
    cid, name, changes, prefix, chunk, sb = case
    w = wl.scaled(wl.config(name), **changes)
    e = Extend(w, prefix, chunk)
    c = e.make_cache(sb)
    got = e.run(c)
    ref = e.oracle()
    _assert_close(got, ref)
    assert c.device_error() == 0
    assert np.abs(ref).max() > 0.1


def test_extend_many_sequences():
    # 70 sequences (the query-block plan's scan spans three warps), chunks of
    # 0..11 tokens and prefixes of 0..90 tokens (some empty), 2-block splits:
    # many blocks and items per CTA
    w = wl.config("llama8b_gqa4_b16_8k")
    rng = np.random.default_rng(21)
    B = 70
    prefix = [int(x) for x in rng.integers(0, 91, B)]
    chunk = [int(x) for x in rng.integers(0, 12, B)]
    for b in rng.choice(B, 6, replace=False):
        prefix[b] = 0
    e = Extend(w, prefix, chunk)
    c = e.make_cache(2)
    got = e.run(c)
    _assert_close(got, e.oracle())
    assert c.device_error() == 0


def test_extend_cuda_graph_replay_with_new_lengths():
    # the grid depends only on the token and sequence counts (the query-block
    # plan is made on the device): capture once, replay with changed prefix
    # lengths and chunk boundaries
    w = wl.config("llama8b_gqa4_b16_8k")
    e = Extend(w, [120, 40, 77], [5, 9, 6])
    c = e.make_cache(2, tail_cap=12)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    q = torch.from_numpy(np.ascontiguousarray(e.Q)).to("cuda", dt)
    bf = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to("cuda", torch.bfloat16)  # noqa: E731
    nk, nv = bf(e.ck), bf(e.cv)
    tab = torch.from_numpy(e.table).cuda()
    pl = torch.tensor(e.prefix, dtype=torch.int32, device="cuda")
    cu = torch.from_numpy(e.cu).cuda()
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c.extend(q, tab, pl, cu, nk, nv, out=out, stream=s)  # warm-up outside capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        c.extend(q, tab, pl, cu, nk, nv, out=out, stream=s)
    for new_prefix, new_cu in (([120, 40, 77], [0, 5, 14, 20]), ([30, 0, 77], [0, 5, 14, 20]),
                               ([120, 16, 1], [0, 10, 14, 20])):
        pl.copy_(torch.tensor(new_prefix, dtype=torch.int32))
        cu.copy_(torch.tensor(new_cu, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        assert c.device_error() == 0
        ref = paged.extend_attention(e.cache, e.P, e.Q.astype(np.float64), e.table, new_prefix,
                                     np.asarray(new_cu, np.int32), e.ck, e.cv)
        _assert_close(out.cpu().numpy(), ref)


def test_extend_invalid_prefix_block_is_flagged():
    # a block-table entry of sequence 1's prefix out of range: flagged, its
    # page skipped; sequence 0 (and its new tokens) are unaffected
    w = wl.config("llama8b_gqa4_b16_8k")
    e = Extend(w, [70, 70], [5, 4])
    c = e.make_cache(2)
    bad = e.table.copy()
    bad[1, 1] = e.num_blocks + 3
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    q = torch.from_numpy(np.ascontiguousarray(e.Q)).to("cuda", dt)
    bf = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to("cuda", torch.bfloat16)  # noqa: E731
    out = c.extend(q, torch.from_numpy(bad).cuda(), torch.tensor(e.prefix, dtype=torch.int32, device="cuda"),
                   torch.from_numpy(e.cu).cuda(), bf(e.ck), bf(e.cv), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert c.device_error() & tq.TQ_DEVERR_BLOCK
    got = out.cpu().numpy()
    _assert_close(got[:5], e.oracle()[:5])
    assert np.isfinite(got).all()


def test_extend_rows_outside_every_chunk_are_zero_and_flagged():
    w = wl.config("llama8b_gqa4_b16_8k")
    e = Extend(w, [40, 20], [3, 4])
    c = e.make_cache(4)
    bad_cu = np.array([0, 3, 5], np.int32)  # rows 5 and 6 belong to no chunk
    got = e.run(c, cu=bad_cu)
    assert c.device_error() == tq.TQ_DEVERR_CHUNK
    assert np.all(got[5:] == 0)
    # rows 0..4 are the extend of sequences with chunks [3, 2]
    ref = paged.extend_attention(e.cache, e.P, e.Q[:5].astype(np.float64), e.table, e.prefix, bad_cu, e.ck[:5],
                                 e.cv[:5])
    _assert_close(got[:5], ref)


def test_extend_chunk_longer_than_tail_cap_is_flagged():
    w = wl.config("llama8b_gqa4_b16_8k")
    e = Extend(w, [32], [6])
    c = e.make_cache(4, tail_cap=4)
    got = e.run(c)
    assert c.device_error() == tq.TQ_DEVERR_TAIL
    _assert_close(got[:4], e.oracle()[:4])  # tokens within the cap are exact


def test_extend_more_tokens_than_max_batch_is_rejected():
    w = wl.config("llama8b_gqa4_b16_8k")
    e = Extend(w, [16], [5])
    c = e.make_cache(4, max_batch=4)
    with pytest.raises(tq.TQError):
        e.run(c)


def test_extend_bf16_output():
    w = wl.config("llama8b_gqa4_b16_8k")
    e = Extend(w, [100], [6])
    c = e.make_cache(4)
    got = e.run(c, out_dtype=torch.bfloat16)
    ref = e.oracle()
    assert np.max(np.abs(got - ref)) <= 8e-3 * max(1.0, np.abs(ref).max())


def test_extend_full_size_sampled():
    """The bench's extend context line (8B shape, 4 sequences x 4096-token
    prefix + 256 new tokens, 128-block splits) in its launch configuration:
    every prefix is filled by the GPU store (not compared); the pages of two
    sampled (sequence, KV head) pairs are then overwritten with the oracle's
    encoding, and sampled new tokens of those pairs are compared."""
    prefix, chunk, batch = 4096, 256, 4
    w = wl.scaled(wl.config("llama8b_gqa4_b16_8k"), batch=batch, seq_lens=[prefix] * batch)
    P = paged.CacheParams(w.d, w.k_bits, w.k_qjl, w.v_mode, w.v_bits, w.seed_rot, w.seed_qjl, w.k_codebook,
                          w.v_codebook)
    table, num_blocks = wl.block_table(w)
    T = batch * chunk
    kw = wl.cache_config_kwargs(w, num_blocks=num_blocks, max_blocks=table.shape[1], max_batch=T, split_blocks=128)
    kw["tail_cap"] = chunk
    c = tq.TQCache(**kw)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    t = np.arange(prefix)
    for b in range(batch):
        K, V = wl.kv_tokens_device(w, prefix, gen)
        c.store(K, V, torch.from_numpy(table[b, t // 16].astype(np.int64) * 16 + t % 16).cuda())
    torch.cuda.synchronize()
    assert c.device_error() == 0
    pages = c.pages()
    picks = [(1, 3), (3, 6)]
    ones = {}
    for b, g in picks:
        one = np.zeros((num_blocks, 1, P.layout.page_bytes), np.uint8)
        K, V = wl.kv_tokens(w, b, 0, prefix, heads=[g])
        paged.store(one, P, K, V, table[b, t // 16].astype(np.int64) * 16 + t % 16)
        used = torch.from_numpy(np.unique(table[b]).astype(np.int64)).cuda()
        pages[used, g] = torch.from_numpy(one[:, 0]).cuda()[used]
        ones[(b, g)] = one
    ck = np.concatenate([wl.round_bf16(wl.kv_tokens(w, b, prefix, chunk)[0]) for b in range(batch)])
    cv = np.concatenate([wl.round_bf16(wl.kv_tokens(w, b, prefix, chunk)[1]) for b in range(batch)])
    Q = wl.queries(w, T)
    bf = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to("cuda", torch.bfloat16)  # noqa: E731
    cu = np.arange(0, T + 1, chunk, dtype=np.int32)
    out = c.extend(bf(Q), torch.from_numpy(table).cuda(), torch.full((batch,), prefix, dtype=torch.int32,
                                                                     device="cuda"),
                   torch.from_numpy(cu).cuda(), bf(ck), bf(cv))
    torch.cuda.synchronize()
    assert c.device_error() == 0
    got = out.cpu().numpy()
    G = w.group
    for (b, g), one in ones.items():
        for j in (0, 100, chunk - 1):
            row = b * chunk + j
            lo = b * chunk
            ref = paged.decode_attention(one, P, Q[row:row + 1, g * G:(g + 1) * G].astype(np.float64), table[b:b + 1],
                                         [prefix], tail_k=ck[None, lo:row + 1, g:g + 1].transpose(0, 2, 1, 3),
                                         tail_v=cv[None, lo:row + 1, g:g + 1].transpose(0, 2, 1, 3),
                                         tail_lens=[j + 1])
            _assert_close(got[row, g * G:(g + 1) * G], ref[0])
