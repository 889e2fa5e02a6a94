"""GPU parity of tq_decode_attention against the oracle on the same compressed
cache.  The cache is written by the oracle's store (never by the GPU) and
uploaded; the GPU output must match the oracle's decode within max-abs 2e-3
and relative-L2 1e-3 (fp32 output)."""

import numpy as np
import pytest

import bench
import parity
import turboquant_bit_kv_tq_gb300 as tq
from oracle import paged
from turboquant_bit_kv_tq_gb300 import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _params(w):
    return paged.CacheParams(w.d, w.k_bits, w.k_qjl, w.v_mode, w.v_bits, w.seed_rot, w.seed_qjl,
                             w.k_codebook, w.v_codebook)


def _dev(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda", torch.bfloat16 if dtype == "bf16" else torch.float32)


class Problem:
    """A decode problem whose cache the oracle writes: per-sequence compressed
    and tail lengths, block table, queries and the oracle's cache image."""

    def __init__(self, w, comp, tail=None, tail_cap=0, spare_blocks=3):
        self.w = w
        self.P = _params(w)
        self.B = len(comp)
        self.comp = list(comp)
        self.tail = list(tail) if tail is not None else None
        self.tail_cap = tail_cap
        need = [(n + 15) // 16 for n in comp]
        self.max_blocks = max(1, max(need))
        self.num_blocks = sum(need) + spare_blocks
        rng = np.random.default_rng((w.seed, 77))
        perm = rng.permutation(self.num_blocks)
        self.table = np.full((self.B, self.max_blocks), 0, np.int32)
        at = 0
        for b, n in enumerate(need):
            self.table[b, :n] = perm[at:at + n]
            at += n
        self.cache = np.zeros((self.num_blocks, w.kv_heads, self.P.layout.page_bytes), np.uint8)
        for b in range(self.B):
            K, V = wl.kv_tokens(w, b, 0, comp[b])
            t = np.arange(comp[b])
            paged.store(self.cache, self.P, K, V, self.table[b, t // 16].astype(np.int64) * 16 + t % 16)
        self.Q = wl.queries(w, self.B)
        if self.tail is not None:
            self.tk = np.zeros((self.B, w.kv_heads, tail_cap, w.d), np.float32)
            self.tv = np.zeros_like(self.tk)
            for b in range(self.B):
                K, V = wl.kv_tokens(w, b, comp[b], self.tail[b])
                K, V = wl.round_bf16(K), wl.round_bf16(V)
                self.tk[b, :, : self.tail[b]] = K.transpose(1, 0, 2)
                self.tv[b, :, : self.tail[b]] = V.transpose(1, 0, 2)

    def oracle(self, scale=None, Q=None):
        Q = self.Q if Q is None else Q
        kw = {}
        if self.tail is not None:
            kw = dict(tail_k=self.tk, tail_v=self.tv, tail_lens=self.tail)
        return paged.decode_attention(self.cache, self.P, np.asarray(Q, np.float64), self.table, self.comp,
                                      scale=scale, **kw)

    def gpu_inputs(self):
        d = dict(block_table=torch.from_numpy(self.table).cuda(), seq_lens=torch.tensor(self.comp, dtype=torch.int32,
                                                                                       device="cuda"))
        if self.tail is not None:
            d.update(tail_k=_dev(self.tk, "bf16"), tail_v=_dev(self.tv, "bf16"),
                     tail_lens=torch.tensor(self.tail, dtype=torch.int32, device="cuda"))
        return d


def _make_cache(prob, split_blocks, max_batch=None):
    kw = wl.cache_config_kwargs(prob.w, num_blocks=prob.num_blocks, max_blocks=prob.max_blocks,
                                max_batch=max_batch or prob.B, split_blocks=split_blocks)
    kw["tail_cap"] = prob.tail_cap
    c = tq.TQCache(**kw)
    c.cache.copy_(torch.from_numpy(prob.cache.reshape(-1)))
    return c


def _decode(prob, c, out_dtype=torch.float32, scale=0.0, Q=None):
    Q = prob.Q if Q is None else Q
    q = _dev(Q, prob.w.dtype)
    out = torch.empty(q.shape, dtype=out_dtype, device="cuda")
    inp = prob.gpu_inputs()
    c.decode(q, inp["block_table"], inp["seq_lens"], out=out, tail_k=inp.get("tail_k"), tail_v=inp.get("tail_v"),
             tail_lens=inp.get("tail_lens"), scale=scale)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def _assert_close(got, ref):
    max_abs, rel = parity.output_errors(got, ref)
    assert max_abs <= parity.MAX_ABS and rel <= parity.REL_L2, (max_abs, rel)


def _wl(name, **kw):
    return wl.scaled(wl.config(name), **kw)


CASES = [
    # id, workload, compressed lens, tail lens, tail cap, split blocks
    ("single_head_full", "single_head_d128_1k", {}, [1024], None, 0, 8),
    ("gqa4_ragged", "llama8b_gqa4_b16_8k", {}, [0, 1, 15, 16, 17, 300], None, 0, 4),
    ("d256_gqa8", "d256_gqa8_b8_32k", {}, [1, 33, 700], None, 0, 8),
    # fp32 queries with eight heads per prep CTA at d=256: the prep's S q on
    # tensor cores, the query in three bf16 parts
    ("d256_gqa8_f32q", "d256_gqa8_b8_32k", dict(dtype="f32"), [65, 300], None, 0, 8),
    ("hybrid_gqa8", "llama70b_gqa8_b4_ragged131k_hybrid", {}, [15, 16, 500, 0], [0, 5, 128, 3], 128, 4),
    ("mse3_tail", "d256_gqa8_b8_32k", dict(v_bits=3, k_bits=4, tail=32), [40, 0], [7, 32], 32, 1),
    ("g32v2_k2", "llama8b_gqa4_b16_8k", dict(v_bits=2, k_bits=2), [129, 64], None, 0, 2),
    ("f32_gqa1", "single_head_d128_1k", dict(q_heads=2, kv_heads=2), [77, 255], None, 0, 3),
    # MSE-only keys (no QJL plane): the ablation of the residual correction
    ("no_qjl_g32", "llama8b_gqa4_b16_8k", dict(k_qjl=False), [300, 129, 17], None, 0, 4),
    ("no_qjl_d256_mse", "d256_gqa8_b8_32k", dict(k_qjl=False), [200, 33], None, 0, 4),
    # uniform codebooks (single-bit score planes only on the warp-specialized
    # kernel at d=128; every plane elsewhere)
    ("uniform_k3_g32", "llama8b_gqa4_b16_8k", dict(k_codebook="uniform"), [300, 129, 17], None, 0, 4),
    ("uniform_k4_v4mse", "llama8b_gqa4_b16_8k",
     dict(k_bits=4, k_codebook="uniform", v_mode="mse", v_bits=4, v_codebook="uniform"), [300, 33, 0, 1], None, 0, 4),
    ("uniform_k4_no_qjl", "llama8b_gqa4_b16_8k", dict(k_bits=4, k_codebook="uniform", k_qjl=False), [257, 64], None,
     0, 2),
    ("uniform_k4_hybrid", "llama70b_gqa8_b4_ragged131k_hybrid", dict(k_bits=4, k_codebook="uniform"), [15, 500],
     [5, 128], 128, 4),
    ("uniform_d256_k3", "d256_gqa8_b8_32k", dict(k_bits=3, k_codebook="uniform", v_codebook="uniform"), [200, 33],
     None, 0, 4),
    ("uniform_k2_f32", "single_head_d128_1k", dict(k_codebook="uniform", v_codebook="uniform"), [1024], None, 0, 8),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_decode_parity_small(case):
    cid, name, changes, comp, tail, cap, sb = case
    w = _wl(name, **changes)
    prob = Problem(w, comp, tail, cap)
    c = _make_cache(prob, sb)
    got = _decode(prob, c)
    ref = prob.oracle()
    _assert_close(got, ref)
    assert c.device_error() == 0
    if sum(comp) + (sum(tail) if tail else 0) > 0:
        assert np.abs(ref).max() > 0.1  # non-trivial output


def test_decode_rotated_output_is_R_times_out():
    # MSE values with TQ_OUT_ROTATED: the output stays in the rotated space, so
    # it must equal R times the oracle's output (R orthogonal: the same error
    # bar applies); group-32 values reject the flag
    w = _wl("d256_gqa8_b8_32k")
    prob = Problem(w, [300, 45])
    c = _make_cache(prob, 4)
    inp = prob.gpu_inputs()
    q = _dev(prob.Q, w.dtype)
    got = c.decode(q, inp["block_table"], inp["seq_lens"], rotated=True)
    torch.cuda.synchronize()
    ref = prob.oracle() @ prob.P.R.T  # out @ R^T = (R out) per row
    _assert_close(got.cpu().numpy(), ref)
    w2 = _wl("llama8b_gqa4_b16_8k")
    prob2 = Problem(w2, [40])
    c2 = _make_cache(prob2, 2)
    inp2 = prob2.gpu_inputs()
    with pytest.raises(tq.TQError):
        c2.decode(_dev(prob2.Q, w2.dtype), inp2["block_table"], inp2["seq_lens"], rotated=True)


def test_decode_empty_sequences_give_zero():
    w = _wl("llama8b_gqa4_b16_8k")
    prob = Problem(w, [0, 0, 0])
    got = _decode(prob, _make_cache(prob, 2))
    assert np.all(got == 0)


def test_decode_bf16_output_and_explicit_scale():
    w = _wl("llama8b_gqa4_b16_8k")
    prob = Problem(w, [100, 250])
    c = _make_cache(prob, 4)
    ref = prob.oracle(scale=0.05)
    got = _decode(prob, c, out_dtype=torch.bfloat16, scale=0.05)
    # bf16 output: oracle value rounded to bf16 plus the fp32 tolerance
    assert np.all(np.abs(got - ref) <= parity.MAX_ABS + 2.0**-8 * np.abs(ref))


def test_decode_extreme_logits_no_nan():
    # queries x1e3: logit spreads of thousands; softmax must stay finite
    w = _wl("llama8b_gqa4_b16_8k")
    prob = Problem(w, [200, 31])
    Q = prob.Q * 1e3
    got = _decode(prob, _make_cache(prob, 2), Q=Q)
    assert np.all(np.isfinite(got))
    _assert_close(got, prob.oracle(Q=Q))


def test_decode_invalid_block_is_flagged_and_skipped():
    w = _wl("llama8b_gqa4_b16_8k")
    prob = Problem(w, [64, 64])
    c = _make_cache(prob, 2)
    bad = prob.table.copy()
    bad[1, 2] = prob.num_blocks + 5  # out of range
    inp = prob.gpu_inputs()
    q = _dev(prob.Q, w.dtype)
    out = c.decode(q, torch.from_numpy(bad).cuda(), inp["seq_lens"])
    torch.cuda.synchronize()
    assert c.device_error() & tq.TQ_DEVERR_BLOCK
    # sequence 0 is untouched; sequence 1 equals attention over its other
    # three blocks, i.e. the oracle reading a table without block 2
    ref = prob.oracle()
    got = out.cpu().numpy()
    _assert_close(got[0], ref[0])
    sub = Problem.__new__(Problem)
    sub.__dict__.update(prob.__dict__)
    table2 = prob.table.copy()
    table2[1, 2:] = np.r_[prob.table[1, 3:], 0]
    sub.table, sub.comp = table2, [64, 48]
    _assert_close(got[1], sub.oracle()[1])


def test_decode_seq_len_beyond_table_is_flagged():
    w = _wl("llama8b_gqa4_b16_8k")
    prob = Problem(w, [32])
    c = _make_cache(prob, 1)
    q = _dev(prob.Q, w.dtype)
    c.decode(q, torch.from_numpy(prob.table).cuda(), torch.tensor([10**6], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert c.device_error() & tq.TQ_DEVERR_SEQLEN


def test_decode_negative_seq_len_is_flagged_and_empty():
    # a negative length is flagged and read as 0; the other sequence is intact
    w = _wl("llama8b_gqa4_b16_8k")
    prob = Problem(w, [32, 64])
    c = _make_cache(prob, 1)
    q = _dev(prob.Q, w.dtype)
    lens = torch.tensor([-5, 64], dtype=torch.int32, device="cuda")
    out = c.decode(q, torch.from_numpy(prob.table).cuda(), lens)
    torch.cuda.synchronize()
    assert c.device_error() & tq.TQ_DEVERR_SEQLEN
    got = out.cpu().numpy()
    assert np.all(got[0] == 0)
    _assert_close(got[1], prob.oracle()[1])


def test_decode_cuda_graph_replay_with_new_lengths():
    # the grid depends only on the configuration: capture once, replay with
    # changed sequence lengths and block tables (fixed-grid requirement of
    # [Roadmap] §3.2)
    w = _wl("llama8b_gqa4_b16_8k")
    prob = Problem(w, [300, 150, 40], spare_blocks=0)
    c = _make_cache(prob, 4)
    q = _dev(prob.Q, w.dtype)
    table = torch.from_numpy(prob.table).cuda()
    lens = torch.tensor(prob.comp, dtype=torch.int32, device="cuda")
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c.decode(q, table, lens, out=out, stream=s)  # warm-up outside capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        c.decode(q, table, lens, out=out, stream=s)
    for new_lens in ([300, 150, 40], [17, 0, 40], [299, 151, 1]):
        lens.copy_(torch.tensor(new_lens, dtype=torch.int32))
        sub_table = prob.table.copy()
        sub_table[[0, 1]] = sub_table[[1, 0]] if new_lens[0] < 200 else sub_table[[0, 1]]
        table.copy_(torch.from_numpy(sub_table))
        g.replay()
        torch.cuda.synchronize()
        ref = paged.decode_attention(prob.cache, prob.P, prob.Q.astype(np.float64), sub_table, new_lens)
        _assert_close(out.cpu().numpy(), ref)


def _sampled_full_size(name, picks, split_blocks, changes=None):
    """Full-size workload in the benchmark's launch configuration: every
    sequence's cache is filled by the GPU store (not compared), then the pages
    of the sampled (sequence, KV head) pairs are overwritten with the oracle's
    encoding and those query-head outputs are compared."""
    w = wl.scaled(wl.config(name), **(changes or {}))
    P = _params(w)
    table, num_blocks = wl.block_table(w)
    comp = w.compressed_lens()
    kw = wl.cache_config_kwargs(w, num_blocks=num_blocks, max_blocks=table.shape[1], split_blocks=split_blocks)
    c = tq.TQCache(**kw)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1)
    for b in range(w.batch):
        t = np.arange(comp[b])
        slots = torch.from_numpy(table[b, t // 16].astype(np.int64) * 16 + t % 16).cuda()
        K, V = wl.kv_tokens_device(w, comp[b], gen)
        c.store(K, V, slots)
    torch.cuda.synchronize()
    assert c.device_error() == 0
    pages = c.pages()
    oracle_caches = {}
    for b, g in picks:
        one = np.zeros((num_blocks, 1, P.layout.page_bytes), np.uint8)
        K, V = wl.kv_tokens(w, b, 0, comp[b], heads=[g])
        t = np.arange(comp[b])
        paged.store(one, P, K, V, table[b, t // 16].astype(np.int64) * 16 + t % 16)
        used = torch.from_numpy(np.unique(table[b, : (comp[b] + 15) // 16]).astype(np.int64)).cuda()
        pages[used, g] = torch.from_numpy(one[:, 0]).cuda()[used]
        oracle_caches[(b, g)] = one
    tail = None
    if w.tail:
        tail_lens = w.tail_lens()
        tk = torch.zeros((w.batch, w.kv_heads, w.tail, w.d), dtype=torch.bfloat16, device="cuda")
        tv = torch.zeros_like(tk)
        tk_np = np.zeros((w.batch, w.kv_heads, w.tail, w.d), np.float32)
        tv_np = np.zeros_like(tk_np)
        for b in range(w.batch):
            K, V = wl.kv_tokens(w, b, comp[b], tail_lens[b])
            tk_np[b, :, : tail_lens[b]] = K.transpose(1, 0, 2)
            tv_np[b, :, : tail_lens[b]] = V.transpose(1, 0, 2)
        tk.copy_(torch.from_numpy(tk_np))
        tv.copy_(torch.from_numpy(tv_np))
        tail = (tk, tv, torch.tensor(tail_lens, dtype=torch.int32, device="cuda"), tk_np, tv_np, tail_lens)
    Q = wl.queries(w)
    q = _dev(Q, w.dtype)
    out = c.decode(q, torch.from_numpy(table).cuda(), torch.tensor(comp, dtype=torch.int32, device="cuda"),
                   tail_k=tail[0] if tail else None, tail_v=tail[1] if tail else None,
                   tail_lens=tail[2] if tail else None)
    torch.cuda.synchronize()
    assert c.device_error() == 0
    got = out.cpu().numpy()
    G = w.group
    for (b, g), one in oracle_caches.items():
        kw = {}
        if tail:
            kw = dict(tail_k=tail[3][b:b + 1, g:g + 1], tail_v=tail[4][b:b + 1, g:g + 1], tail_lens=[tail[5][b]])
        ref = paged.decode_attention(one, P, Q[b:b + 1, g * G:(g + 1) * G].astype(np.float64), table[b:b + 1],
                                     [comp[b]], **kw)
        _assert_close(got[b, g * G:(g + 1) * G], ref[0])


def test_decode_full_size_llama8b_sampled():
    _sampled_full_size("llama8b_gqa4_b16_8k", [(0, 0), (9, 5), (15, 7)],
                       split_blocks=bench._split_blocks(wl.config("llama8b_gqa4_b16_8k")))


def test_decode_full_size_d256_sampled():
    _sampled_full_size("d256_gqa8_b8_32k", [(3, 1), (7, 3)],
                       split_blocks=bench._split_blocks(wl.config("d256_gqa8_b8_32k")))


def test_decode_full_size_llama8b_uniform_k4_sampled():
    _sampled_full_size("llama8b_gqa4_b16_8k", [(2, 1), (12, 6)],
                       split_blocks=bench._split_blocks(wl.config("llama8b_gqa4_b16_8k")),
                       changes=dict(k_bits=4, k_codebook="uniform"))


def test_decode_full_size_hybrid131k_sampled():
    w = wl.config("llama70b_gqa8_b4_ragged131k_hybrid")
    longest = int(np.argmax(w.seq_lens))
    _sampled_full_size("llama70b_gqa8_b4_ragged131k_hybrid", [(longest, 2)], split_blocks=bench._split_blocks(w))
