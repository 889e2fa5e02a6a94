"""The fused decode step (tq_store_decode_attention): store the new tokens,
then decode, in one call.

Its contract is the two calls in order, bit for bit: the same cache bytes and
the same outputs as tq_store followed by tq_decode_attention.  Inside the call
the decode's query pass reads the queries while the store kernel still runs,
and must write nothing (and the split kernel read no page) before the store
has finished; a decode that missed the new token, or read a page half written,
would differ from the two-call sequence.  The steps below append one token per
sequence several times in a row, so each decode reads the token its own call
stored.
"""

import numpy as np
import pytest

import parity
import turboquant_bit_kv_tq_gb300 as tq
from turboquant_bit_kv_tq_gb300 import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _caches(w, lens, steps, split_blocks, tail_cap=0, seed=0):
    """Two caches filled alike with lens[b] tokens per sequence, with room for
    `steps` more; the block table and the fill's generator are shared."""
    need = [(n + steps + 15) // 16 for n in lens]
    num_blocks = sum(need) + 2
    table = np.zeros((len(lens), max(need)), np.int32)
    perm = np.random.default_rng(seed).permutation(num_blocks)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[at:at + n]
        at += n
    kw = wl.cache_config_kwargs(w, num_blocks=num_blocks, max_blocks=table.shape[1], max_batch=len(lens),
                                split_blocks=split_blocks)
    kw["tail_cap"] = tail_cap
    out = []
    for _ in range(2):
        c = tq.TQCache(**kw)
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed)
        for b, n in enumerate(lens):
            if n == 0:
                continue
            t = np.arange(n)
            slots = torch.from_numpy(table[b, t // 16].astype(np.int64) * 16 + t % 16).cuda()
            K, V = wl.kv_tokens_device(w, n, gen)
            c.store(K, V, slots)
        out.append(c)
    torch.cuda.synchronize()
    return out[0], out[1], table


def _same(got, ref, what):
    if not np.array_equal(got, ref):
        max_abs, _ = parity.output_errors(got.astype(np.float64), ref.astype(np.float64))
        raise AssertionError(f"{what} differ: {np.count_nonzero(got != ref)} elements, max-abs {max_abs:.3e}")


def _run_steps(w, lens, steps, split_blocks, q_dtype, tail_cap=0, seed=0):
    ca, cb, table = _caches(w, lens, steps, split_blocks, tail_cap, seed)
    B = len(lens)
    table_d = torch.from_numpy(table).cuda()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed + 100)
    tail = (None, None, None)
    if tail_cap:
        tk = torch.randn((B, w.kv_heads, tail_cap, w.d), generator=gen, device="cuda").to(torch.bfloat16)
        tv = torch.randn((B, w.kv_heads, tail_cap, w.d), generator=gen, device="cuda").to(torch.bfloat16)
        tl = torch.tensor([(3 * b + 1) % (tail_cap + 1) for b in range(B)], dtype=torch.int32, device="cuda")
        tail = (tk, tv, tl)
    cur = np.array(lens, np.int64)
    for step in range(steps):
        K, V = wl.kv_tokens_device(w, B, gen)
        slots = torch.from_numpy(table[np.arange(B), cur // 16].astype(np.int64) * 16 + cur % 16).cuda()
        cur += 1
        seq = torch.from_numpy(cur.astype(np.int32)).cuda()
        q = torch.randn((B, w.q_heads, w.d), generator=gen, device="cuda").to(q_dtype)
        ref = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        got = torch.empty_like(ref)
        ca.store(K, V, slots)
        tq.tq_decode_attention(ca.handle, q, ca.cache, table_d, seq, ref, *tail)
        tq.tq_store_decode_attention(cb.handle, K, V, slots, q, cb.cache, table_d, seq, got, *tail)
        torch.cuda.synchronize()
        _same(cb.cache.cpu().numpy(), ca.cache.cpu().numpy(), f"step {step}: cache bytes")
        _same(got.cpu().numpy(), ref.cpu().numpy(), f"step {step}: outputs")
        assert np.abs(ref.cpu().numpy()).max() > 0.05
    assert ca.device_error() == 0 and cb.device_error() == 0
    return ca, cb, table_d


@pytest.mark.parametrize("name,lens,split_blocks,q_dtype,tail_cap", [
    # the grouped-query decode the split kernel's staged schedule serves, ragged lengths
    ("llama8b_gqa4_b16_8k", [700, 33, 1, 250], 4, torch.bfloat16, 0),
    # fp32 queries, a length that starts a new page on the first append
    ("llama8b_gqa4_b16_8k", [16, 511, 95], 8, torch.float32, 0),
    # d = 256, MSE values, exact tail
    ("d256_gqa8_b8_32k", [300, 17], 8, torch.bfloat16, 16),
])
def test_store_decode_matches_store_then_decode(name, lens, split_blocks, q_dtype, tail_cap):
    w = wl.scaled(wl.config(name), batch=len(lens), tail=tail_cap)
    _run_steps(w, lens, 3, split_blocks, q_dtype, tail_cap, seed=len(lens))


def test_store_decode_with_no_new_token_is_the_decode():
    w = wl.scaled(wl.config("llama8b_gqa4_b16_8k"), batch=2)
    ca, cb, table = _caches(w, [200, 64], 0, 4, seed=3)
    seq = torch.tensor([200, 64], dtype=torch.int32, device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(9)
    q = torch.randn((2, w.q_heads, w.d), generator=gen, device="cuda").to(torch.bfloat16)
    K = torch.zeros((0, w.kv_heads, w.d), dtype=torch.bfloat16, device="cuda")
    slots = torch.zeros(0, dtype=torch.int64, device="cuda")
    ref = ca.decode(q, torch.from_numpy(table).cuda(), seq)
    got = cb.store_decode(K, K, slots, q, torch.from_numpy(table).cuda(), seq)
    torch.cuda.synchronize()
    _same(got.cpu().numpy(), ref.cpu().numpy(), "outputs")
    _same(cb.cache.cpu().numpy(), ca.cache.cpu().numpy(), "cache bytes")


def test_store_decode_checks_every_argument_before_storing():
    w = wl.scaled(wl.config("llama8b_gqa4_b16_8k"), batch=2)
    ca, cb, table = _caches(w, [40, 8], 1, 4, seed=4)
    before = cb.cache.cpu().numpy()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(11)
    K, V = wl.kv_tokens_device(w, 2, gen)
    slots = torch.tensor([table[0, 2] * 16 + 8, table[1, 0] * 16 + 8], dtype=torch.int64, device="cuda")
    # three query rows against a cache made for two sequences: the decode's
    # batch check fails, and the store must not have run
    q = torch.randn((3, w.q_heads, w.d), generator=gen, device="cuda").to(torch.bfloat16)
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    seq = torch.tensor([41, 9, 0], dtype=torch.int32, device="cuda")
    with pytest.raises(tq.TQError) as e:
        tq.tq_store_decode_attention(cb.handle, K, V, slots, q, cb.cache, torch.from_numpy(table).cuda(), seq, out)
    assert e.value.status == -1  # TQ_ERR_INVALID_ARG
    torch.cuda.synchronize()
    _same(cb.cache.cpu().numpy(), before, "cache bytes after a rejected call")
