"""The allocation-free decode entry point (tq_decode_attention_noalloc).

It exists for callers that cannot allocate device memory themselves -- an
engine whose memory manager owns the whole GPU, or code that must not cause the
synchronisation a cudaMalloc can bring -- and keeps its split-KV scratch in the
library's static device array instead of a caller workspace.  It runs the same
kernels on the same inputs as tq_decode_attention, whose work is dealt out and
reduced in a fixed order, so its outputs must equal that entry point's bit for
bit, call after call, although the array keeps whatever the previous call left
in it (a stale scratch read would show up as a difference of any size).  This
file is collected last on purpose.
"""

import numpy as np
import pytest

import parity
import turboquant_bit_kv_tq_gb300 as tq
from turboquant_bit_kv_tq_gb300 import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _filled_cache(w, lens, split_blocks, tail_cap=0, seed=0):
    need = [(n + 15) // 16 for n in lens]
    num_blocks = sum(need) + 2
    table = np.zeros((len(lens), max(1, max(need))), np.int32)
    perm = np.random.default_rng(seed).permutation(num_blocks)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[at:at + n]
        at += n
    kw = wl.cache_config_kwargs(w, num_blocks=num_blocks, max_blocks=table.shape[1], max_batch=len(lens),
                                split_blocks=split_blocks)
    kw["tail_cap"] = tail_cap
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
    torch.cuda.synchronize()
    return c, torch.from_numpy(table).cuda(), torch.tensor(lens, dtype=torch.int32, device="cuda")


def _both(c, q, table, lens, tail=None):
    ref = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    got = torch.empty_like(ref)
    tk, tv, tl = tail if tail else (None, None, None)
    tq.tq_decode_attention(c.handle, q, c.cache, table, lens, ref, tk, tv, tl)
    tq.tq_decode_attention_noalloc(c.handle, q, c.cache, table, lens, got, tk, tv, tl)
    torch.cuda.synchronize()
    return got.cpu().numpy(), ref.cpu().numpy()


def _close(got, ref):
    if not np.array_equal(got, ref):
        max_abs, rel = parity.output_errors(got, ref)
        raise AssertionError(f"outputs differ: {np.count_nonzero(got != ref)} elements, max-abs {max_abs:.3e}")


def test_noalloc_decode_matches_workspace_decode_on_consecutive_calls():
    # call 1: grouped-query decode with 4-bit group-32 values, ragged lengths
    w1 = wl.scaled(wl.config("llama8b_gqa4_b16_8k"), batch=3)
    c1, table1, lens1 = _filled_cache(w1, [700, 33, 0], split_blocks=4, seed=1)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    q1 = torch.randn((3, w1.q_heads, w1.d), generator=gen, device="cuda").to(torch.bfloat16)
    got1, ref1 = _both(c1, q1, table1, lens1)
    _close(got1, ref1)
    assert np.abs(ref1).max() > 0.1
    # call 2, right after: another configuration (MSE values, exact tail),
    # reusing the scratch the first call left behind
    w2 = wl.scaled(wl.config("d256_gqa8_b8_32k"), batch=2, tail=16)
    c2, table2, lens2 = _filled_cache(w2, [300, 17], split_blocks=8, tail_cap=16, seed=2)
    q2 = torch.randn((2, w2.q_heads, w2.d), generator=gen, device="cuda").to(torch.bfloat16)
    tk = torch.randn((2, w2.kv_heads, 16, w2.d), generator=gen, device="cuda").to(torch.bfloat16)
    tv = torch.randn((2, w2.kv_heads, 16, w2.d), generator=gen, device="cuda").to(torch.bfloat16)
    tl = torch.tensor([16, 5], dtype=torch.int32, device="cuda")
    got2, ref2 = _both(c2, q2, table2, lens2, (tk, tv, tl))
    _close(got2, ref2)
    # and the first problem again: no state carried over
    got3, ref3 = _both(c1, q1, table1, lens1)
    _close(got3, ref1)
    assert c1.device_error() == 0 and c2.device_error() == 0


def test_noalloc_rejects_workspace_beyond_the_static_array():
    # 16 sequences x 32 query heads x 128 splits of 128 floats: just over 32 MiB
    w = wl.scaled(wl.config("llama8b_gqa4_b16_8k"), batch=1)
    kw = wl.cache_config_kwargs(w, num_blocks=4, max_blocks=4096, max_batch=16, split_blocks=32)
    c = tq.TQCache(**kw)
    assert c.sizes["workspace_bytes"] > 32 << 20
    q = torch.zeros((1, w.q_heads, w.d), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((1, w.q_heads, w.d), dtype=torch.float32, device="cuda")
    table = torch.zeros((1, 4096), dtype=torch.int32, device="cuda")
    lens = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_attention_noalloc(c.handle, q, c.cache, table, lens, out)
    assert e.value.status == -3  # TQ_ERR_BUFFER_TOO_SMALL
