"""Runtime behaviour on the GPU: the per-device launch set-up made by the first
calls of several host threads at once, and the error path of the decode
kernels' bounded waits."""

import os
import subprocess
import sys
import time

import numpy as np
import pytest

import turboquant_bit_kv_tq_gb300 as tq
from turboquant_bit_kv_tq_gb300 import workloads as wl

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Runs in a fresh process, so that the threads make the first store and decode
# calls on the device: four threads (two cache configurations, each twice),
# each with its own cache and stream, store and decode at the same time after a
# barrier.  Their outputs must equal a single-threaded rerun of the same calls.
_CHILD = r"""
import sys, threading
import numpy as np, torch
sys.path.insert(0, {root!r})
import turboquant_bit_kv_tq_gb300 as tq
from turboquant_bit_kv_tq_gb300 import workloads as wl

torch.cuda.set_device(0)
tq.load_library()

def setup(name, batch, lens, seed):
    w = wl.scaled(wl.config(name), batch=batch, seq_lens=lens)
    table, nb = wl.block_table(w)
    kw = wl.cache_config_kwargs(w, num_blocks=nb, max_blocks=table.shape[1], split_blocks=4)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    n = sum(lens)
    K, V = wl.kv_tokens_device(w, n, gen)
    slots = []
    for b, m in enumerate(lens):
        t = np.arange(m)
        slots.append(table[b, t // 16].astype(np.int64) * 16 + t % 16)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    q = torch.randn((batch, w.q_heads, w.d), generator=gen, device="cuda").to(dt)
    return dict(kw=kw, K=K, V=V, slots=torch.from_numpy(np.concatenate(slots)).cuda(),
                table=torch.from_numpy(table).cuda(), lens=torch.tensor(lens, dtype=torch.int32, device="cuda"), q=q)

problems = [setup("llama8b_gqa4_b16_8k", 3, [300, 40, 129], 1), setup("d256_gqa8_b8_32k", 2, [200, 77], 2)]
jobs = [problems[i % 2] for i in range(4)]
caches = [tq.TQCache(**p["kw"]) for p in jobs]
streams = [torch.cuda.Stream() for _ in jobs]
outs = [None] * len(jobs)
errs = []
torch.cuda.synchronize()
gate = threading.Barrier(len(jobs))

def work(i):
    try:
        p, c, s = jobs[i], caches[i], streams[i]
        gate.wait()
        c.store(p["K"], p["V"], p["slots"], stream=s)
        out = c.decode(p["q"], p["table"], p["lens"], stream=s)
        s.synchronize()
        outs[i] = out.cpu().numpy()
    except Exception as e:
        errs.append(repr(e))

threads = [threading.Thread(target=work, args=(i,)) for i in range(len(jobs))]
for t in threads:
    t.start()
for t in threads:
    t.join()
assert not errs, errs
for i, (p, c) in enumerate(zip(jobs, caches)):
    assert c.device_error() == 0
    again = tq.TQCache(**p["kw"])
    again.store(p["K"], p["V"], p["slots"])
    ref = again.decode(p["q"], p["table"], p["lens"]).cpu().numpy()
    assert np.array_equal(outs[i], ref), (i, float(np.abs(outs[i] - ref).max()))
    assert torch.equal(c.cache, again.cache), i
print("threads ok", len(jobs))
"""


def test_first_calls_from_several_threads_at_once():
    r = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT)], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "threads ok 4" in r.stdout


def test_bounded_wait_gives_up_with_an_error_status():
    # an mbarrier phase nothing completes, waited for through the kernels'
    # bounded polling loop with a 20 ms time limit added: the kernel must end
    # by itself, set TQ_DEVERR_TIMEOUT, and leave the context usable
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    tq.tq_check_wait_timeout(err, 20000)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(err.item()) == tq.TQ_DEVERR_TIMEOUT
    assert 0.015 <= elapsed < 5.0, elapsed
    # a decode afterwards runs normally
    w = wl.scaled(wl.config("llama8b_gqa4_b16_8k"), batch=1, seq_lens=[64])
    table, nb = wl.block_table(w)
    c = tq.TQCache(**wl.cache_config_kwargs(w, num_blocks=nb, max_blocks=table.shape[1], split_blocks=2))
    K, V = wl.kv_tokens(w, 0, 0, 64)
    t = np.arange(64)
    slots = torch.from_numpy(table[0, t // 16].astype(np.int64) * 16 + t % 16).cuda()
    c.store(torch.from_numpy(K).cuda().to(torch.bfloat16), torch.from_numpy(V).cuda().to(torch.bfloat16), slots)
    q = torch.from_numpy(wl.queries(w)).cuda().to(torch.bfloat16)
    out = c.decode(q, torch.from_numpy(table).cuda(), torch.tensor([64], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert c.device_error() == 0
    assert torch.isfinite(out).all() and out.abs().max().item() > 0


def test_wait_timeout_rejects_bad_arguments():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for limit in (0, 4 * 10**6 + 1):
        with pytest.raises(tq.TQError):
            tq.tq_check_wait_timeout(err, limit)
