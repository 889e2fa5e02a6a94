#!/usr/bin/env python
"""Throughput of the TurboQuant KV-cache hot path on GB300.

One step = one decode step of one attention layer for the whole batch: the
fused store of every sequence's new token followed by decode attention over
the compressed paged cache, in one tq_store_decode_attention call (the same
results as tq_store then tq_decode_attention), on seeded
synthetic data with the workload's shapes.  Default workload: the
Llama-3.1-8B-shaped decode layer (32 query / 8 KV heads, d=128, batch 16,
8,192-token contexts, 3-bit keys + QJL, 4-bit group-32 values).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is KV tokens attended per second over
the whole job (sum of context lengths / step time, summed over ranks; every
rank runs its own replica: weak scaling).  Beside the headline, the same line
carries the d=256 GQA-8 decode and the 70B-shaped ragged 131K hybrid decode
(`decode_workloads`, each with its split kernel's roofline), the store and
extend workloads, the oracle's CPU timing (one thread and all host cores) and
the counted boundary cases of a re-encoded store sample.  The reference arm
(--impl reference) times the CPU oracle on a bounded sample of the same
workload, on all host cores.
"""

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 256 << 20
DEFAULT_WORKLOAD = "llama8b_gqa4_b16_8k"
METRIC = "decode-attn KV tokens/s & achieved HBM GB/s vs peak; store tokens/s"
UNIT = "KV tokens/s"


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--split-blocks", type=int, default=0, help="KV blocks per decode split (0: per workload)")
    p.add_argument("--no-qjl", action="store_true",
                   help="ablation: MSE-only keys (no QJL sign plane or residual norm) on the same workload")
    p.add_argument("--k-bits", type=int, default=0, help="key code bits (0: the workload's)")
    p.add_argument("--codebook", choices=["lloyd", "uniform"], default="lloyd",
                   help="codebook of the keys (and of MSE values): Lloyd-Max or the uniform grid")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-store-workload", action="store_true")
    p.add_argument("--no-extend-workload", action="store_true")
    p.add_argument("--no-decode-workloads", action="store_true",
                   help="skip the d=256 and 70B-shaped hybrid decode lines")
    p.add_argument("--no-boundary-cases", action="store_true")
    p.add_argument("--store-only", action="store_true",
                   help="time only the store workload and print its line (a profiling entry point)")
    p.add_argument("--extend-only", action="store_true",
                   help="time only the extend workload and print its line (a profiling entry point)")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    return p.parse_args()


# the decode workloads timed beside the headline, each with its own roofline
EXTRA_DECODES = ["d256_gqa8_b8_32k", "llama70b_gqa8_b4_ragged131k_hybrid"]
# arithmetic of the timed path: scores as four e4m3 pieces of the query
# operand against exact e4m3 bit-plane operands, probabilities x values as fp16
# high/low pieces against exact fp16 code operands, fp32 accumulation and
# softmax; the store in fp32 with bf16-split tensor-core projections
DTYPE = "e4m3x4 score pieces, f16 hi/lo P.V, f32 accumulate"


# ------------------------------------------------------------------ helpers
def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# the sources the decode split kernels are compiled from and launched by: a
# change to any of them makes a traffic record stale (other kernels' files,
# e.g. the store's or extend's prefix kernel, do not)
_SPLIT_SOURCES = ("tq_decode_ws.cuh", "tq_decode_kernels.cuh", "tq_device.cuh", "tq_internal.h", "tq_decode.cu",
                  "tq_host.cpp")


def _kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "turboquant_bit_kv_tq_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name in _SPLIT_SOURCES or name.startswith("tq_decode_split_"):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


_TRAFFIC_RE = re.compile(r"traffic record: kernel=(\S+) workload=(\S+) source_hash=([0-9a-f]+) "
                         r"dram_bytes_per_launch=(\d+)")


def _ncu_traffic(kernel, workload):
    """DRAM bytes (read + write) per launch from a committed ncu summary under
    profiles/ (its "traffic record" line), if that capture was taken on the
    current kernel sources; else None."""
    want = _kernel_source_hash()
    pdir = os.path.join(ROOT, "profiles")
    try:
        names = sorted(os.listdir(pdir))
    except OSError:
        return None
    for name in names:
        if not name.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, name)) as f:
            for m in _TRAFFIC_RE.finditer(f.read()):
                if m.group(1) == kernel and m.group(2) == workload and m.group(3) == want:
                    return int(m.group(4))
    return None


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 50 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "50"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, device):
    """The largest of every rank's x (the job's step time is its slowest
    replica's); x itself on one process."""
    import torch

    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def traffic_key(w):
    """Workload key of a traffic record: the workload name plus the key
    format (bits, codebook initial, q when the QJL plane is kept)."""
    return f"{w.name}:k{w.k_bits}{w.k_codebook[0]}{'q' if w.k_qjl else ''}"


def job_value(world_size, units_per_rank, ms):
    """Whole-job throughput of world_size replicas that each process
    units_per_rank units in ms milliseconds (weak scaling)."""
    return world_size * units_per_rank / (ms * 1e-3)


# ------------------------------------------------------------ CPU baseline
def host_cores():
    """Cores this process may run on (its CPU affinity set)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_sequence_worker(task):
    """One oracle run (numpy fp64, one thread): sequence b of the workload, its
    first `cap` compressed tokens and its exact tail, all heads; repeats the
    step -- the oracle's store of the step's new token, then its decode
    attention -- for `seconds` or `max_steps` steps.  Runs in a spawned worker
    process (or inline); returns tokens attended, steps and seconds."""
    name, b, cap, seconds, max_steps = task
    import numpy as np

    from oracle import paged
    from turboquant_bit_kv_tq_gb300 import workloads as wl

    w = wl.config(name)
    P = paged.CacheParams(w.d, w.k_bits, w.k_qjl, w.v_mode, w.v_bits, w.seed_rot, w.seed_qjl, w.k_codebook,
                          w.v_codebook)
    b = b % w.batch
    n = min(w.compressed_lens()[b], cap)
    nb = max(1, (n + 15) // 16)
    cache = np.zeros((nb, w.kv_heads, P.layout.page_bytes), np.uint8)
    K, V = wl.kv_tokens(w, b, 0, n)
    t = np.arange(n)
    if n > 1:
        paged.store(cache, P, K[:-1], V[:-1], t[:-1])
    Q = wl.queries(w)[b:b + 1].astype(np.float64)
    tail = w.tail_lens()[b] if w.tail else 0
    kw = {}
    if tail:
        tk, tv = wl.kv_tokens(w, b, w.compressed_lens()[b], tail)
        kw = dict(tail_k=tk.transpose(1, 0, 2)[None], tail_v=tv.transpose(1, 0, 2)[None], tail_lens=[tail])
    steps, t0 = 0, time.perf_counter()
    while True:
        if n:
            paged.store(cache, P, K[-1:], V[-1:], t[-1:])  # the step's new token
        paged.decode_attention(cache, P, Q, np.arange(nb)[None], [n], **kw)
        steps += 1
        el = time.perf_counter() - t0
        if el >= seconds or steps >= max_steps:
            break
    return dict(tokens=(n + tail) * steps, steps=steps, seconds=el, seq_tokens=n + tail)


_CPU_SNIPPET = r"""
import json, multiprocessing as mp, os, sys
sys.path.insert(0, {root!r})
import bench
cores = {cores}
tasks = [({name!r}, i, {cap}, {seconds}, {max_steps}) for i in range(cores)]
if cores == 1:
    res = [bench._oracle_sequence_worker(tasks[0])]
else:
    with mp.get_context("spawn").Pool(cores) as pool:
        res = pool.map(bench._oracle_sequence_worker, tasks)
el = max(r["seconds"] for r in res)
print(json.dumps(dict(tokens=sum(r["tokens"] for r in res), seconds=el, steps=min(r["steps"] for r in res),
                      seq_tokens=res[0]["seq_tokens"], workers=len(res))))
"""


def cpu_oracle_run(name, seconds, max_steps=10**6, cap=8192, cores=1):
    """Time the oracle on the host, in a spawned process (so that no worker is
    forked from a process holding a CUDA context): `cores` single-threaded
    workers at once, worker i on sequence i of the workload (its first `cap`
    compressed tokens + tail, all heads).  value = tokens attended by all
    workers / the slowest worker's time."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = _CPU_SNIPPET.format(root=ROOT, name=name, cap=cap, seconds=seconds, max_steps=max_steps, cores=cores)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    res = json.loads(r.stdout.strip().splitlines()[-1])
    res["value"] = res["tokens"] / res["seconds"]
    res["cores"] = res["workers"]
    seqs = "sequence 0" if cores == 1 else f"sequences 0..{cores - 1} (mod the batch), one per worker process"
    res["sample"] = (f"oracle (numpy fp64, {cores} single-threaded process{'es' if cores > 1 else ''}) on {seqs} "
                     f"of {name}: first {res['seq_tokens']} tokens (compressed + tail), all {wl_heads(name)} query "
                     f"heads, store of the step's new token + decode, {res['steps']}+ steps each in "
                     f"{res['seconds']:.1f} s")
    return res


def wl_heads(name):
    from turboquant_bit_kv_tq_gb300 import workloads as wl

    return wl.config(name).q_heads


def cpu_baseline(name, seconds):
    """The oracle's throughput on the host: all cores (the reported value) and
    one thread; cores = the worker processes used, host_cores = the affinity
    set's size."""
    cores = host_cores()
    allc = cpu_oracle_run(name, seconds, cores=cores)
    one = cpu_oracle_run(name, seconds) if cores > 1 else allc
    return {"value": allc["value"], "unit": UNIT, "cores": allc["cores"], "kind": "oracle", "sample": allc["sample"],
            "host_cores": cores, "single_thread": {"value": one["value"], "cores": 1, "sample": one["sample"]}}


def boundary_cases(torch, pages, K, V, slots, w, count=1024):
    """Re-encode `count` random tokens of a store the GPU made with the oracle
    and compare the bytes (after the timed region; tests/parity.py's bar):
    the counted boundary cases of each class beside the count the density
    predicts, and the bytes that differed."""
    import numpy as np

    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import parity
    from oracle import paged

    P = paged.CacheParams(w.d, w.k_bits, w.k_qjl, w.v_mode, w.v_bits, w.seed_rot, w.seed_qjl, w.k_codebook,
                          w.v_codebook)
    rng = np.random.default_rng(0)
    pick = np.sort(rng.choice(len(slots), min(count, len(slots)), replace=False))
    blocks = np.unique(slots[pick] // 16)
    sub = pages[torch.from_numpy(blocks).to(pages.device)].cpu().numpy()
    remap = {int(b): i for i, b in enumerate(blocks)}
    sub_slots = np.array([remap[int(s) // 16] * 16 + int(s) % 16 for s in slots[pick]], np.int64)
    Kh = K[torch.from_numpy(pick).to(K.device)].float().cpu().numpy()
    Vh = V[torch.from_numpy(pick).to(V.device)].float().cpu().numpy()
    r = parity.compare_store(sub, P, Kh, Vh, sub_slots, w.kv_heads)
    return {"workload": w.name, "tokens": int(len(pick)), "vectors": r["vectors"], "checked_bytes": r["checked_bytes"],
            "mismatched_bytes": r["mismatched_bytes"], "unexplained_bytes": len(r["unexplained"]),
            "counted": r["counts"], "expected_from_density": {k: round(v, 3) for k, v in r["expected"].items()},
            "bar": "codes within 1e-6 of a boundary, |S r|/||k|| < 1e-6, fp16 values within 1e-6 of a "
                   "midpoint, group-32 half-integers: counted and excused; every other byte bit-exact"}


# ---------------------------------------------------------- reference arm
def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    from turboquant_bit_kv_tq_gb300 import workloads as wl

    w = wl.config(args.workload)
    cores = host_cores()
    per_step = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    cpu_oracle_run(args.workload, per_step, max_steps=max(1, args.warmup), cores=cores)  # warm-up steps
    res = cpu_oracle_run(args.workload, per_step * args.steps, max_steps=args.steps, cores=cores)
    ms = 1e3 * res["seconds"] / res["steps"]
    line = {
        "impl": "reference", "metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": args.gpus,
        "steps": res["steps"], "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample": res["sample"]},
        "cpu_baseline": {"value": res["value"], "unit": UNIT, "cores": res["cores"], "kind": "oracle",
                         "sample": res["sample"], "host_cores": cores},
        "e2e": {"value": res["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- our arm
def _split_blocks(w, override=0):
    """Blocks per decode split: longer splits for long contexts; a short one
    (a few work items in all) needs short splits to spread over the SMs.  Each
    CTA takes a contiguous run of equal numbers of splits, so the choice sets
    the balance: measured on the 8B-shaped decode (16 x 8192 tokens), 80-block
    splits (three per CTA) took the split kernel 72.3 us against 74.2 at 32
    and 80.7 at 56; on the d=256 and 70B-shaped decodes 64 was best or within
    noise of the best."""
    longest = max(w.seq_lens)
    return override or (64 if longest > 16384 else 80 if longest > 4096 else 32 if longest > 2048 else 8)


def _setup_decode(w, split_blocks, torch, tq, wl, device):
    import numpy as np

    table, num_blocks = wl.block_table(w)
    comp = w.compressed_lens()
    kw = wl.cache_config_kwargs(w, num_blocks=num_blocks, max_blocks=table.shape[1], split_blocks=split_blocks)
    c = tq.TQCache(device=device, **kw)
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    for b in range(w.batch):
        for s0 in range(0, comp[b], 65536):
            n = min(65536, comp[b] - s0)
            t = np.arange(s0, s0 + n)
            slots = torch.from_numpy(table[b, t // 16].astype(np.int64) * 16 + t % 16).to(device)
            K, V = wl.kv_tokens_device(w, n, gen, device)
            c.store(K, V, slots)
    torch.cuda.synchronize()
    if c.device_error():
        raise RuntimeError("device error while filling the cache")
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    st = dict(
        q=torch.from_numpy(wl.queries(w)).to(device, dt),
        table=torch.from_numpy(table).to(device),
        lens=torch.tensor(comp, dtype=torch.int32, device=device),
        out=torch.empty((w.batch, w.q_heads, w.d), dtype=torch.bfloat16, device=device),
    )
    # the step's new token per sequence overwrites the newest compressed slot,
    # so the context length stays fixed from step to step
    last = [max(0, n - 1) for n in comp]
    st["new_slots"] = torch.tensor([int(table[b, p // 16]) * 16 + p % 16 if comp[b] else -1
                                    for b, p in enumerate(last)], dtype=torch.int64, device=device)
    K, V = wl.kv_tokens_device(w, w.batch, gen, device)
    st["new_k"], st["new_v"] = K, V
    if w.tail:
        # the newest tokens of each sequence, exact bf16, from the workload's
        # own generator (positions compressed_len .. seq_len - 1)
        tl = w.tail_lens()
        tk = np.zeros((w.batch, w.kv_heads, w.tail, w.d), np.float32)
        tv = np.zeros_like(tk)
        for b in range(w.batch):
            kb, vb = wl.kv_tokens(w, b, comp[b], tl[b])
            tk[b, :, :tl[b]] = kb.transpose(1, 0, 2)
            tv[b, :, :tl[b]] = vb.transpose(1, 0, 2)
        st["tail_k"] = torch.from_numpy(tk).to(device, torch.bfloat16)
        st["tail_v"] = torch.from_numpy(tv).to(device, torch.bfloat16)
        st["tail_lens"] = torch.tensor(tl, dtype=torch.int32, device=device)
    return c, st, table


def _step(c, st, stream):
    c.store_decode(st["new_k"], st["new_v"], st["new_slots"], st["q"], st["table"], st["lens"], out=st["out"],
                   tail_k=st.get("tail_k"), tail_v=st.get("tail_v"), tail_lens=st.get("tail_lens"), stream=stream)


def _events(torch, n, stream):
    """n timing-event pairs, each recorded once so that its CUDA handle exists
    before the library is given it."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in ev:
        a.record(stream)
        b.record(stream)
    return ev


def _time_steps(torch, tq, c, st, stream, steps, flush, split_events=True):
    """Per-step CUDA events on `stream`, L2 flushed between steps (outside the
    events).  Returns (step_ms list, split_ms list)."""
    ev = _events(torch, steps, stream)
    sev = _events(torch, steps, stream)
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.zero_()
            if split_events:
                tq.tq_set_profile_events(c.handle, tq.TQ_PROF_DECODE_SPLIT, sev[i][0], sev[i][1])
            ev[i][0].record(stream)
            _step(c, st, stream)
            ev[i][1].record(stream)
    tq.tq_set_profile_events(c.handle, tq.TQ_PROF_DECODE_SPLIT, None, None)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    split_ms = [a.elapsed_time(b) for a, b in sev] if split_events else []
    return step_ms, split_ms


def _e2e(torch, c, st, w, stream, steps, warmup, flush):
    """Same step through the public API with host buffers: pinned host inputs
    copied in (one transfer), result copied out, inside the timed region."""
    names = ["q", "new_k", "new_v", "new_slots", "lens", "table"] + (["tail_lens"] if w.tail else [])
    # the step's inputs staged back to back (256-byte aligned) in one pinned
    # host buffer and copied in with one transfer per step; the library is
    # called on views of the device copy
    segs, off = [], 0
    for k in names:
        nb = st[k].numel() * st[k].element_size()
        segs.append((k, off, nb))
        off = (off + nb + 255) // 256 * 256
    host_buf = torch.empty(off, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(off, dtype=torch.uint8, device=st["q"].device)
    for k, o, nb in segs:
        host_buf[o:o + nb].copy_(st[k].contiguous().cpu().reshape(-1).view(torch.uint8))
    dev = {k: dev_buf[o:o + nb].view(st[k].dtype).view(st[k].shape) for k, o, nb in segs}
    out_h = torch.empty(st["out"].shape, dtype=st["out"].dtype).pin_memory()
    h2d = off
    d2h = out_h.numel() * out_h.element_size()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    st2 = dict(st)
    st2.update(dev)
    with torch.cuda.stream(stream):
        for i in range(warmup + steps):
            flush.zero_()
            if i >= warmup:
                ev[i - warmup][0].record(stream)
            dev_buf.copy_(host_buf, non_blocking=True)
            _step(c, st2, stream)
            out_h.copy_(st2["out"], non_blocking=True)
            if i >= warmup:
                ev[i - warmup][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    return ms, h2d, d2h


def _ws_path(w):
    """Whether the decode runs the warp-specialized split kernel: every
    configuration whose score planes fit its tensor-memory plan (d=128 with 2-
    or 3-bit keys or any uniform-codebook keys, d=256 with 2-bit keys); the
    one-warpgroup split kernel the rest.  With the warp-specialized kernel an
    exact tail runs as its own kernel before it."""
    return (w.d == 128 and (w.k_bits <= 3 or w.k_codebook == "uniform")) or (w.d == 256 and w.k_bits == 2)


def _split_roofline(w, page_bytes, split_ms, peak, peak_kind):
    """Roofline of the split-KV kernel: ALGORITHMIC bytes per launch (the
    compressed page bytes of every attended token-head plus the block-table
    entries; the exact tail K/V too when the split kernel reads it itself)
    over its average event-timed duration."""
    per_token_head = page_bytes // 16
    token_heads = sum(w.compressed_lens()) * w.kv_heads
    blocks = sum((n + 15) // 16 for n in w.compressed_lens())
    tail_bytes = sum(w.tail_lens()) * w.kv_heads * w.d * 2 * 2
    ws = _ws_path(w)
    split_bytes = token_heads * per_token_head + blocks * 4 + (0 if ws else tail_bytes)
    avg = statistics.mean(split_ms)
    achieved = split_bytes / (avg * 1e-3) / 1e9
    kernel = "tq::split_ws_kernel" if ws else "tq::split_kernel"
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": _ncu_traffic(kernel, traffic_key(w)), "kernel": kernel, "peak_kind": peak_kind,
            "algorithmic_bytes_per_launch": split_bytes, "bytes_per_token_head": per_token_head,
            "units_per_launch": token_heads, "unit_of_work": "token-head", "avg_launch_ms": avg,
            "launches": len(split_ms)}


def _decode_workload(torch, tq, wl, w, device, steps, warmup, flush, peak, peak_kind, split_blocks=0):
    """One decode workload beside the headline: the same step (store of each
    sequence's new token + decode), timed with L2 flushed between steps and
    without profiling events; its split kernel's roofline from as many steps
    again with CUDA events around the split launch."""
    sb = _split_blocks(w, split_blocks)
    c, st, _ = _setup_decode(w, sb, torch, tq, wl, device)
    stream = torch.cuda.Stream(device=device)
    _time_steps(torch, tq, c, st, stream, warmup, flush, split_events=False)
    step_ms = _time_steps(torch, tq, c, st, stream, steps, flush, split_events=False)[0]
    ev_ms, split_ms = _time_steps(torch, tq, c, st, stream, steps, flush)
    if c.device_error():
        raise RuntimeError(f"device error during the {w.name} steps")
    attended = sum(w.compressed_lens()) + sum(w.tail_lens())
    ms = statistics.mean(step_ms)
    line = {"workload": w.name, "value": attended / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms,
            "kv_tokens_per_step": attended, "compressed_tokens": sum(w.compressed_lens()),
            "tail_tokens": sum(w.tail_lens()), "batch": w.batch, "q_heads": w.q_heads, "kv_heads": w.kv_heads,
            "head_dim": w.d, "k_bits": w.k_bits, "v_mode": w.v_mode, "v_bits": w.v_bits, "split_blocks": sb,
            "steps": steps, "roofline": _split_roofline(w, c.page_bytes, split_ms, peak, peak_kind),
            "with_profiling_events": {"ms_per_step": statistics.mean(ev_ms),
                                      "value": attended / (statistics.mean(ev_ms) * 1e-3)},
            "gpu_launches_per_step": 4 + (1 if (w.tail and _ws_path(w)) else 0)}
    c.close()
    del c, st
    torch.cuda.empty_cache()
    return line


def _store_workload(torch, tq, wl, device, steps, warmup, flush, peak, with_boundary_cases=True):
    """Store throughput on the 65,536-token scattered append (context line);
    then, outside the timed region, the oracle's re-encoding of a 1,024-token
    sample of what the last timed store wrote."""
    w = wl.config("store_64seq_65536tok")
    lens, prior, table, slots = wl.store_layout(w)
    c = tq.TQCache(device=device, **wl.cache_config_kwargs(w, num_blocks=w.pool_blocks, max_blocks=4, max_batch=1))
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    K, V = wl.kv_tokens_device(w, w.store_tokens, gen, device)
    s = torch.from_numpy(slots).to(device)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        c.store(K, V, s)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        ev[i][0].record(stream)
        c.store(K, V, s)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if c.device_error():
        raise RuntimeError("device error during the store workload")
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    read = K.numel() * 2 * 2 + s.numel() * 8
    written = w.store_tokens * w.kv_heads * c.page_bytes // 16
    gbs = (read + written) / (ms * 1e-3) / 1e9
    line = {"workload": w.name, "tokens_per_s": w.store_tokens / (ms * 1e-3), "ms": ms,
            "achieved_gbs": gbs, "frac_of_peak": gbs / peak, "algorithmic_bytes": read + written,
            "bytes_per_token_head": 2 * w.d * 2 + c.page_bytes // 16 + 8 / w.kv_heads, "launches": steps}
    cases = boundary_cases(torch, c.pages(), K, V, slots, w) if with_boundary_cases else None
    c.close()
    return line, cases


def _extend_workload(torch, tq, wl, device, steps, warmup, flush, prefix=4096, chunk=256, batch=4, split_blocks=128,
                     shape="llama8b_gqa4_b16_8k"):
    """Extend (prefill) attention on the 8B shape (context line; the 70B shape
    with shape="llama70b_gqa8_b4_ragged131k_hybrid"): batch sequences, each
    with `prefix` compressed tokens and `chunk` new exact tokens that attend
    causally among themselves."""
    import numpy as np

    w = wl.scaled(wl.config(shape), batch=batch, seq_lens=[prefix] * batch, tail=0)
    table, num_blocks = wl.block_table(w)
    T = batch * chunk
    c = tq.TQCache(device=device, **{**wl.cache_config_kwargs(w, num_blocks=num_blocks, max_blocks=table.shape[1],
                                                               max_batch=T, split_blocks=split_blocks),
                         "tail_cap": chunk})
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    for b in range(batch):
        t = np.arange(prefix)
        slots = torch.from_numpy(table[b, t // 16].astype(np.int64) * 16 + t % 16).to(device)
        K, V = wl.kv_tokens_device(w, prefix, gen, device)
        c.store(K, V, slots)
    new_k, new_v = wl.kv_tokens_device(w, T, gen, device)
    q = (torch.randn((T, w.q_heads, w.d), generator=gen, device=device)).to(torch.bfloat16)
    tab = torch.from_numpy(table).to(device)
    pl = torch.full((batch,), prefix, dtype=torch.int32, device=device)
    cu = torch.arange(0, T + 1, chunk, dtype=torch.int32, device=device)
    out = torch.empty((T, w.q_heads, w.d), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        c.extend(q, tab, pl, cu, new_k, new_v, out=out)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        ev[i][0].record(stream)
        c.extend(q, tab, pl, cu, new_k, new_v, out=out)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if c.device_error():
        raise RuntimeError("device error during the extend workload")
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    attended = T * prefix + batch * chunk * (chunk + 1) // 2
    tag = "llama8b_gqa4" if shape.startswith("llama8b") else "llama70b_gqa8"
    return {"workload": f"{tag} extend: {batch} seqs x {prefix}-token compressed prefix + {chunk} new tokens",
            "new_tokens_per_s": T / (ms * 1e-3), "attended_kv_tokens_per_s": attended / (ms * 1e-3), "ms": ms,
            "split_blocks": split_blocks, "calls": steps}


def run_ours(args):
    import torch

    import turboquant_bit_kv_tq_gb300 as tq
    from turboquant_bit_kv_tq_gb300 import workloads as wl

    ws, rank, local = _dist()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=device)
    tq.load_library()
    w = wl.config(args.workload)
    if args.no_qjl:
        w = wl.scaled(w, k_qjl=False)
    if args.k_bits:
        w = wl.scaled(w, k_bits=args.k_bits)
    if args.codebook != "lloyd":
        w = wl.scaled(w, k_codebook=args.codebook, v_codebook=args.codebook if w.v_mode == "mse" else "lloyd")
    if args.extend_only:
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        line = _extend_workload(torch, tq, wl, device, max(1, args.steps), max(3, args.warmup), flush)
        if rank == 0:
            print(json.dumps({"extend_workload": line}), flush=True)
        return
    if args.store_only:
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        line, _ = _store_workload(torch, tq, wl, device, max(1, args.steps), max(3, args.warmup), flush,
                                  _peaks()[0], with_boundary_cases=False)
        if rank == 0:
            print(json.dumps({"store_workload": line}), flush=True)
        return
    split_blocks = _split_blocks(w, args.split_blocks)
    c, st, table = _setup_decode(w, split_blocks, torch, tq, wl, device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device=device)
    peak, peak_kind = _peaks()

    # warm-up, then the timed steps (barrier + sync on both sides)
    _time_steps(torch, tq, c, st, stream, max(3, args.warmup), flush, split_events=False)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_clk = time.perf_counter()
        # the headline: the K timed steps as a caller runs them, without
        # profiling events (the library then launches its decode kernels
        # programmatically, each prologue overlapping its predecessor's tail)
        step_ms = _time_steps(torch, tq, c, st, stream, args.steps, flush, split_events=False)[0]
        # the split kernel's own duration for the roofline: the same K steps
        # again with CUDA events around its launch (events between the
        # launches turn the programmatic launches off, so these steps are
        # slower; reported beside the headline)
        ev_step_ms, split_ms = _time_steps(torch, tq, c, st, stream, args.steps, flush)
        # keep the same load running until the sampler has seen enough of it
        # (a short timed region may fall between two samples)
        while time.perf_counter() - t_clk < 0.6:
            _time_steps(torch, tq, c, st, stream, 20, flush, split_events=False)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    if c.device_error():
        raise RuntimeError("device error during the timed steps")
    ms = max_over_ranks(statistics.mean(step_ms), device)

    attended = sum(w.compressed_lens()) + sum(w.tail_lens())
    value = job_value(ws, attended, ms)
    roof = _split_roofline(w, c.page_bytes, split_ms, peak, peak_kind)
    # whole-step algorithmic bytes: the split kernel's bytes + the exact tail
    # + q read + out written + the store's bf16 read and packed write
    per_token_head = c.page_bytes // 16
    tail_bytes = sum(w.tail_lens()) * w.kv_heads * w.d * 2 * 2
    step_bytes = (roof["algorithmic_bytes_per_launch"] + (tail_bytes if _ws_path(w) else 0) +
                  w.batch * w.q_heads * w.d * (2 + 2) + w.batch * w.kv_heads * w.d * 2 * 2 +
                  w.batch * w.kv_heads * per_token_head)
    roof["step_achieved_gbs"] = step_bytes / (ms * 1e-3) / 1e9
    e2e_ms, h2d, d2h = _e2e(torch, c, st, w, stream, args.steps, max(3, args.warmup), flush)
    e2e_ms_max = max_over_ranks(e2e_ms, device)
    ev_ms_max = max_over_ranks(statistics.mean(ev_step_ms), device)
    c.close()
    del c, st
    torch.cuda.empty_cache()

    extra = store_line = cases = extend_line = extend_line8 = None
    if rank == 0 and not args.no_decode_workloads and args.workload == DEFAULT_WORKLOAD:
        extra = [_decode_workload(torch, tq, wl, wl.config(name), device, max(5, min(args.steps, 20)),
                                  max(3, args.warmup), flush, peak, peak_kind) for name in EXTRA_DECODES]
    if not args.no_store_workload and rank == 0:
        store_line, cases = _store_workload(torch, tq, wl, device, max(3, min(args.steps, 20)), 3, flush, peak,
                                            with_boundary_cases=not args.no_boundary_cases)
    if not args.no_extend_workload and rank == 0:
        extend_line = _extend_workload(torch, tq, wl, device, max(3, min(args.steps, 20)), 3, flush)
        extend_line8 = _extend_workload(torch, tq, wl, device, max(3, min(args.steps, 20)), 3, flush,
                                        shape="llama70b_gqa8_b4_ragged131k_hybrid")

    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and ws == 1:
            try:
                cpu = cpu_baseline(args.workload, args.cpu_seconds)
            except Exception as e:  # reported, not fatal
                cpu = {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": f"failed: {e}"[:300]}
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": DTYPE, "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "q_heads": w.q_heads, "kv_heads": w.kv_heads,
                       "head_dim": w.d, "context_lens": sorted(set(w.seq_lens)), "tail": w.tail,
                       "k_bits": w.k_bits, "k_qjl": w.k_qjl, "v_mode": w.v_mode, "v_bits": w.v_bits,
                       "k_codebook": w.k_codebook, "v_codebook": w.v_codebook,
                       "split_blocks": split_blocks, "out_dtype": "bf16",
                       "l2": "flushed: 256 MiB buffer written between timed steps (outside the events)",
                       "clocks": "sampled every 50 ms over the timed steps plus untimed steps of the same "
                                 "load up to 0.6 s",
                       "step": "tq_store_decode_attention: each sequence's new token stored, then the decode",
                       "timing": "value: K steps without profiling events; roofline: the split kernel's "
                                 "CUDA-event durations over K more steps with events around it"},
            "roofline": roof,
            "cpu_baseline": cpu,
            "clocks": clk.summary(),
            "e2e": {"value": job_value(ws, attended, e2e_ms_max), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms_max},
            # the K steps that carried the split kernel's profiling events (the
            # roofline's kernel durations come from them)
            "with_profiling_events": {"ms_per_step": ev_ms_max,
                                      "value": job_value(ws, attended, ev_ms_max),
                                      "unit": UNIT, "steps": len(ev_step_ms)},
            # per step: store, prep, split, combine, and the exact-tail kernel
            # beside the warp-specialized split when the workload has a tail
            "gpu_launches": (4 + (1 if (w.tail and _ws_path(w)) else 0)) * args.steps,
            "decode_workloads": extra,
            "store_workload": store_line,
            "boundary_cases": cases,
            "extend_workload": extend_line,
            "extend_workload_gqa8": extend_line8,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def main():
    args = _args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
