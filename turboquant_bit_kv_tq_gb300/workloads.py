"""Seeded synthetic inputs shaped like the pages' workloads.

Random draws, outlier channels, block tables, slot maps and sequence lengths
only -- none of TurboQuant's arithmetic lives here.  Both the CUDA path (tests,
bench) and the CPU oracle (tests) take their inputs from these functions.

Recipe (every draw from numpy's PCG64 seeded by a tuple of integers):
  * Q, K, V ~ N(0, 1); within KV head g a fixed set of outlier channels
    (a seeded permutation's first n_outlier entries) is multiplied by
    outlier_scale in K and V of head g and in Q of every query head of group g.
  * K/V of sequence b are drawn in segments of 1024 positions, each segment
    seeded by (seed, 1, b, segment), so any token range is reproducible alone.
  * bf16 workloads round the fp32 draws to bf16 (round-to-nearest-even).
  * block tables map each sequence's logical blocks to a seeded random
    permutation of the pool (identity for the single-sequence case).
"""

from dataclasses import dataclass, field

import numpy as np

SEGMENT = 1024
BLOCK = 16


@dataclass
class Workload:
    name: str
    d: int
    q_heads: int
    kv_heads: int
    k_bits: int
    v_mode: str  # "mse" | "g32"
    v_bits: int
    dtype: str  # "f32" | "bf16"
    n_outlier: int
    outlier_scale: float
    seed: int
    seed_rot: int = 2
    seed_qjl: int = 1
    k_qjl: bool = True
    k_codebook: str = "lloyd"  # "lloyd" | "uniform"
    v_codebook: str = "lloyd"
    # decode shape
    batch: int = 0
    seq_lens: list = field(default_factory=list)  # total tokens per sequence (compressed + tail)
    tail: int = 0  # newest tokens kept exact (bf16)
    identity_table: bool = False
    # store shape
    store_tokens: int = 0
    store_seqs: int = 0
    pool_blocks: int = 0

    @property
    def group(self):
        return self.q_heads // self.kv_heads

    def compressed_lens(self):
        return [max(0, n - self.tail) for n in self.seq_lens]

    def tail_lens(self):
        return [min(self.tail, n) for n in self.seq_lens]


def _lens_c4():
    rng = np.random.default_rng(7)
    return [int(x) for x in rng.integers(1024, 131072, size=4, endpoint=True)]


def config(name):
    """The five workloads: single-head check, Llama-3.1-8B-shaped decode,
    d=256 GQA decode, 70B-shaped long-context hybrid decode, store throughput."""
    if name == "single_head_d128_1k":
        return Workload(name, 128, 1, 1, 2, "mse", 2, "f32", 4, 20.0, seed=0, batch=1, seq_lens=[1024],
                        identity_table=True)
    if name == "llama8b_gqa4_b16_8k":
        return Workload(name, 128, 32, 8, 3, "g32", 4, "bf16", 3, 10.0, seed=1, batch=16, seq_lens=[8192] * 16)
    if name == "d256_gqa8_b8_32k":
        return Workload(name, 256, 32, 4, 2, "mse", 2, "bf16", 5, 15.0, seed=2, batch=8, seq_lens=[32768] * 8)
    if name == "llama70b_gqa8_b4_ragged131k_hybrid":
        return Workload(name, 128, 64, 8, 3, "g32", 4, "bf16", 3, 10.0, seed=3, batch=4, seq_lens=_lens_c4(),
                        tail=128)
    if name == "store_64seq_65536tok":
        return Workload(name, 128, 8, 8, 3, "mse", 2, "bf16", 3, 10.0, seed=4, store_tokens=65536, store_seqs=64,
                        pool_blocks=65536)
    raise KeyError(name)


NAMES = ["single_head_d128_1k", "llama8b_gqa4_b16_8k", "d256_gqa8_b8_32k", "llama70b_gqa8_b4_ragged131k_hybrid",
         "store_64seq_65536tok"]


def scaled(w, **changes):
    """A copy of workload ``w`` with some fields replaced (smaller test sizes)."""
    import dataclasses

    return dataclasses.replace(w, **changes)


def round_bf16(x):
    """fp32 array -> the bf16 values it rounds to (round-to-nearest-even), fp32."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    u = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return u.view(np.float32)


def _finish(w, x):
    return round_bf16(x) if w.dtype == "bf16" else np.asarray(x, np.float32)


def outlier_channels(w):
    """[kv_heads, n_outlier] channel indices per KV head."""
    rng = np.random.default_rng((w.seed, 0))
    return np.stack([rng.permutation(w.d)[: w.n_outlier] for _ in range(w.kv_heads)])


def _outlier_gain(w):
    gain = np.ones((w.kv_heads, w.d), np.float32)
    for g, ch in enumerate(outlier_channels(w)):
        gain[g, ch] = w.outlier_scale
    return gain


def kv_tokens(w, b, start, count, heads=None):
    """K, V float32 [count, len(heads), d] of sequence b, positions
    [start, start+count), KV heads `heads` (default all)."""
    heads = np.arange(w.kv_heads) if heads is None else np.atleast_1d(heads)
    gain = _outlier_gain(w)[heads]
    ks, vs = [], []
    first, last = start // SEGMENT, (start + count - 1) // SEGMENT
    for seg in range(first, last + 1 if count > 0 else first):
        rng = np.random.default_rng((w.seed, 1, b, seg))
        kv = rng.standard_normal((2, SEGMENT, w.kv_heads, w.d), dtype=np.float32)
        lo = max(start, seg * SEGMENT) - seg * SEGMENT
        hi = min(start + count, (seg + 1) * SEGMENT) - seg * SEGMENT
        ks.append(kv[0, lo:hi][:, heads])
        vs.append(kv[1, lo:hi][:, heads])
    if not ks:
        z = np.zeros((0, len(heads), w.d), np.float32)
        return z, z
    K = np.concatenate(ks) * gain[None]
    V = np.concatenate(vs) * gain[None]
    return _finish(w, K), _finish(w, V)


def kv_tokens_device(w, count, generator, device="cuda"):
    """The same recipe drawn by torch on the device (bulk cache fills where no
    oracle comparison is made): K, V [count, kv_heads, d] in the workload dtype."""
    import torch

    gain = torch.from_numpy(_outlier_gain(w)).to(device)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    K = torch.randn((count, w.kv_heads, w.d), generator=generator, device=device) * gain
    V = torch.randn((count, w.kv_heads, w.d), generator=generator, device=device) * gain
    return K.to(dt), V.to(dt)


def queries(w, batch=None):
    """Q float32 [batch, q_heads, d]."""
    batch = w.batch if batch is None else batch
    rng = np.random.default_rng((w.seed, 2))
    q = rng.standard_normal((batch, w.q_heads, w.d), dtype=np.float32)
    q *= np.repeat(_outlier_gain(w), w.group, axis=0)[None]
    return _finish(w, q)


def block_table(w):
    """(table int32 [batch, max_blocks], num_blocks): each sequence's compressed
    tokens occupy ceil(len/16) blocks of a shared pool."""
    lens = w.compressed_lens()
    need = [(n + BLOCK - 1) // BLOCK for n in lens]
    max_blocks = max(1, max(need))
    num_blocks = max(1, sum(need))
    perm = np.arange(num_blocks) if w.identity_table else np.random.default_rng((w.seed, 3)).permutation(num_blocks)
    table = np.zeros((w.batch, max_blocks), np.int32)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[at:at + n]
        at += n
    return table, num_blocks


def store_layout(w):
    """Store workload: (chunk lengths, prior lengths, block table, slot_mapping).

    Chunk lengths ~ U[256, 2048] rescaled to sum to store_tokens (largest
    remainder, clamped to [1, 2048]); prior context lengths ~ U[0, 4096) so
    writes start mid-block; each sequence's blocks come from a seeded
    permutation of the pool."""
    rng = np.random.default_rng((w.seed, 4))
    raw = rng.integers(256, 2048, size=w.store_seqs, endpoint=True).astype(np.float64)
    share = raw / raw.sum() * w.store_tokens
    lens = np.floor(share).astype(np.int64)
    rest = w.store_tokens - lens.sum()
    lens[np.argsort(-(share - lens))[:rest]] += 1
    lens = np.clip(lens, 1, 2048)
    lens[-1] += w.store_tokens - lens.sum()
    prior = rng.integers(0, 4096, size=w.store_seqs)
    need = (prior + lens + BLOCK - 1) // BLOCK
    perm = rng.permutation(w.pool_blocks)
    assert need.sum() <= w.pool_blocks
    table = np.zeros((w.store_seqs, int(need.max())), np.int64)
    at = 0
    slots = []
    for s in range(w.store_seqs):
        table[s, : need[s]] = perm[at:at + need[s]]
        at += need[s]
        pos = prior[s] + np.arange(lens[s])
        slots.append(table[s, pos // BLOCK] * BLOCK + pos % BLOCK)
    return lens, prior, table, np.concatenate(slots).astype(np.int64)


def store_tokens(w, start=0, count=None):
    """K, V float32 [count, kv_heads, d] of the store workload's new tokens."""
    count = w.store_tokens - start if count is None else count
    return kv_tokens(w, 0, start, count)


def cache_config_kwargs(w, num_blocks, max_blocks, max_batch=None, split_blocks=32):
    """Keyword arguments for turboquant_bit_kv_tq_gb300.tq_cache_config."""
    return dict(head_dim=w.d, num_kv_heads=w.kv_heads, num_q_heads=w.q_heads, num_blocks=num_blocks,
                k_bits=w.k_bits, k_qjl=int(w.k_qjl), v_mode=0 if w.v_mode == "mse" else 1, v_bits=w.v_bits,
                seed_rot=w.seed_rot, seed_qjl=w.seed_qjl, max_batch=max_batch or max(1, w.batch),
                max_blocks_per_seq=max_blocks, split_blocks=split_blocks, tail_cap=w.tail,
                k_codebook=0 if w.k_codebook == "lloyd" else 1, v_codebook=0 if w.v_codebook == "lloyd" else 1)
