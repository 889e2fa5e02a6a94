"""Paged compressed KV cache: page layout, bit packing, store and decode attention.

[Paged] "Which path vLLM takes": new K/V vectors are quantised, packed and
written into a paged KV cache (fixed-size blocks found through a block table);
decode reads the compressed blocks through the block table, decodes them and
runs attention.  [Hub] step 5 fixes only the packing density: 2-bit codes take
a quarter byte each and 4-bit codes half a byte.

Layout reading (parity unpinned -- the pages fix none of it; chosen so that a
tensor-core decode can turn stored bits into matrix operands with one logic
operation per register):
  * cache = uint8 [num_blocks, num_kv_heads, page_bytes]; a page holds the 16
    tokens of one block for one KV head; token t of a sequence lives in block
    block_table[b][t // 16] at row t % 16 (slot = block * 16 + row).
  * bit c of a d-bit row is bit (c % 8) of byte c // 8 (LSB first).
  * a page is a run of planes, each of 16 token rows:
      K code planes  kb x 16 x (d/8)  bit-sliced: plane p, bit c of row r is
                                      bit p of the key code of coordinate c
      K signs        16 x (d/8)       (keys with QJL) bit c = [(S r)_c >= 0]
      K norm         16 x fp16        n16, little-endian
      K rnorm        16 x fp16        rho16 (keys with QJL)
      V codes  MSE:  vb x 16 x (d/8)  bit-sliced like the keys
              G32:   16 x (d*vb/8)    vb-bit fields, LSB-first: field slot k
                                      holds the code of coordinate tau(k)
      V meta   MSE:  16 x fp16        value norm
              G32:   16 x (d/32) x (fp16 scale, fp16 zero)   (natural groups)
  * tau (group-32 slots): with w = d/8, slot k = w*g + 2*m + e
    (0 <= g < 8, 0 <= m < d/16, e in {0, 1}) holds coordinate
    32*(m // 2) + 4*g + 2*(m % 2) + e.  The 16 slots (w*g + 2m + e) for fixed
    m all lie in group m // 2, and the two slots of a pair are neighbours.
"""

import numpy as np

from . import quant

BLOCK = 16


def group32_slot_coordinates(d):
    """tau: coordinate held by each group-32 field slot (array of length d)."""
    w = d // 8
    k = np.arange(d)
    g, rest = k // w, k % w
    m, e = rest // 2, rest % 2
    return 32 * (m // 2) + 4 * g + 2 * (m % 2) + e


class PageLayout:
    """Byte offsets of the planes of one (block, KV head) page."""

    def __init__(self, d, k_bits, k_qjl, v_mode, v_bits):
        assert v_mode in ("mse", "g32")
        assert v_mode == "mse" or v_bits in (2, 4)
        self.d, self.k_bits, self.k_qjl, self.v_mode, self.v_bits = d, k_bits, bool(k_qjl), v_mode, v_bits
        self.bit_row = d // 8                      # one bit per coordinate
        self.v_code_row = d * v_bits // 8          # group-32 bitstream row
        self.v_meta_row = 2 if v_mode == "mse" else 4 * (d // 32)
        off = 0
        self.k_codes = off
        off += k_bits * BLOCK * self.bit_row
        self.k_signs = off
        off += BLOCK * self.bit_row if self.k_qjl else 0
        self.k_norm = off
        off += BLOCK * 2
        self.k_rnorm = off
        off += BLOCK * 2 if self.k_qjl else 0
        self.v_codes = off
        off += (v_bits * BLOCK * self.bit_row) if v_mode == "mse" else BLOCK * self.v_code_row
        self.v_meta = off
        off += BLOCK * self.v_meta_row
        self.page_bytes = off

    def planes(self):
        """(name, byte offset of row 0, row width) of every plane."""
        out = [(f"k_code{p}", self.k_codes + p * BLOCK * self.bit_row, self.bit_row) for p in range(self.k_bits)]
        if self.k_qjl:
            out.append(("k_signs", self.k_signs, self.bit_row))
        out.append(("k_norm", self.k_norm, 2))
        if self.k_qjl:
            out.append(("k_rnorm", self.k_rnorm, 2))
        if self.v_mode == "mse":
            out += [(f"v_code{p}", self.v_codes + p * BLOCK * self.bit_row, self.bit_row)
                    for p in range(self.v_bits)]
        else:
            out.append(("v_codes", self.v_codes, self.v_code_row))
        out.append(("v_meta", self.v_meta, self.v_meta_row))
        return out


def pack_codes(idx, bits):
    """[N, d] codes -> [N, d*bits/8] bytes, LSB-first bitstream per row."""
    idx = np.asarray(idx, np.int64)
    stream = (idx[..., None] >> np.arange(bits)) & 1
    return np.packbits(stream.reshape(idx.shape[0], idx.shape[1] * bits).astype(np.uint8), axis=1,
                       bitorder="little")


def unpack_codes(rows, d, bits):
    stream = np.unpackbits(np.asarray(rows, np.uint8), axis=1, bitorder="little")[:, : d * bits]
    return (stream.reshape(len(rows), d, bits).astype(np.int64) << np.arange(bits)).sum(axis=2)


def pack_bits(flags):
    """[N, d] booleans -> [N, d/8] bytes, flag c -> bit (c % 8) of byte c // 8."""
    return np.packbits(np.asarray(flags, np.uint8), axis=1, bitorder="little")


def unpack_bits(rows, d):
    return np.unpackbits(np.asarray(rows, np.uint8), axis=1, bitorder="little")[:, :d].astype(bool)


def pack_bit_planes(idx, bits):
    """[N, d] codes -> list of `bits` planes, plane p = pack_bits(bit p of each code)."""
    idx = np.asarray(idx, np.int64)
    return [pack_bits((idx >> p) & 1) for p in range(bits)]


def unpack_bit_planes(planes, d):
    return sum(unpack_bits(pl, d).astype(np.int64) << p for p, pl in enumerate(planes))


def f16_bytes(x):
    """float16 array [N, m] -> little-endian bytes [N, 2m]."""
    x = np.ascontiguousarray(np.asarray(x, "<f2"))
    return x.view(np.uint8).reshape(x.shape[0], 2 * x.shape[1])


def bytes_f16(b):
    return np.ascontiguousarray(b).view("<f2")


class CacheParams:
    """Everything one cache's quantisers need, generated by the oracle itself."""

    def __init__(self, d, k_bits, k_qjl, v_mode, v_bits, seed_rot, seed_qjl, k_codebook="lloyd",
                 v_codebook="lloyd"):
        """k_codebook / v_codebook: "lloyd" (Lloyd-Max, [Hub] step 2) or
        "uniform" (equally spaced centroids, [Roadmap] §4.3)."""
        from . import codebook, prng, rotation

        self.layout = PageLayout(d, k_bits, k_qjl, v_mode, v_bits)
        self.d = d
        self.signs = prng.rotation_signs(d, seed_rot)
        self.R = rotation.rotation_matrix(self.signs)
        self.S = prng.qjl_matrix(d, seed_qjl)
        self.k_centroids, self.k_boundaries = codebook.sphere_codebook_of_kind(d, k_bits, k_codebook)
        if v_mode == "mse":
            self.v_centroids, self.v_boundaries = codebook.sphere_codebook_of_kind(d, v_bits, v_codebook)
        else:
            self.v_centroids = self.v_boundaries = None


def encode(P, K, V):
    """Quantise rows of K and V ([N, d] each) into the page-row byte images.

    Returns (fields, pre) where fields maps a plane name (PageLayout.planes)
    to its [N, row_bytes] uint8 rows and pre holds the fp64 pre-images of every
    decision."""
    L = P.layout
    fields, pre = {}, {}
    n16, idx, pk = quant.mse_quantise(K, P.R, P.k_boundaries)
    for p, plane in enumerate(pack_bit_planes(idx, L.k_bits)):
        fields[f"k_code{p}"] = plane
    fields["k_norm"] = f16_bytes(n16[:, None])
    pre.update(k_n=pk["n"], k_y=pk["y"], k_idx=idx)
    if L.k_qjl:
        rho16, bits, pz = quant.qjl_residual(K, n16, idx, P.R, P.k_centroids, P.S)
        fields["k_signs"] = pack_bits(bits)
        fields["k_rnorm"] = f16_bytes(rho16[:, None])
        pre.update(k_rho=pz["rho"], k_z=pz["z"], k_bits=bits)
    if L.v_mode == "mse":
        vn16, vidx, pv = quant.mse_quantise(V, P.R, P.v_boundaries)
        for p, plane in enumerate(pack_bit_planes(vidx, L.v_bits)):
            fields[f"v_code{p}"] = plane
        fields["v_meta"] = f16_bytes(vn16[:, None])
        pre.update(v_n=pv["n"], v_y=pv["y"], v_idx=vidx)
    else:
        s16, z16, q, pg = quant.group32_quantise(V, L.v_bits)
        tau = group32_slot_coordinates(P.d)
        fields["v_codes"] = pack_codes(q[:, tau], L.v_bits)
        fields["v_meta"] = f16_bytes(np.stack([s16, z16], axis=2).reshape(len(V), 2 * s16.shape[1]))
        pre.update(v_scale=pg["scale"], v_zero=pg["zero"], v_t=pg["t"], v_q=q)
    return fields, pre


def _plane(L, name):
    for n, base, width in L.planes():
        if n == name:
            return base, width
    raise KeyError(name)


def store(cache, P, K, V, slot_mapping):
    """Fused store ([Roadmap] §3.1, [Paged] store kernel): quantise every
    (token, KV head) vector of K and V ([T, H_kv, d]) and write its rows at
    slot_mapping[t] (block = slot // 16, row = slot % 16); slot -1 skips the
    token.  Writes ``cache`` in place; returns the pre-images, flattened over
    (token, head) in the order of the valid tokens."""
    T, H, d = K.shape
    slots = np.asarray(slot_mapping, np.int64)
    keep = np.nonzero(slots >= 0)[0]
    Kf = np.asarray(K, np.float64)[keep].reshape(-1, d)
    Vf = np.asarray(V, np.float64)[keep].reshape(-1, d)
    fields, pre = encode(P, Kf, Vf)
    blk = np.repeat(slots[keep] // BLOCK, H)
    row = np.repeat(slots[keep] % BLOCK, H)
    head = np.tile(np.arange(H), len(keep))
    for name, rows in fields.items():
        base, width = _plane(P.layout, name)
        cols = base + row[:, None] * width + np.arange(width)[None, :]
        cache[blk[:, None], head[:, None], cols] = rows
    return pre


def gather_rows(cache, P, blocks, rows, head, name):
    base, width = _plane(P.layout, name)
    cols = base + rows[:, None] * width + np.arange(width)[None, :]
    return cache[blocks[:, None], head, cols]


def read_tokens(cache, P, block_table_row, length, head):
    """Decode the stored fields of tokens 0..length-1 of one sequence, one KV
    head, through its block table row."""
    L = P.layout
    t = np.arange(length)
    blocks = np.asarray(block_table_row, np.int64)[t // BLOCK]
    rows = t % BLOCK
    g = lambda name: gather_rows(cache, P, blocks, rows, head, name)  # noqa: E731
    out = {
        "k_idx": unpack_bit_planes([g(f"k_code{p}") for p in range(L.k_bits)], P.d),
        "k_n16": bytes_f16(g("k_norm"))[:, 0],
    }
    if L.v_mode == "mse":
        out["v_codes"] = unpack_bit_planes([g(f"v_code{p}") for p in range(L.v_bits)], P.d)
    else:
        slots = unpack_codes(g("v_codes"), P.d, L.v_bits)
        codes = np.zeros_like(slots)
        codes[:, group32_slot_coordinates(P.d)] = slots
        out["v_codes"] = codes
    if L.k_qjl:
        out["k_bits"] = unpack_bits(g("k_signs"), P.d)
        out["k_rho16"] = bytes_f16(g("k_rnorm"))[:, 0]
    meta = bytes_f16(g("v_meta"))
    if L.v_mode == "mse":
        out["v_n16"] = meta[:, 0]
    else:
        sz = meta.reshape(length, P.d // 32, 2)
        out["v_s16"], out["v_z16"] = sz[:, :, 0], sz[:, :, 1]
    return out


def decode_attention(cache, P, Q, block_table, seq_lens, scale=None, tail_k=None, tail_v=None, tail_lens=None):
    """Decode attention over the compressed paged cache ([Paged] decode kernel,
    [Roadmap] §3-4), one query per sequence.

    Q [B, H_q, d]; query head h reads KV head h // (H_q / H_kv) (grouped query
    heads, [Roadmap] §3.2).  For sequence b, tokens 0..seq_lens[b]-1 come from
    the cache; optionally tail_lens[b] newest tokens are kept exact in
    tail_k/tail_v [B, H_kv, cap, d] ([Hub] "vLLM integration", hybrid mode
    keeps the newest tokens in full precision).

      s_t  = scale * estimated <q, k_t>     (compressed, quant.key_scores)
      s_t  = scale * <q, k_t>               (tail)
      p    = softmax(s)
      v_t  = n16 R^T c[idx]  (MSE)  |  q s16 + z16  (group-32)  |  v_t (tail)
      out  = sum_t p_t v_t ;  out = 0 when there is no token at all.

    scale defaults to 1/sqrt(d) (score = Q.K, [Paged] "why not just round").
    Returns fp64 [B, H_q, d]."""
    B, Hq, d = Q.shape
    H = cache.shape[1]
    G = Hq // H
    scale = 1.0 / np.sqrt(d) if scale is None or scale <= 0 else scale
    out = np.zeros((B, Hq, d))
    L = P.layout
    for b in range(B):
        n_tail = 0 if tail_lens is None else int(tail_lens[b])
        for g in range(H):
            f = read_tokens(cache, P, block_table[b], int(seq_lens[b]), g)
            if L.v_mode == "mse":
                v_hat = quant.mse_reconstruct(f["v_n16"], f["v_codes"], P.R, P.v_centroids)
            else:
                v_hat = quant.group32_reconstruct(f["v_s16"], f["v_z16"], f["v_codes"])
            kt = np.asarray(tail_k[b, g, :n_tail], np.float64) if n_tail else np.zeros((0, d))
            vt = np.asarray(tail_v[b, g, :n_tail], np.float64) if n_tail else np.zeros((0, d))
            values = np.concatenate([v_hat, vt])
            if len(values) == 0:
                continue
            for h in range(g * G, (g + 1) * G):
                q = np.asarray(Q[b, h], np.float64)
                s = quant.key_scores(q, f["k_n16"], f["k_idx"], f.get("k_rho16"), f.get("k_bits"),
                                     P.R, P.k_centroids, P.S)
                s = scale * np.concatenate([s, kt @ q])
                p = np.exp(s - s.max())
                p /= p.sum()
                out[b, h] = p @ values
    return out


def extend_attention(cache, P, Q, block_table, prefix_lens, cu_q, chunk_k, chunk_v, scale=None):
    """Extend (prefill) attention over the compressed paged cache ([Roadmap]
    §4.1: SGLang's fused extend kernel reads the compressed pool like the
    decode kernel does).

    Sequence b brings n_b = cu_q[b+1] - cu_q[b] new tokens, rows
    cu_q[b] .. cu_q[b+1]-1 of Q [T, H_q, d] and of the exact new keys and
    values chunk_k / chunk_v [T, H_kv, d].  Its first prefix_lens[b] tokens
    are already in the cache (block table row b).  New token j (0-based within
    its chunk) attends to every prefix token through the compressed scores and
    values, and to new tokens 0..j exactly (causal):

      out[cu_q[b] + j] = decode attention of that query over the prefix, with
                         the new tokens 0..j as exact tail tokens.

    Returns fp64 [T, H_q, d]."""
    T, Hq, d = Q.shape
    out = np.zeros((T, Hq, d))
    for b in range(len(prefix_lens)):
        lo, hi = int(cu_q[b]), int(cu_q[b + 1])
        for j in range(hi - lo):
            t = lo + j
            tk = np.asarray(chunk_k[lo:t + 1], np.float64).transpose(1, 0, 2)[None]
            tv = np.asarray(chunk_v[lo:t + 1], np.float64).transpose(1, 0, 2)[None]
            out[t] = decode_attention(cache, P, Q[t:t + 1], block_table[b:b + 1], [prefix_lens[b]], scale=scale,
                                      tail_k=tk, tail_v=tv, tail_lens=[j + 1])[0]
    return out
