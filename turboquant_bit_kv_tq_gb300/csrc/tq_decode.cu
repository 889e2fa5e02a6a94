// Decode attention entry point: query prep, split-KV partials (compiled per
// head dim and key bits in tq_decode_split_*.cu) and the split combine.

#include <algorithm>

#include "tq_extend_prefix.cuh"

namespace tq {

// The score geometry the warp-specialized split kernel and the extend prefix
// kernel run with: a uniform key codebook expands over its k_bits single-bit
// planes only (every multi-bit Walsh term is zero), so its score contraction
// is shorter; both kernels have instances for that at d = 128.
static DecodeGeom ws_geom(const DecodeGeom& g, const Layout& L, bool k_uniform) {
    DecodeGeom gw = g;
    if (L.d == 128 && k_uniform && gw.npk > L.k_bits) {
        gw.npk = L.k_bits;
        gw.npl = gw.npk + (L.k_qjl ? 1 : 0);
        gw.bimg_bytes = gw.n_cols * gw.npl * L.d;
    }
    return gw;
}

template <int D>
static tq_status launch_dim(DecodeArgs a, cudaStream_t s, void* ev0, void* ev1) {
    if (a.group > kMaxG) return TQ_ERR_UNSUPPORTED;
    // the most virtual heads a prep CTA takes (S^T of d = 256 leaves room for 16)
    constexpr int kPrepV = D == 128 ? kPrepMaxV : kMaxG;
    constexpr size_t kPrepMax = prep_smem_bytes<D>(kPrepV);
    // per-device set-up (the first call on a device does it; before any capture)
    int sms = 0;
    {
        tq_status fs = device_sms(&sms);
        if (fs == TQ_OK) fs = ensure_dynamic_smem((const void*)prep_kernel<D>, (int)kPrepMax, "prep_kernel");
        if (fs != TQ_OK) return fs;
    }
    size_t smem = 0;
    int grid = 0;
    const DecodeGeom gw = ws_geom(a.gm, a.lay, a.k_uniform);
    // extend with a query-block plan: the compressed prefix of every block in
    // one GEMM-shaped pass (extend_prefix_kernel), no split kernel
    const bool xp = D == 128 && a.xblocks != nullptr && xp_supported(gw, D) &&
                    xp_layout(a.lay.page_bytes, gw.bimg_bytes).total <= 227 * 1024;
    if (xp) {
        a.gm = gw;
        // the query prep takes as many entries per CTA as its virtual-head
        // limit allows (S^T staged once for them)
        a.prep_entries = std::max(1, std::min(xp_block_tokens(), kPrepMaxV / a.group));
        a.prep_late_release = true;
    } else if (ws_fits(gw, D)) {
        // persistent warp-specialized split kernel: two CTAs per SM, the
        // deepest ring that fits; the exact tail runs as its own kernel
        const int n_items = a.batch * a.heads * a.gm.nhg * a.sp.n_chunks;
        const int kitems = ws_items_per_cta(n_items, std::min(n_items, kWsCtasPerSm * sms));
        grid = (n_items + kitems - 1) / kitems;  // contiguous runs of kitems items
        const int nsets = a.lay.v_mode == TQ_V_G32 ? D / 32 : (1 << (a.lay.v_bits - 1));
        a.stages = 0;
        for (int st = kWsMaxStages; st >= 2 && a.stages == 0; --st) {
            const WsLayout wl = ws_layout<D>(a.lay.page_bytes, gw, nsets, st, kitems, a.split_blocks);
            if (wl.total <= 112 * 1024) {
                a.stages = st;
                smem = std::max(wl.total, (size_t)77 * 1024);  // never a third CTA per SM (tensor memory)
            }
        }
        if (a.stages == 0) grid = 0;  // too many items per CTA for the staged schedule
        if (grid > 0) a.gm = gw;      // (the other kernels keep every plane)
    }
    if (grid == 0 && !xp) {
        const tq_status cfg = split_config<D>(a, &a.stages, &smem);
        if (cfg != TQ_OK) return cfg;
    }
    if constexpr (D == 128) {
        // extend: the exact causal part of every new token in one pass over
        // the new-token tiles (the tail split of each entry), in stream order
        // before the query prep
        if (a.tail_base != nullptr && a.tail_cap > 0) {
            a.chunk_attn = true;
            const int warps = std::min(a.group, kChunkMaxWarps);
            chunk_attn_kernel<D><<<dim3((a.batch + kChunkRows - 1) / kChunkRows, a.heads), 32 * warps,
                                   chunk_smem_bytes(), s>>>(a);
            const tq_status st = cuda_status(cudaGetLastError());
            if (st != TQ_OK) return st;
            // it began after the queries' writer had finished: the prep may
            // read them beside it
            a.q_early = true;
        }
    }
    {
        // the split (and tail) and combine kernels launch programmatically
        // (each one's prologue overlaps the previous kernel's tail) unless
        // profiling events sit between the launches; the query prep launches
        // programmatically too, but waits for its predecessor before any read
        // (that hides the launch gap; running it beside a preceding store
        // measured slower)
        a.pdl = ev0 == nullptr && ev1 == nullptr;
        if (a.prep_entries < 1 || a.prep_entries * a.group > kPrepV) a.prep_entries = 1;
        const size_t prep_smem = prep_smem_bytes<D>(a.prep_entries * a.group);
        const dim3 pgrid(a.heads, (a.batch + a.prep_entries - 1) / a.prep_entries);
        const cudaError_t e = launch_pdl(true, prep_kernel<D>, pgrid, dim3(kPrepThreads), prep_smem, s, a);
        if (e != cudaSuccess) return cuda_status(e);
    }
    if (grid > 0 && a.tail_cap > 0 && !a.chunk_attn) {
        // one query head per CTA
        const size_t tail_smem = tail_smem_bytes<D>(1);
        const cudaError_t e =
            launch_pdl(a.pdl, tail_kernel<D>, dim3(a.heads, a.batch, a.group), dim3(128), tail_smem, s, a);
        if (e != cudaSuccess) return cuda_status(e);
    }
    if (ev0) cudaEventRecord((cudaEvent_t)ev0, s);
    tq_status st;
    if (xp) {
        // enough CTAs (one per SM at least) that none takes more than
        // kXpMaxItems items
        const int64_t ub = (int64_t)a.xblocks_max * a.heads * a.gm.nhg * a.sp.n_chunks;
        const int64_t xg = std::min<int64_t>(ub, std::max<int64_t>(sms, (ub + kXpMaxItems - 1) / kXpMaxItems));
        if (xg <= 0) {
            st = TQ_OK;
        } else {
            const int kb = a.lay.k_bits;
            const bool ku = a.gm.npk == kb && kb >= 3;
            st = kb == 2 ? dispatch_extend_prefix<2, false>(a, s, (int)xg)
               : kb == 3 ? (ku ? dispatch_extend_prefix<3, true>(a, s, (int)xg)
                               : dispatch_extend_prefix<3, false>(a, s, (int)xg))
                         : dispatch_extend_prefix<4, true>(a, s, (int)xg);
        }
    } else {
        switch (a.lay.k_bits) {
            case 2: st = dispatch_split<D, 2>(a, s, smem, grid); break;
            case 3: st = dispatch_split<D, 3>(a, s, smem, grid); break;
            default: st = dispatch_split<D, 4>(a, s, smem, grid); break;
        }
    }
    if (st != TQ_OK) return st;
    if (ev1) cudaEventRecord((cudaEvent_t)ev1, s);
    return cuda_status(launch_pdl(a.pdl, a.sp.n_splits <= 8 ? combine_kernel<D, 8> : combine_kernel<D, 32>,
                                  dim3(a.q_heads, a.batch), dim3(128), (size_t)a.sp.n_splits * sizeof(float), s, a));
}

tq_status launch_decode(const DecodeArgs& a, cudaStream_t s, void* ev0, void* ev1) {
    return a.lay.d == 128 ? launch_dim<128>(a, s, ev0, ev1) : launch_dim<256>(a, s, ev0, ev1);
}

}  // namespace tq

using namespace tq;

namespace tq {

tq_status decode_args(const tq_cache* c, const void* q, int q_dtype, const void* cache_buf,
                      const int32_t* block_table, const int32_t* seq_lens, const void* tail_k, const void* tail_v,
                      const int32_t* tail_lens, float scale, int batch, void* out, int out_dtype, DecodeArgs* a) {
    if (!c || !q || !cache_buf || !block_table || !seq_lens || !out) return TQ_ERR_INVALID_ARG;
    if (batch < 1 || batch > c->cfg.max_batch) return TQ_ERR_INVALID_ARG;
    if (q_dtype != TQ_DTYPE_F32 && q_dtype != TQ_DTYPE_BF16) return TQ_ERR_INVALID_ARG;
    const bool out_rot = (out_dtype & TQ_OUT_ROTATED) != 0;
    out_dtype &= ~TQ_OUT_ROTATED;
    if (out_dtype != TQ_DTYPE_F32 && out_dtype != TQ_DTYPE_BF16) return TQ_ERR_INVALID_ARG;
    if (out_rot && c->cfg.v_mode != TQ_V_MSE) return TQ_ERR_INVALID_ARG;
    const bool has_tail = tail_k != nullptr || tail_v != nullptr || tail_lens != nullptr;
    if (has_tail && (!tail_k || !tail_v || !tail_lens || c->cfg.tail_cap == 0)) return TQ_ERR_INVALID_ARG;
    if (((uintptr_t)tail_k | (uintptr_t)tail_v) & 15) return TQ_ERR_MISALIGNED;
    if ((uintptr_t)cache_buf & 15) return TQ_ERR_MISALIGNED;
    a->q = q;
    a->q_dtype = q_dtype;
    a->cache = static_cast<const uint8_t*>(cache_buf);
    a->block_table = block_table;
    a->seq_lens = seq_lens;
    a->tail_k = static_cast<const uint16_t*>(tail_k);
    a->tail_v = static_cast<const uint16_t*>(tail_v);
    a->tail_lens = tail_lens;
    a->out = out;
    a->out_dtype = out_dtype;
    a->out_rotated = out_rot;
    a->k_uniform = c->cfg.k_codebook == TQ_CODEBOOK_UNIFORM;
    const int d = c->cfg.head_dim;
    const float sc = scale > 0.f ? scale : 1.0f / sqrtf((float)d);
    a->scale_log2e = sc * 1.4426950408889634f;
    a->batch = batch;
    a->num_blocks = c->cfg.num_blocks;
    a->heads = c->cfg.num_kv_heads;
    a->q_heads = c->cfg.num_q_heads;
    a->group = a->q_heads / a->heads;
    a->max_blocks = c->cfg.max_blocks_per_seq;
    a->split_blocks = c->cfg.split_blocks;
    a->tail_cap = has_tail ? c->cfg.tail_cap : 0;
    a->sp = c->splits;
    a->lay = c->lay;
    a->dp = c->dp;
    a->gm = c->geom;
    a->ws_bimg = c->ws_bimg;
    a->ws_cst = c->ws_cst;
    a->ws_acc = c->ws_acc;
    a->ws_ml = c->ws_ml;
    return TQ_OK;
}

}  // namespace tq

extern "C" tq_status tq_decode_attention(const tq_cache* c, const void* q, int q_dtype, const void* cache_buf,
                                         const int32_t* block_table, const int32_t* seq_lens, const void* tail_k,
                                         const void* tail_v, const int32_t* tail_lens, float scale, int batch,
                                         void* out, int out_dtype, void* stream) {
    DecodeArgs a;
    const tq_status st = decode_args(c, q, q_dtype, cache_buf, block_table, seq_lens, tail_k, tail_v, tail_lens,
                                     scale, batch, out, out_dtype, &a);
    if (st != TQ_OK) return st;
    void *e0 = c->prof_start[TQ_PROF_DECODE_SPLIT], *e1 = c->prof_stop[TQ_PROF_DECODE_SPLIT];
    return launch_decode(a, (cudaStream_t)stream, e0, e1);
}

extern "C" tq_status tq_store_decode_attention(const tq_cache* c, const void* k, const void* v, int in_dtype,
                                               int64_t num_tokens, const int64_t* slot_mapping, const void* q,
                                               int q_dtype, void* cache_buf, const int32_t* block_table,
                                               const int32_t* seq_lens, const void* tail_k, const void* tail_v,
                                               const int32_t* tail_lens, float scale, int batch, void* out,
                                               int out_dtype, void* stream) {
    // both calls' arguments are checked before either launches
    DecodeArgs a;
    tq_status st = decode_args(c, q, q_dtype, cache_buf, block_table, seq_lens, tail_k, tail_v, tail_lens, scale,
                               batch, out, out_dtype, &a);
    if (st != TQ_OK) return st;
    if (num_tokens < 0) return TQ_ERR_INVALID_ARG;
    if (num_tokens > 0) {
        if (!k || !v || !slot_mapping) return TQ_ERR_INVALID_ARG;
        if (in_dtype != TQ_DTYPE_F32 && in_dtype != TQ_DTYPE_BF16) return TQ_ERR_INVALID_ARG;
        if (((uintptr_t)k & 3) || ((uintptr_t)v & 3)) return TQ_ERR_MISALIGNED;
        st = tq_store(c, k, v, in_dtype, num_tokens, slot_mapping, cache_buf, stream);
        if (st != TQ_OK) return st;
        // the store kernel, launched in plain stream order, began after the
        // queries' writer had finished: the query prep may read them at once
        a.q_early = true;
    }
    void *e0 = c->prof_start[TQ_PROF_DECODE_SPLIT], *e1 = c->prof_stop[TQ_PROF_DECODE_SPLIT];
    return launch_decode(a, (cudaStream_t)stream, e0, e1);
}

namespace tq {

// One thread waits for phase 0 of a shared-memory mbarrier that expects one
// arrival and gets none, through the decode kernels' bounded wait.
__global__ void wait_timeout_kernel(uint32_t* err, uint32_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_wait_timed(smem_u32(&bar), 0, err, limit_ns);
}

// One thread per new token t: find the sequence whose chunk holds row t (the
// last b with cu_q[b] <= t) and write the token's decode-entry view: compressed
// length = the prefix, block-table row b, exact tail = chunk rows
// cu_q[b] .. t.  A row outside every chunk gets no token at all (output 0)
// and sets TQ_DEVERR_CHUNK; the rows it names always lie in [0, t].
__global__ void extend_entries_kernel(const int32_t* __restrict__ prefix_lens, const int32_t* __restrict__ cu_q,
                                      int batch, int n_tokens, int32_t* seq_len, int32_t* tail_len, int32_t* row_of,
                                      int32_t* tail_base, uint32_t* err) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n_tokens) return;
    int lo = 0, hi = batch - 1, b = -1;
    while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        if (cu_q[mid] <= t) {
            b = mid;
            lo = mid + 1;
        } else {
            hi = mid - 1;
        }
    }
    const int start = b >= 0 ? cu_q[b] : -1;
    if (b < 0 || start < 0 || t >= cu_q[b + 1]) {
        seq_len[t] = tail_len[t] = row_of[t] = tail_base[t] = 0;
        set_error(err, TQ_DEVERR_CHUNK);
        return;
    }
    seq_len[t] = prefix_lens[b];
    tail_len[t] = t - start + 1;
    row_of[t] = b;
    tail_base[t] = start;
}

// One CTA: extend's query blocks for the prefix kernel.  The chunk of
// sequence b (rows cu_q[b] .. cu_q[b+1] - 1), when b has a compressed prefix,
// splits into blocks of up to tpb consecutive new tokens; blocks[k] = {first
// row, rows, b, index of the block's first prefix work item}, a block having
// hn x (the prefix's non-empty splits) items.  counts = {blocks, items}.  A
// cu_q that decreases or leaves [0, n_tokens] sets TQ_DEVERR_CHUNK and its
// chunks are clamped; if the blocks would then exceed the capacity cap, the
// plan is left empty (no prefix work) with the same error.
__global__ void __launch_bounds__(1024) extend_blocks_kernel(const int32_t* __restrict__ prefix_lens,
                                                             const int32_t* __restrict__ cu_q, int batch,
                                                             int n_tokens, int tpb, int hn, int split_tokens,
                                                             int max_len, int cap, int4* blocks, int32_t* counts,
                                                             uint32_t* err) {
    __shared__ int wsum[2][32];
    __shared__ int carry[2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    if (tid == 0) carry[0] = carry[1] = 0;
    __syncthreads();
    for (int base = 0; base < batch; base += blockDim.x) {
        const int b = base + tid;
        int lo = 0, chunk = 0, ns = 0, nb = 0, ni = 0;
        if (b < batch) {
            int l0 = cu_q[b], l1 = cu_q[b + 1];
            if (l0 < 0 || l1 < l0 || l1 > n_tokens) {
                set_error(err, TQ_DEVERR_CHUNK);
                l0 = min(max(l0, 0), n_tokens);
                l1 = min(max(l1, l0), n_tokens);
            }
            lo = l0;
            chunk = l1 - l0;
            const int len = min(max(prefix_lens[b], 0), max_len);
            ns = (len + split_tokens - 1) / split_tokens;
            nb = ns > 0 ? (chunk + tpb - 1) / tpb : 0;
            ni = nb * hn * ns;
        }
        // block-wide inclusive scans of the block and item counts
        int sb = nb, si = ni;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int xb = __shfl_up_sync(0xffffffffu, sb, o), xi = __shfl_up_sync(0xffffffffu, si, o);
            if (lane >= o) {
                sb += xb;
                si += xi;
            }
        }
        if (lane == 31) {
            wsum[0][warp] = sb;
            wsum[1][warp] = si;
        }
        __syncthreads();
        if (warp == 0) {
            int vb = lane < nw ? wsum[0][lane] : 0, vi = lane < nw ? wsum[1][lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int xb = __shfl_up_sync(0xffffffffu, vb, o), xi = __shfl_up_sync(0xffffffffu, vi, o);
                if (lane >= o) {
                    vb += xb;
                    vi += xi;
                }
            }
            wsum[0][lane] = vb;
            wsum[1][lane] = vi;
        }
        __syncthreads();
        const int bb = carry[0] + (warp ? wsum[0][warp - 1] : 0) + sb - nb;
        const int ib = carry[1] + (warp ? wsum[1][warp - 1] : 0) + si - ni;
        for (int j = 0; j < nb; ++j)
            if (bb + j < cap) blocks[bb + j] = make_int4(lo + tpb * j, min(tpb, chunk - tpb * j), b, ib + j * hn * ns);
        __syncthreads();
        if (tid == 0) {
            carry[0] += wsum[0][nw - 1];
            carry[1] += wsum[1][nw - 1];
        }
        __syncthreads();
    }
    if (tid == 0) {
        const bool over = carry[0] > cap;
        if (over) set_error(err, TQ_DEVERR_CHUNK);
        counts[0] = over ? 0 : carry[0];
        counts[1] = over ? 0 : carry[1];
    }
}

}  // namespace tq

extern "C" tq_status tq_extend_attention(const tq_cache* c, const void* q, int q_dtype, const void* cache_buf,
                                         const int32_t* block_table, const int32_t* prefix_lens, const int32_t* cu_q,
                                         const void* new_k, const void* new_v, float scale, int batch, int n_tokens,
                                         void* out, int out_dtype, void* stream) {
    if (!c || !q || !cache_buf || !block_table || !prefix_lens || !cu_q || !new_k || !new_v || !out)
        return TQ_ERR_INVALID_ARG;
    if (batch < 1 || n_tokens < 0 || n_tokens > c->cfg.max_batch || c->cfg.tail_cap < 1) return TQ_ERR_INVALID_ARG;
    if (q_dtype != TQ_DTYPE_F32 && q_dtype != TQ_DTYPE_BF16) return TQ_ERR_INVALID_ARG;
    const bool out_rot = (out_dtype & TQ_OUT_ROTATED) != 0;
    out_dtype &= ~TQ_OUT_ROTATED;
    if (out_dtype != TQ_DTYPE_F32 && out_dtype != TQ_DTYPE_BF16) return TQ_ERR_INVALID_ARG;
    if (out_rot && c->cfg.v_mode != TQ_V_MSE) return TQ_ERR_INVALID_ARG;
    if (((uintptr_t)cache_buf | (uintptr_t)new_k | (uintptr_t)new_v) & 15) return TQ_ERR_MISALIGNED;
    if (n_tokens == 0) return TQ_OK;
    cudaStream_t s = (cudaStream_t)stream;
    const int B = c->cfg.max_batch;
    int32_t* seq_len = c->ws_ext;
    int32_t* tail_len = seq_len + B;
    int32_t* row_of = tail_len + B;
    int32_t* tail_base = row_of + B;
    extend_entries_kernel<<<(n_tokens + 255) / 256, 256, 0, s>>>(prefix_lens, cu_q, batch, n_tokens, seq_len,
                                                                 tail_len, row_of, tail_base, c->dp.err);
    {
        const tq_status st = cuda_status(cudaGetLastError());
        if (st != TQ_OK) return st;
    }
    DecodeArgs a;
    a.q = q;
    a.q_dtype = q_dtype;
    a.cache = static_cast<const uint8_t*>(cache_buf);
    a.block_table = block_table;
    a.seq_lens = seq_len;
    a.tail_k = static_cast<const uint16_t*>(new_k);
    a.tail_v = static_cast<const uint16_t*>(new_v);
    a.tail_lens = tail_len;
    a.row_of = row_of;
    a.tail_base = tail_base;
    a.out = out;
    a.out_dtype = out_dtype;
    a.out_rotated = out_rot;
    a.k_uniform = c->cfg.k_codebook == TQ_CODEBOOK_UNIFORM;
    const int d = c->cfg.head_dim;
    const float sc = scale > 0.f ? scale : 1.0f / sqrtf((float)d);
    a.scale_log2e = sc * 1.4426950408889634f;
    a.batch = n_tokens;
    a.num_blocks = c->cfg.num_blocks;
    a.heads = c->cfg.num_kv_heads;
    a.q_heads = c->cfg.num_q_heads;
    a.group = a.q_heads / a.heads;
    a.max_blocks = c->cfg.max_blocks_per_seq;
    a.split_blocks = c->cfg.split_blocks;
    a.tail_cap = c->cfg.tail_cap;
    a.sp = c->splits;
    a.lay = c->lay;
    a.dp = c->dp;
    a.gm = c->geom;
    a.ws_bimg = c->ws_bimg;
    a.ws_cst = c->ws_cst;
    a.ws_acc = c->ws_acc;
    a.ws_ml = c->ws_ml;
    // d = 128 with full head groups: the query-block plan of the prefix
    // kernel (launch_decode runs it when the score planes fit)
    const DecodeGeom gw = ws_geom(a.gm, a.lay, a.k_uniform);
    if (xp_supported(gw, d)) {
        const int tpb = xp_block_tokens();
        a.xcounts = tail_base + B;
        a.xblocks = reinterpret_cast<const int4*>(tail_base + B + 4);
        a.xblocks_max = std::min(n_tokens, (n_tokens + tpb - 1) / tpb + batch);
        extend_blocks_kernel<<<1, 1024, 0, s>>>(prefix_lens, cu_q, batch, n_tokens, tpb, a.heads * gw.nhg,
                                                a.split_blocks * kBlock, a.max_blocks * kBlock, B,
                                                const_cast<int4*>(a.xblocks), const_cast<int32_t*>(a.xcounts),
                                                c->dp.err);
        const tq_status st = cuda_status(cudaGetLastError());
        if (st != TQ_OK) return st;
    }
    return launch_decode(a, s, c->prof_start[TQ_PROF_DECODE_SPLIT], c->prof_stop[TQ_PROF_DECODE_SPLIT]);
}

extern "C" tq_status tq_check_wait_timeout(uint32_t* err_word, uint32_t limit_us, void* stream) {
    if (!err_word || limit_us == 0 || limit_us > 4000000u) return TQ_ERR_INVALID_ARG;
    if ((uintptr_t)err_word & 3) return TQ_ERR_MISALIGNED;
    wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err_word, limit_us * 1000u);
    return cuda_status(cudaGetLastError());
}
