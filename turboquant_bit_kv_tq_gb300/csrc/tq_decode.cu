// Decode attention entry point: query prep, split-KV partials (compiled per
// head dim and key bits in tq_decode_split_*.cu) and the split combine.

#include <algorithm>

#include "tq_decode_ws.cuh"

namespace tq {

template <int D>
static tq_status launch_dim(DecodeArgs a, cudaStream_t s, void* ev0, void* ev1) {
    const size_t prep_smem = prep_smem_bytes<D>(a.group);
    constexpr size_t kPrepMax = prep_smem_bytes<D>(kMaxG);  // the largest head group's need
    if (prep_smem > kPrepMax) return TQ_ERR_UNSUPPORTED;
    // per-device set-up (the first call on a device does it; before any capture)
    int sms = 0;
    {
        tq_status fs = device_sms(&sms);
        if (fs == TQ_OK) fs = ensure_dynamic_smem((const void*)prep_kernel<D>, (int)kPrepMax, "prep_kernel");
        if (fs != TQ_OK) return fs;
    }
    size_t smem = 0;
    int grid = 0;
    // a uniform key codebook expands over its k_bits single-bit planes only
    // (every multi-bit Walsh term is zero), so its score contraction is
    // shorter; the warp-specialized kernel has instances for that at d = 128
    DecodeGeom gw = a.gm;
    if (D == 128 && a.k_uniform && gw.npk > a.lay.k_bits) {
        gw.npk = a.lay.k_bits;
        gw.npl = gw.npk + (a.lay.k_qjl ? 1 : 0);
        gw.bimg_bytes = gw.n_cols * gw.npl * D;
    }
    if (ws_fits(gw, D)) {
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
    if (grid == 0) {
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
        }
    }
    {
        // the split (and tail) and combine kernels launch programmatically
        // (each one's prologue overlaps the previous kernel's tail) unless
        // profiling events sit between the launches; the query prep launches
        // in stream order (overlapping it with a preceding store measured
        // slower)
        a.pdl = ev0 == nullptr && ev1 == nullptr;
        const cudaError_t e = launch_pdl(false, prep_kernel<D>, dim3(a.heads, a.batch), dim3(kPrepThreads), prep_smem, s, a);
        if (e != cudaSuccess) return cuda_status(e);
    }
    if (grid > 0 && a.tail_cap > 0 && !a.chunk_attn) {
        const size_t tail_smem = (size_t)a.group * D * 4 + (size_t)a.group * kTile * 4 + kMaxG * 4;
        const cudaError_t e = launch_pdl(a.pdl, tail_kernel<D>, dim3(a.heads, a.batch), dim3(128), tail_smem, s, a);
        if (e != cudaSuccess) return cuda_status(e);
    }
    if (ev0) cudaEventRecord((cudaEvent_t)ev0, s);
    tq_status st;
    switch (a.lay.k_bits) {
        case 2: st = dispatch_split<D, 2>(a, s, smem, grid); break;
        case 3: st = dispatch_split<D, 3>(a, s, smem, grid); break;
        default: st = dispatch_split<D, 4>(a, s, smem, grid); break;
    }
    if (st != TQ_OK) return st;
    if (ev1) cudaEventRecord((cudaEvent_t)ev1, s);
    return cuda_status(launch_pdl(a.pdl, combine_kernel<D>, dim3(a.q_heads, a.batch), dim3(128),
                                  (size_t)a.sp.n_splits * sizeof(float), s, a));
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
    a->ws_q = c->ws_q;
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
    a.ws_q = c->ws_q;
    a.ws_bimg = c->ws_bimg;
    a.ws_cst = c->ws_cst;
    a.ws_acc = c->ws_acc;
    a.ws_ml = c->ws_ml;
    return launch_decode(a, s, c->prof_start[TQ_PROF_DECODE_SPLIT], c->prof_stop[TQ_PROF_DECODE_SPLIT]);
}

extern "C" tq_status tq_check_wait_timeout(uint32_t* err_word, uint32_t limit_us, void* stream) {
    if (!err_word || limit_us == 0 || limit_us > 4000000u) return TQ_ERR_INVALID_ARG;
    if ((uintptr_t)err_word & 3) return TQ_ERR_MISALIGNED;
    wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err_word, limit_us * 1000u);
    return cuda_status(cudaGetLastError());
}
