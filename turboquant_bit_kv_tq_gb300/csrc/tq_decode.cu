// Decode attention over the compressed paged cache ([Paged] "Which path vLLM
// takes": the decode kernel reads compressed K/V through the block table,
// decodes and attends; [Roadmap] §3.2: grouped query heads, exp2 scaling and a
// fixed NUM_KV_SPLITS grid for CUDA graphs; §4.4: fully-masked rows and empty
// splits must give neither NaN nor a division by zero).
//
// Three launches on the caller's stream:
//   prep     per (b, q head): R q, S q and q, pre-scaled by scale*log2(e)
//   split    per (split, KV head, b): scores of the G grouped query heads
//            against the split's compressed tokens (or the exact tail), online
//            softmax, value accumulation -> (m, l, acc) partials
//   combine  per (b, q head): merge the partials, undo the rotation for
//            TurboQuant-MSE values, write out.

#include <algorithm>

#include "tq_device.cuh"

namespace tq {

constexpr int kTile = 128;  // tokens per smem tile (8 cache blocks)
constexpr int kMaxG = 16;

struct DecodeArgs {
    const void* q;
    int q_dtype;
    const uint8_t* cache;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const uint16_t* tail_k;
    const uint16_t* tail_v;
    const int32_t* tail_lens;
    void* out;
    int out_dtype;
    float scale_log2e;  // softmax scale * log2(e)
    int batch;
    int64_t num_blocks;
    int heads, q_heads, group;
    int max_blocks, split_blocks, tail_cap;
    Splits sp;
    Layout lay;
    DeviceParams dp;
    float* ws_q;
    float* ws_acc;
    float* ws_ml;
};

// ------------------------------------------------------------------ prep
// ws_q[b][h] = { R q * f, S q * f * sqrt(pi/2)/d, q * f },  f = scale*log2(e).
template <int D>
__global__ void __launch_bounds__(128) prep_kernel(DecodeArgs a) {
    const int h = blockIdx.x, b = blockIdx.y;
    __shared__ float qs[D];
    const int64_t base = ((int64_t)b * a.q_heads + h) * D;
    for (int i = threadIdx.x; i < D; i += blockDim.x)
        qs[i] = a.q_dtype == TQ_DTYPE_F32 ? static_cast<const float*>(a.q)[base + i]
                                          : bf16_bits_to_float(static_cast<const uint16_t*>(a.q)[base + i]);
    __syncthreads();
    const float f = a.scale_log2e;
    const float kq = f * sqrtf(1.5707963267948966f) / (float)D;
    const float rsd = rsqrtf((float)D);
    float* dst = a.ws_q + ((int64_t)b * a.q_heads + h) * 3 * D;
    for (int i = threadIdx.x; i < D; i += blockDim.x) {
        // (R q)_i = sum_j H_ij D_j q_j / sqrt(d),  H_ij = (-1)^popcount(i & j)
        float rq = 0.f, sq = 0.f;
        for (int j = 0; j < D; ++j) {
            const float t = a.dp.signs[j] * qs[j];
            rq += (__popc(i & j) & 1) ? -t : t;
            sq = fmaf(a.dp.st_f32[j * D + i], qs[j], sq);
        }
        dst[i] = rq * rsd * f;
        dst[D + i] = sq * kq;
        dst[2 * D + i] = qs[i] * f;
    }
}

// ----------------------------------------------------------------- split
__device__ __forceinline__ uint32_t code_at(const uint8_t* row, int i, int b) {
    const int pos = i * b;
    const uint32_t two = (uint32_t)row[pos >> 3] | ((uint32_t)row[(pos >> 3) + 1] << 8);
    return (two >> (pos & 7)) & ((1u << b) - 1);
}

template <int D>
__global__ void __launch_bounds__(128) split_kernel(DecodeArgs a) {
    constexpr int kPerThread = D / 128;  // value coordinates per thread
    const int chunk = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    if (b >= a.batch) return;
    const Layout& L = a.lay;
    const int G = a.group;
    const int tid = threadIdx.x;

    extern __shared__ __align__(16) uint8_t smem[];
    float* qs = reinterpret_cast<float*>(smem);                 // [G][3][D]
    float* pr = qs + G * 3 * D;                                 // [G][kTile] scores -> probs
    float* kc = pr + G * kTile;                                 // [16]
    float* vc = kc + kMaxLevels;                                // [16]
    float* sm_alpha = vc + kMaxLevels;                          // [G]
    int* blk_ok = reinterpret_cast<int*>(sm_alpha + kMaxG);     // [8] block id valid
    uint8_t* pages = reinterpret_cast<uint8_t*>(blk_ok + kTile / kBlock);  // [8][page]

    for (int e = tid; e < G * 3 * D; e += blockDim.x)
        qs[e] = a.ws_q[((int64_t)b * a.q_heads + g * G) * 3 * D + e];
    if (tid < kMaxLevels) {
        kc[tid] = a.dp.k_cent[tid];
        vc[tid] = a.dp.v_cent[tid];
    }

    // token range of this split
    const bool is_tail = a.tail_cap > 0 && chunk == a.sp.n_chunks;
    int t0 = 0, t1 = 0;
    if (is_tail) {
        int tl = a.tail_lens ? a.tail_lens[b] : 0;
        if (tl < 0 || tl > a.tail_cap) {
            if (tid == 0 && g == 0) set_error(a.dp.err, TQ_DEVERR_TAIL);
            tl = max(0, min(tl, a.tail_cap));
        }
        t1 = tl;
    } else {
        int len = a.seq_lens[b];
        if (len < 0 || len > a.max_blocks * kBlock) {
            if (tid == 0 && g == 0 && chunk == 0) set_error(a.dp.err, TQ_DEVERR_SEQLEN);
            len = max(0, min(len, a.max_blocks * kBlock));
        }
        t0 = min(len, chunk * a.split_blocks * kBlock);
        t1 = min(len, (chunk + 1) * a.split_blocks * kBlock);
    }

    float m_run[kMaxG], l_run[kMaxG], acc[kMaxG][kPerThread];
#pragma unroll
    for (int h = 0; h < kMaxG; ++h) {
        m_run[h] = -INFINITY;
        l_run[h] = 0.f;
#pragma unroll
        for (int p = 0; p < kPerThread; ++p) acc[h][p] = 0.f;
    }
    __syncthreads();

    const int nb_k = (1 << L.k_bits);
    (void)nb_k;
    for (int tt = t0; tt < t1; tt += kTile) {
        const int n_tok = min(kTile, t1 - tt);
        // ---- stage the tile's pages (compressed) ----
        if (!is_tail) {
            const int nblk = (n_tok + kBlock - 1) / kBlock;
            const int words = L.page_bytes / 16;
            for (int e = tid; e < nblk * words; e += blockDim.x) {
                const int j = e / words, wv = e - j * words;
                const int blk = a.block_table[(int64_t)b * a.max_blocks + tt / kBlock + j];
                const bool ok = blk >= 0 && blk < a.num_blocks;
                uint4 val = make_uint4(0, 0, 0, 0);
                if (ok) val = reinterpret_cast<const uint4*>(a.cache + ((int64_t)blk * a.heads + g) * L.page_bytes)[wv];
                if (wv == 0) {
                    blk_ok[j] = ok;
                    if (!ok) set_error(a.dp.err, TQ_DEVERR_BLOCK);
                }
                reinterpret_cast<uint4*>(pages + j * L.page_bytes)[wv] = val;
            }
        }
        __syncthreads();
        // ---- scores: thread = token ----
        if (tid < n_tok) {
            float s[kMaxG];
            if (!is_tail) {
                const uint8_t* page = pages + (tid / kBlock) * L.page_bytes;
                const int row = tid % kBlock;
                const uint8_t* crow = page + L.k_codes + row * L.k_code_row;
                float dc[kMaxG], ds[kMaxG];
#pragma unroll
                for (int h = 0; h < kMaxG; ++h) dc[h] = ds[h] = 0.f;
                for (int i = 0; i < D; ++i) {
                    const float c = kc[code_at(crow, i, L.k_bits)];
#pragma unroll
                    for (int h = 0; h < kMaxG; ++h)
                        if (h < G) dc[h] = fmaf(qs[h * 3 * D + i], c, dc[h]);
                }
                const float n16 = __half2float(reinterpret_cast<const __half*>(page + L.k_norm)[row]);
                float rho = 0.f;
                if (L.k_qjl) {
                    const uint8_t* srow = page + L.k_signs + row * L.k_sign_row;
                    for (int j = 0; j < D; ++j) {
                        const bool pos = (srow[j >> 3] >> (j & 7)) & 1;
#pragma unroll
                        for (int h = 0; h < kMaxG; ++h)
                            if (h < G) {
                                const float sq = qs[h * 3 * D + D + j];
                                ds[h] += pos ? sq : -sq;
                            }
                    }
                    rho = __half2float(reinterpret_cast<const __half*>(page + L.k_rnorm)[row]);
                }
                const bool ok = blk_ok[tid / kBlock];
#pragma unroll
                for (int h = 0; h < kMaxG; ++h) s[h] = ok ? n16 * dc[h] + rho * ds[h] : -INFINITY;
            } else {
                const uint16_t* krow = a.tail_k + (((int64_t)b * a.heads + g) * a.tail_cap + tt + tid) * D;
#pragma unroll
                for (int h = 0; h < kMaxG; ++h) s[h] = 0.f;
                for (int i = 0; i < D; ++i) {
                    const float kv = bf16_bits_to_float(krow[i]);
#pragma unroll
                    for (int h = 0; h < kMaxG; ++h)
                        if (h < G) s[h] = fmaf(qs[h * 3 * D + 2 * D + i], kv, s[h]);
                }
            }
#pragma unroll
            for (int h = 0; h < kMaxG; ++h)
                if (h < G) pr[h * kTile + tid] = s[h];
        } else {
            for (int h = 0; h < G; ++h) pr[h * kTile + tid] = -INFINITY;
        }
        __syncthreads();
        // ---- online softmax per head (warp w handles heads w, w+4, ...) ----
        {
            const int lane = tid & 31, warp = tid >> 5;
            for (int h = warp; h < G; h += 4) {
                float mx = -INFINITY;
                for (int t = lane; t < kTile; t += 32) mx = fmaxf(mx, pr[h * kTile + t]);
                mx = warp_max(mx);
                // m_run is replicated per thread; every thread of the CTA
                // recomputes the same max below, here only probabilities.
                const float m_old = m_run[h];
                const float m_new = fmaxf(m_old, mx);
                for (int t = lane; t < kTile; t += 32) {
                    const float sv = pr[h * kTile + t];
                    pr[h * kTile + t] = sv == -INFINITY ? 0.f : exp2f(sv - m_new);
                }
                if (lane == 0) sm_alpha[h] = m_new;
            }
        }
        __syncthreads();
        // every thread updates its copy of (m, l) and rescales its accumulators
        for (int h = 0; h < G; ++h) {
            const float m_new = sm_alpha[h];
            const float alpha = m_run[h] == -INFINITY ? 0.f : exp2f(m_run[h] - m_new);
            float psum = 0.f;
            for (int t = 0; t < n_tok; ++t) psum += pr[h * kTile + t];
            l_run[h] = l_run[h] * alpha + psum;
            m_run[h] = m_new;
#pragma unroll
            for (int p = 0; p < kPerThread; ++p) acc[h][p] *= alpha;
        }
        // ---- value accumulation: thread = coordinate ----
#pragma unroll
        for (int p = 0; p < kPerThread; ++p) {
            const int i = tid + 128 * p;
            for (int t = 0; t < n_tok; ++t) {
                float vhat;
                if (!is_tail) {
                    const uint8_t* page = pages + (t / kBlock) * L.page_bytes;
                    const int row = t % kBlock;
                    const uint32_t code = code_at(page + L.v_codes + row * L.v_code_row, i, L.v_bits);
                    if (L.v_mode == TQ_V_MSE) {
                        const float vn = __half2float(reinterpret_cast<const __half*>(page + L.v_meta)[row]);
                        vhat = vn * vc[code];
                    } else {
                        const __half* sz = reinterpret_cast<const __half*>(page + L.v_meta + row * L.v_meta_row);
                        vhat = (float)code * __half2float(sz[2 * (i >> 5)]) + __half2float(sz[2 * (i >> 5) + 1]);
                    }
                } else {
                    vhat = bf16_bits_to_float(
                        a.tail_v[(((int64_t)b * a.heads + g) * a.tail_cap + tt + t) * D + i]);
                }
#pragma unroll
                for (int h = 0; h < kMaxG; ++h)
                    if (h < G) acc[h][p] = fmaf(pr[h * kTile + t], vhat, acc[h][p]);
            }
        }
        __syncthreads();
    }

    // tail accumulators live in original space; MSE values are combined in the
    // rotated space, so rotate them: acc <- R acc = H D acc / sqrt(d)
    if (is_tail && L.v_mode == TQ_V_MSE) {
        float* buf = pr;  // reuse: needs G*D floats <= G*kTile*... use qs region instead
        buf = qs;         // qs no longer needed
        __syncthreads();
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int p = 0; p < kPerThread; ++p) buf[h * D + tid + 128 * p] = acc[h][p] * a.dp.signs[tid + 128 * p];
        __syncthreads();
        const float rsd = rsqrtf((float)D);
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int p = 0; p < kPerThread; ++p) {
                const int i = tid + 128 * p;
                float sacc = 0.f;
                for (int j = 0; j < D; ++j) sacc += (__popc(i & j) & 1) ? -buf[h * D + j] : buf[h * D + j];
                acc[h][p] = sacc * rsd;
            }
    }

    // ---- write partials ----
    for (int h = 0; h < G; ++h) {
        const int64_t idx = (((int64_t)b * a.q_heads + g * G + h) * a.sp.n_splits + chunk);
#pragma unroll
        for (int p = 0; p < kPerThread; ++p) a.ws_acc[idx * D + tid + 128 * p] = acc[h][p];
        if (tid == 0) {
            a.ws_ml[idx * 2] = m_run[h];
            a.ws_ml[idx * 2 + 1] = l_run[h];
        }
    }
}

// --------------------------------------------------------------- combine
template <int D>
__global__ void __launch_bounds__(128) combine_kernel(DecodeArgs a) {
    constexpr int kPerThread = D / 128;
    const int h = blockIdx.x, b = blockIdx.y;
    if (b >= a.batch) return;
    const int S = a.sp.n_splits;
    const int64_t base = ((int64_t)b * a.q_heads + h) * S;
    __shared__ float o[D];
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, a.ws_ml[(base + s) * 2]);
    float lsum = 0.f, acc[kPerThread];
#pragma unroll
    for (int p = 0; p < kPerThread; ++p) acc[p] = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < S; ++s) {
            const float m = a.ws_ml[(base + s) * 2];
            if (m == -INFINITY) continue;  // empty split
            const float w = exp2f(m - M);
            lsum = fmaf(w, a.ws_ml[(base + s) * 2 + 1], lsum);
#pragma unroll
            for (int p = 0; p < kPerThread; ++p) acc[p] = fmaf(w, a.ws_acc[(base + s) * D + threadIdx.x + 128 * p], acc[p]);
        }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
    for (int p = 0; p < kPerThread; ++p) o[threadIdx.x + 128 * p] = acc[p] * inv;
    __syncthreads();
    const int64_t ob = ((int64_t)b * a.q_heads + h) * D;
#pragma unroll
    for (int p = 0; p < kPerThread; ++p) {
        const int i = threadIdx.x + 128 * p;
        float v = o[i];
        if (a.lay.v_mode == TQ_V_MSE) {
            // out = R^T o = D H o / sqrt(d)
            float sacc = 0.f;
            for (int j = 0; j < D; ++j) sacc += (__popc(i & j) & 1) ? -o[j] : o[j];
            v = sacc * a.dp.signs[i] * rsqrtf((float)D);
        }
        if (a.out_dtype == TQ_DTYPE_F32)
            static_cast<float*>(a.out)[ob + i] = v;
        else
            static_cast<__nv_bfloat16*>(a.out)[ob + i] = __float2bfloat16_rn(v);
    }
}

template <int D>
static tq_status launch(const DecodeArgs& a, cudaStream_t s, void* ev0, void* ev1) {
    prep_kernel<D><<<dim3(a.q_heads, a.batch), 128, 0, s>>>(a);
    const size_t smem = (size_t)a.group * 3 * D * 4 + (size_t)a.group * kTile * 4 + 2 * kMaxLevels * 4 + kMaxG * 4 +
                        (kTile / kBlock) * 4 + (size_t)(kTile / kBlock) * a.lay.page_bytes;
    auto kern = split_kernel<D>;
    static bool attr_set = false;  // once per kernel instance, before any capture
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) != cudaSuccess)
            return TQ_ERR_CUDA;
        attr_set = true;
    }
    if (smem > 200 * 1024) return TQ_ERR_UNSUPPORTED;
    if (ev0) cudaEventRecord((cudaEvent_t)ev0, s);
    kern<<<dim3(a.sp.n_splits, a.heads, a.batch), 128, smem, s>>>(a);
    if (ev1) cudaEventRecord((cudaEvent_t)ev1, s);
    combine_kernel<D><<<dim3(a.q_heads, a.batch), 128, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace tq

using namespace tq;

extern "C" tq_status tq_decode_attention(const tq_cache* c, const void* q, int q_dtype, const void* cache_buf,
                                         const int32_t* block_table, const int32_t* seq_lens, const void* tail_k,
                                         const void* tail_v, const int32_t* tail_lens, float scale, int batch,
                                         void* out, int out_dtype, void* stream) {
    if (!c || !q || !cache_buf || !block_table || !seq_lens || !out) return TQ_ERR_INVALID_ARG;
    if (batch < 1 || batch > c->cfg.max_batch) return TQ_ERR_INVALID_ARG;
    if (q_dtype != TQ_DTYPE_F32 && q_dtype != TQ_DTYPE_BF16) return TQ_ERR_INVALID_ARG;
    if (out_dtype != TQ_DTYPE_F32 && out_dtype != TQ_DTYPE_BF16) return TQ_ERR_INVALID_ARG;
    const bool has_tail = tail_k != nullptr || tail_v != nullptr || tail_lens != nullptr;
    if (has_tail && (!tail_k || !tail_v || !tail_lens || c->cfg.tail_cap == 0)) return TQ_ERR_INVALID_ARG;
    if ((uintptr_t)cache_buf & 15) return TQ_ERR_MISALIGNED;
    DecodeArgs a;
    a.q = q;
    a.q_dtype = q_dtype;
    a.cache = static_cast<const uint8_t*>(cache_buf);
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.tail_k = static_cast<const uint16_t*>(tail_k);
    a.tail_v = static_cast<const uint16_t*>(tail_v);
    a.tail_lens = tail_lens;
    a.out = out;
    a.out_dtype = out_dtype;
    const int d = c->cfg.head_dim;
    const float sc = scale > 0.f ? scale : 1.0f / sqrtf((float)d);
    a.scale_log2e = sc * 1.4426950408889634f;
    a.batch = batch;
    a.num_blocks = c->cfg.num_blocks;
    a.heads = c->cfg.num_kv_heads;
    a.q_heads = c->cfg.num_q_heads;
    a.group = a.q_heads / a.heads;
    a.max_blocks = c->cfg.max_blocks_per_seq;
    a.split_blocks = c->cfg.split_blocks;
    a.tail_cap = has_tail ? c->cfg.tail_cap : 0;
    a.sp = c->splits;
    a.lay = c->lay;
    a.dp = c->dp;
    a.ws_q = c->ws_q;
    a.ws_acc = c->ws_acc;
    a.ws_ml = c->ws_ml;
    cudaStream_t s = (cudaStream_t)stream;
    void *e0 = c->prof_start[TQ_PROF_DECODE_SPLIT], *e1 = c->prof_stop[TQ_PROF_DECODE_SPLIT];
    return d == 128 ? launch<128>(a, s, e0, e1) : launch<256>(a, s, e0, e1);
}
