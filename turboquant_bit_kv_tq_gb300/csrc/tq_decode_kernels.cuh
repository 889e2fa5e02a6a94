// Kernels of the decode path (included by the decode translation units).
//
// Decode attention over the compressed paged cache ([Paged] "Which path vLLM
// takes": the decode kernel reads compressed K/V through the block table,
// decodes and attends; [Roadmap] §3.2: grouped query heads, exp2 scaling and a
// fixed NUM_KV_SPLITS grid for CUDA graphs; §4.4: fully-masked rows and empty
// splits must give neither NaN nor a division by zero).
//
// Three launches on the caller's stream:
//   prep     per (KV head, b): R q, S q and q for the grouped query heads,
//            pre-scaled by scale*log2(e); the score operands of the tensor-core
//            contraction (fp8 pieces, register-fragment order) and per-head
//            constants
//   split    per (split, KV head x head group, b): four warps stream 16-token
//            pages through per-warp shared-memory rings filled by bulk async
//            copies; scores are fp8 tensor-core contractions (key code
//            bit-planes x R q, QJL sign plane x S q), then online exp2
//            softmax, then the value contraction on fp16 tensor cores; the
//            newest exact tokens (hybrid tail) are one extra split on CUDA
//            cores -> (m, l, acc) partials
//   combine  per (b, q head): merge the partials, undo the rotation for
//            TurboQuant-MSE values, write out.
//
// Score contraction.  A symmetric codebook value is c[i] = alpha + sum_P
// beta_P u_P(i), u_P an XOR of code bits (host: walsh_planes), so
//   <R q, c[idx]> = alpha sum(R q) + sum_P beta_P <u_P, R q>
// and every <u_P, R q> is a 0/1 matrix times a dense vector.  A stored bit at
// position m of a byte becomes an exact fp8 (e4m3) operand with one AND (m < 7:
// value 2^k_m, k = -9,-8,-7,-6,-5,-3,1) or one AND+OR (m = 7: +-1); the
// per-position factor is folded into the query-side operand, which carries 4
// fp8 pieces (~16 significant bits) as extra matrix columns.
//
// Value contraction.  Group-32 codes become exact fp16 subnormals (q * 2^-24,
// q * 2^-20 by nibble position); the per-(token, group) scale multiplies the
// probabilities (hi + lo fp16 pieces), the zero points add on CUDA cores.
// MSE values use XOR bit-planes of their codes the same way.
#pragma once

#include <cuda_fp8.h>

#include <algorithm>

#include "tq_device.cuh"

namespace tq {

constexpr int kTile = 128;  // tail split: tokens per smem tile
constexpr int kMaxG = 16;
constexpr int kStages = 3;  // per-warp page ring depth
constexpr int kWarpsPerGroup = 4;

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
    DecodeGeom gm;
    float* ws_q;
    uint32_t* ws_frag;
    float* ws_cst;
    float* ws_acc;
    float* ws_ml;
};

// ------------------------------------------------------------ helpers
__device__ __forceinline__ void mma_e4m3(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// fp8 operand of byte-bit position M: u * 2^k_M (M < 7), or 1 - 2u (M = 7)
template <int M>
__device__ __forceinline__ uint32_t bit_operand(uint32_t x) {
    if constexpr (M < 7)
        return x & (0x01010101u << M);
    else
        return (x & 0x80808080u) | 0x38383838u;
}

// factor folded into the query operand for a coordinate at byte-bit m:
// 1 / (value of the single bit) for m < 7, -1/2 for the +-1 form at m = 7
__device__ __forceinline__ float bit_weight(int m) {
    return m == 0 ? 512.f : m == 1 ? 256.f : m == 2 ? 128.f : m == 3 ? 64.f : m == 4 ? 32.f : m == 5 ? 8.f
                                                                                            : m == 6 ? 0.5f : -0.5f;
}

__device__ __forceinline__ float e4m3_to_float(uint8_t v) {
    __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)v, __NV_E4M3);
    return __half2float(__half(hr));
}
__device__ __forceinline__ uint8_t float_to_e4m3(float x) {
    return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

// piece k (0..3) of x * scale: successive e4m3 roundings of the residual, each
// piece scaled by 16 over the previous one
__device__ __forceinline__ uint8_t e4m3_piece(float x, float scale, int k) {
    float y = x * scale;
    uint8_t p = 0;
    for (int i = 0; i <= k; ++i) {
        p = float_to_e4m3(y);
        y = (y - e4m3_to_float(p)) * 16.f;
    }
    return p;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// bounded mbarrier wait; records TQ_DEVERR_TIMEOUT and returns false if the
// phase never completes
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* err) {
    for (int it = 0; it < (1 << 24); ++it) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
    }
    set_error(err, TQ_DEVERR_TIMEOUT);
    return false;
}

// ------------------------------------------------------------------ prep
// ws_q[b][h] = { R q * f, S q * f * sqrt(pi/2)/d, q * f },  f = scale*log2(e);
// ws_cst[b][h] = { C_h, Q_h, 2^-sigmaK, 2^-sigmaQ } and the fp8 score operands:
//   C_h = alpha sum_i (Rq)_i + 1/2 sum_P beta_P sum_{i%8=7} (Rq)_i
//   Q_h = -sum_j (Sq)_j + sum_{j%8=7} (Sq)_j
// (the i%8=7 terms undo the +-1 form of byte-bit 7, see bit_operand).
template <int D>
__global__ void __launch_bounds__(256) prep_kernel(DecodeArgs a) {
    const int g = blockIdx.x, b = blockIdx.y;
    if (b >= a.batch) return;
    const int G = a.group, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    extern __shared__ __align__(16) uint8_t smem[];
    float* qv = reinterpret_cast<float*>(smem);  // [G][D]
    float* rq = qv + G * D;                      // [G][D]
    float* sq = rq + G * D;                      // [G][D]
    float* sig = sq + G * D;                     // [G][2] = 2^sigmaK, 2^sigmaQ
    const int64_t hbase = (int64_t)b * a.q_heads + (int64_t)g * G;
    for (int e = tid; e < G * D; e += blockDim.x)
        qv[e] = a.q_dtype == TQ_DTYPE_F32 ? static_cast<const float*>(a.q)[hbase * D + e]
                                          : bf16_bits_to_float(static_cast<const uint16_t*>(a.q)[hbase * D + e]);
    __syncthreads();
    const float f = a.scale_log2e;
    // R q by an in-warp Hadamard transform (one warp per head)
    for (int h = warp; h < G; h += nwarps) {
        float x[D / 32];
#pragma unroll
        for (int k = 0; k < D / 32; ++k) x[k] = qv[h * D + lane + 32 * k] * a.dp.signs[lane + 32 * k];
        fwht_warp<D / 32>(x, lane);
#pragma unroll
        for (int k = 0; k < D / 32; ++k) rq[h * D + lane + 32 * k] = x[k] * rsqrtf((float)D) * f;
    }
    // S q (thread per output coordinate)
    const float kq = f * sqrtf(1.5707963267948966f) / (float)D;
    for (int e = tid; e < G * D; e += blockDim.x) {
        const int h = e / D, j = e % D;
        float s = 0.f;
        for (int i = 0; i < D; ++i) s = fmaf(a.dp.st_f32[i * D + j], qv[h * D + i], s);
        sq[e] = s * kq;
    }
    __syncthreads();
    float* dst = a.ws_q + hbase * 3 * D;
    for (int e = tid; e < G * D; e += blockDim.x) {
        const int h = e / D, i = e % D;
        dst[h * 3 * D + i] = rq[e];
        dst[h * 3 * D + D + i] = sq[e];
        dst[h * 3 * D + 2 * D + i] = qv[e] * f;
    }
    // per-head constants and operand scales (one warp per head)
    const DecodeGeom gm = a.gm;
    const float* kw = a.dp.k_walsh;
    float bmax = 0.f, bsum = 0.f;
    for (int p = 0; p < gm.npk; ++p) {
        bmax = fmaxf(bmax, fabsf(kw[1 + p]));
        bsum += kw[1 + p];
    }
    for (int h = warp; h < G; h += nwarps) {
        float s_rq = 0.f, s_rq7 = 0.f, s_sq = 0.f, s_sq7 = 0.f, m_rq = 0.f, m_sq = 0.f;
        for (int i = lane; i < D; i += 32) {
            const float r = rq[h * D + i], s = sq[h * D + i];
            s_rq += r;
            s_sq += s;
            if ((i & 7) == 7) {
                s_rq7 += r;
                s_sq7 += s;
            }
            m_rq = fmaxf(m_rq, fabsf(r) * fabsf(bit_weight(i & 7)));
            m_sq = fmaxf(m_sq, fabsf(s) * fabsf(bit_weight(i & 7)));
        }
        s_rq = warp_sum(s_rq);
        s_rq7 = warp_sum(s_rq7);
        s_sq = warp_sum(s_sq);
        s_sq7 = warp_sum(s_sq7);
        m_rq = warp_max(m_rq) * bmax;
        m_sq = warp_max(m_sq) * 2.f;
        if (lane == 0) {
            const int ek = m_rq > 0.f ? (int)floorf(log2f(224.f / m_rq)) : 0;
            const int eq = m_sq > 0.f ? (int)floorf(log2f(224.f / m_sq)) : 0;
            float* c = a.ws_cst + (hbase + h) * 4;
            c[0] = kw[0] * s_rq + 0.5f * bsum * s_rq7;
            c[1] = -s_sq + s_sq7;
            c[2] = ldexpf(1.f, -ek);
            c[3] = ldexpf(1.f, -eq);
            sig[2 * h] = ldexpf(1.f, ek);
            sig[2 * h + 1] = ldexpf(1.f, eq);
        }
    }
    __syncthreads();
    // score operand fragments: word (head group, plane, chunk, tile, reg, lane);
    // byte j of a word is K-row 4*(lane%4) + j (+16 for reg 1) of column lane/4
    constexpr int NCH = D / 32;
    const int words = gm.frag_words;
    uint32_t* fr = a.ws_frag + ((int64_t)b * a.heads + g) * words;
    for (int wi = tid; wi < words; wi += blockDim.x) {
        int x = wi;
        const int ln = x % 32;
        x /= 32;
        const int r = x % 2;
        x /= 2;
        const int T = x % gm.nt;
        x /= gm.nt;
        const int ch = x % NCH;
        x /= NCH;
        const int P = x % gm.npl;
        const int hgi = x / gm.npl;
        const int gq = ln >> 2, tq = ln & 3;
        int head, piece;
        if (gm.nt == 2) {
            head = gq >> 1;
            piece = 2 * T + (gq & 1);
        } else {
            head = gq >> 2;
            piece = gq & 3;
        }
        uint32_t word = 0;
        if (head < gm.hg) {
            const int h = hgi * 4 + head;
            const bool qjl_plane = P == gm.npk;
            const float beta = qjl_plane ? 2.f : kw[1 + P];
            const float* src = qjl_plane ? sq + h * D : rq + h * D;
            const float sc = sig[2 * h + (qjl_plane ? 1 : 0)];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int coord = 128 * (ch >> 2) + 32 * tq + 8 * j + 2 * (ch & 3) + r;
                const float v = beta * src[coord] * bit_weight(coord & 7);
                word |= (uint32_t)e4m3_piece(v, sc, piece) << (8 * j);
            }
        }
        fr[wi] = word;
    }
}

// ----------------------------------------------------------- tail split
// Exact bf16 tail tokens on CUDA cores (scores by (token, head), values by
// coordinate); partial in the same form as the compressed splits.
template <int D>
__device__ void tail_split(const DecodeArgs& a, int g, int b, uint8_t* smem) {
    constexpr int kPerThread = D / 128;
    const int G = a.group, tid = threadIdx.x;
    const int chunk = a.sp.n_chunks;
    float* qs = reinterpret_cast<float*>(smem);  // [G][D] = q * f
    float* pr = qs + G * D;                      // [G][kTile]
    float* sm_m = pr + G * kTile;                // [G]
    for (int e = tid; e < G * D; e += blockDim.x)
        qs[e] = a.ws_q[((int64_t)b * a.q_heads + g * G + e / D) * 3 * D + 2 * D + e % D];
    int tl = a.tail_lens ? a.tail_lens[b] : 0;
    if (tl < 0 || tl > a.tail_cap) {
        if (tid == 0 && g == 0) set_error(a.dp.err, TQ_DEVERR_TAIL);
        tl = max(0, min(tl, a.tail_cap));
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
    const int64_t kv_base = ((int64_t)b * a.heads + g) * a.tail_cap;
    for (int tt = 0; tt < tl; tt += kTile) {
        const int n_tok = min(kTile, tl - tt);
        for (int e = tid; e < G * kTile; e += blockDim.x) pr[e] = -INFINITY;
        __syncthreads();
        for (int e = tid; e < n_tok * G; e += blockDim.x) {
            const int t = e / G, h = e % G;
            const uint16_t* krow = a.tail_k + (kv_base + tt + t) * D;
            float s = 0.f;
            for (int i = 0; i < D; ++i) s = fmaf(qs[h * D + i], bf16_bits_to_float(krow[i]), s);
            pr[h * kTile + t] = s;
        }
        __syncthreads();
        {
            const int lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
            for (int h = warp; h < G; h += nw) {
                float mx = -INFINITY;
                for (int t = lane; t < kTile; t += 32) mx = fmaxf(mx, pr[h * kTile + t]);
                mx = warp_max(mx);
                if (lane == 0) sm_m[h] = fmaxf(mx, m_run[h]);
            }
        }
        __syncthreads();
        for (int e = tid; e < G * kTile; e += blockDim.x) {
            const float sv = pr[e];
            pr[e] = sv == -INFINITY ? 0.f : exp2f(sv - sm_m[e / kTile]);
        }
        __syncthreads();
        for (int h = 0; h < G; ++h) {
            const float m_new = sm_m[h];
            const float alpha = m_run[h] == -INFINITY ? 0.f : exp2f(m_run[h] - m_new);
            float psum = 0.f;
            for (int t = 0; t < n_tok; ++t) psum += pr[h * kTile + t];
            l_run[h] = l_run[h] * alpha + psum;
            m_run[h] = m_new;
#pragma unroll
            for (int p = 0; p < kPerThread; ++p) acc[h][p] *= alpha;
        }
        if (tid < 128) {
#pragma unroll
            for (int p = 0; p < kPerThread; ++p) {
                const int i = tid + 128 * p;
                for (int t = 0; t < n_tok; ++t) {
                    const float v = bf16_bits_to_float(a.tail_v[(kv_base + tt + t) * D + i]);
                    for (int h = 0; h < G; ++h) acc[h][p] = fmaf(pr[h * kTile + t], v, acc[h][p]);
                }
            }
        }
        __syncthreads();
    }
    // MSE values are combined in the rotated space: acc <- R acc = H D acc / sqrt(d)
    if (a.lay.v_mode == TQ_V_MSE) {
        float* buf = qs;
        __syncthreads();
        if (tid < 128)
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int p = 0; p < kPerThread; ++p) buf[h * D + tid + 128 * p] = acc[h][p] * a.dp.signs[tid + 128 * p];
        __syncthreads();
        if (tid < 128)
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int p = 0; p < kPerThread; ++p) {
                    const int i = tid + 128 * p;
                    float s = 0.f;
                    for (int j = 0; j < D; ++j) s += (__popc(i & j) & 1) ? -buf[h * D + j] : buf[h * D + j];
                    acc[h][p] = s * rsqrtf((float)D);
                }
    }
    if (tid < 128)
        for (int h = 0; h < G; ++h) {
            const int64_t idx = ((int64_t)b * a.q_heads + g * G + h) * a.sp.n_splits + chunk;
#pragma unroll
            for (int p = 0; p < kPerThread; ++p) a.ws_acc[idx * D + tid + 128 * p] = acc[h][p];
            if (tid == 0) {
                a.ws_ml[idx * 2] = m_run[h];
                a.ws_ml[idx * 2 + 1] = l_run[h];
            }
        }
}

// -------------------------------------------------------------- split
// shared memory of a compressed-split CTA: per warp a page ring and the
// probability operands, then the rings' mbarriers, then the merge buffer
template <int D>
struct SplitSmem {
    static constexpr int kPbufHalves = 8 * 4 * 2 * 16;  // [<=8 groups/planes][4 heads][2 pieces][16 tokens]
    static __host__ __device__ size_t stride(int page_bytes) { return (size_t)((page_bytes + 127) & ~127); }
    static __host__ __device__ size_t per_warp(int page_bytes) { return kStages * stride(page_bytes) + kPbufHalves * 2; }
    static __host__ __device__ size_t total(int page_bytes) {
        return (size_t)kWarpsPerGroup * per_warp(page_bytes) + (size_t)kWarpsPerGroup * kStages * 8 +
               (size_t)kWarpsPerGroup * 4 * (D + 2) * 4;
    }
};

template <int D, int KB, int NT, bool G32, int VB>
__global__ void __launch_bounds__(128, 2) split_kernel(DecodeArgs a) {
    constexpr int NPK = 1 << (KB - 1);  // key code planes
    constexpr int NCH = D / 32;         // score k-chunks (32 coordinates)
    constexpr int NMT = D / 16;         // value m-tiles (16 coordinates)
    constexpr int NW = D / 128;         // 32-bit words of a bit-plane row per thread role
    constexpr int NPV = G32 ? 1 : (1 << (VB - 1));
    constexpr int NZ = G32 ? D / 32 : 1;
    // one CTA = one head group (4 warps) of one KV head for one split
    const DecodeGeom gm = a.gm;
    const int chunk = blockIdx.x, g = blockIdx.y / gm.nhg, hg = blockIdx.y % gm.nhg, b = blockIdx.z;
    if (b >= a.batch) return;
    extern __shared__ __align__(128) uint8_t smem[];
    if (a.tail_cap > 0 && chunk == a.sp.n_chunks) {
        if (hg == 0) tail_split<D>(a, g, b, smem);  // all G heads of the tail in one CTA
        return;
    }
    const Layout& L = a.lay;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pw = warp;  // page worker: pages pw, pw + 4, ...
    const int gq = lane >> 2, tq = lane & 3;
    const int HG = gm.hg;
    const bool qjl = L.k_qjl;

    // this split's token range
    int len = a.seq_lens[b];
    if (len < 0 || len > a.max_blocks * kBlock) {
        if (threadIdx.x == 0 && g == 0 && chunk == 0 && hg == 0) set_error(a.dp.err, TQ_DEVERR_SEQLEN);
        len = max(0, min(len, a.max_blocks * kBlock));
    }
    const int t0 = chunk * a.split_blocks * kBlock;
    const int t1 = min(len, t0 + a.split_blocks * kBlock);
    const int n_pages = t1 > t0 ? (t1 - t0 + kBlock - 1) / kBlock : 0;

    const int pb = L.page_bytes;
    const size_t pstride = SplitSmem<D>::stride(pb);
    const size_t rings = (size_t)kWarpsPerGroup * SplitSmem<D>::per_warp(pb);
    uint8_t* ring = smem + (size_t)warp * SplitSmem<D>::per_warp(pb);
    __half* pbuf = reinterpret_cast<__half*>(ring + kStages * pstride);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + rings) + warp * kStages;
    float* red = reinterpret_cast<float*>(smem + rings + (size_t)kWarpsPerGroup * kStages * 8);

    // score operands of this head group (registers for the whole split)
    uint32_t bf[NPK + 1][NCH][NT][2];
    {
        const uint32_t* fr = a.ws_frag + ((int64_t)b * a.heads + g) * gm.frag_words;
#pragma unroll
        for (int P = 0; P < NPK + 1; ++P)
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
                for (int T = 0; T < NT; ++T)
#pragma unroll
                    for (int r = 0; r < 2; ++r)
                        bf[P][ch][T][r] = (P == NPK && !qjl)
                                              ? 0u
                                              : fr[((((hg * gm.npl + P) * NCH + ch) * NT + T) * 2 + r) * 32 + lane];
    }
    const int my_head = hg * 4 + tq;  // softmax / value head of this thread (valid if tq < HG)
    const bool head_ok = tq < HG;
    float C = 0.f, Qc = 0.f, scK = 0.f, scQ = 0.f;
    if (head_ok) {
        const float* c = a.ws_cst + ((int64_t)b * a.q_heads + g * a.group + my_head) * 4;
        C = c[0];
        Qc = c[1];
        scK = c[2];
        scQ = c[3];
    }
    float v_alpha = 0.f, v_beta[NPV];
#pragma unroll
    for (int P = 0; P < NPV; ++P) v_beta[P] = G32 ? 0.f : a.dp.v_walsh[1 + P];
    if (!G32) v_alpha = a.dp.v_walsh[0];

    float m_run = -INFINITY, l_part = 0.f;
    float pv[NMT][4];
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt) pv[mt][0] = pv[mt][1] = pv[mt][2] = pv[mt][3] = 0.f;
    float zacc[NZ];
#pragma unroll
    for (int i = 0; i < NZ; ++i) zacc[i] = 0.f;
    for (int e = lane; e < SplitSmem<D>::kPbufHalves; e += 32) pbuf[e] = __float2half(0.f);

    // page ring: lane 0 issues bulk copies completing on the stage's mbarrier
    const int32_t* btab = a.block_table + (int64_t)b * a.max_blocks + t0 / kBlock;
    uint32_t invalid = 0;  // bit s: stage s holds a page with a bad block id (not copied)
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bars[s])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    auto issue = [&](int i, int s) {
        const int blk = btab[i];
        const bool ok = blk >= 0 && blk < a.num_blocks;
        if (ok) {
            if (lane == 0) {
                const uint32_t bar = smem_u32(&bars[s]);
                const uint8_t* src = a.cache + ((int64_t)blk * a.heads + g) * pb;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(pb) : "memory");
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                        smem_u32(ring + s * pstride)),
                    "l"(src), "r"(pb), "r"(bar)
                    : "memory");
            }
            invalid &= ~(1u << s);
        } else {
            if (lane == 0) set_error(a.dp.err, TQ_DEVERR_BLOCK);
            invalid |= 1u << s;
        }
    };
    const int my_pages = n_pages > pw ? (n_pages - pw + kWarpsPerGroup - 1) / kWarpsPerGroup : 0;
    for (int j = 0; j < kStages && j < my_pages; ++j) issue(pw + kWarpsPerGroup * j, j);
    uint32_t phase = 0;  // bit s = parity to wait for on stage s
    int consumed = 0;

    for (int j = 0; j < my_pages; ++j) {
        const int s = j % kStages;
        const int pi = pw + kWarpsPerGroup * j;
        const bool page_ok = !((invalid >> s) & 1);
        if (page_ok) {
            if (!mbar_wait(smem_u32(&bars[s]), (phase >> s) & 1, a.dp.err)) break;
            phase ^= 1u << s;
        }
        consumed = j + 1;
        const uint8_t* pg = ring + s * pstride;
        const int n_valid = min(kBlock, t1 - (t0 + kBlock * pi));
        const bool v0 = page_ok && gq < n_valid, v1 = page_ok && gq + 8 < n_valid;

        // ---------------- scores: key code planes x R q, sign plane x S q
        float ck[NT][4], cq[NT][4];
#pragma unroll
        for (int T = 0; T < NT; ++T)
#pragma unroll
            for (int i = 0; i < 4; ++i) ck[T][i] = cq[T][i] = 0.f;
        {
            uint32_t up[NPK][NW][2];
            {
                uint32_t kw[KB][NW][2];
#pragma unroll
                for (int p = 0; p < KB; ++p)
#pragma unroll
                    for (int w = 0; w < NW; ++w)
#pragma unroll
                        for (int h8 = 0; h8 < 2; ++h8)
                            kw[p][w][h8] = *reinterpret_cast<const uint32_t*>(
                                pg + L.k_codes + (p * kBlock + gq + 8 * h8) * (D / 8) + 4 * (tq + 4 * w));
#pragma unroll
                for (int P = 0; P < NPK; ++P)
#pragma unroll
                    for (int w = 0; w < NW; ++w)
#pragma unroll
                        for (int h8 = 0; h8 < 2; ++h8) {
                            uint32_t x = 0;
#pragma unroll
                            for (int p = 0; p < KB; ++p)
                                if ((plane_subset(KB, P) >> p) & 1) x ^= kw[p][w][h8];
                            up[P][w][h8] = x;
                        }
            }
            uint32_t sw[NW][2] = {};
            if (qjl)
#pragma unroll
                for (int w = 0; w < NW; ++w)
#pragma unroll
                    for (int h8 = 0; h8 < 2; ++h8)
                        sw[w][h8] = *reinterpret_cast<const uint32_t*>(pg + L.k_signs + (gq + 8 * h8) * (D / 8) +
                                                                       4 * (tq + 4 * w));
#define TQ_SCORE_CHUNK(CH, M0)                                                                                  \
    {                                                                                                           \
        constexpr int w_ = (CH) / 4;                                                                            \
        _Pragma("unroll") for (int P = 0; P < NPK; ++P) {                                                       \
            const uint32_t a0 = bit_operand<M0>(up[P][w_][0]), a1 = bit_operand<M0>(up[P][w_][1]);             \
            const uint32_t a2 = bit_operand<M0 + 1>(up[P][w_][0]), a3 = bit_operand<M0 + 1>(up[P][w_][1]);     \
            _Pragma("unroll") for (int T = 0; T < NT; ++T)                                                      \
                mma_e4m3(ck[T], a0, a1, a2, a3, bf[P][CH][T][0], bf[P][CH][T][1]);                             \
        }                                                                                                       \
        if (qjl) {                                                                                              \
            const uint32_t a0 = bit_operand<M0>(sw[w_][0]), a1 = bit_operand<M0>(sw[w_][1]);                   \
            const uint32_t a2 = bit_operand<M0 + 1>(sw[w_][0]), a3 = bit_operand<M0 + 1>(sw[w_][1]);           \
            _Pragma("unroll") for (int T = 0; T < NT; ++T)                                                      \
                mma_e4m3(cq[T], a0, a1, a2, a3, bf[NPK][CH][T][0], bf[NPK][CH][T][1]);                         \
        }                                                                                                       \
    }
            TQ_SCORE_CHUNK(0, 0)
            TQ_SCORE_CHUNK(1, 2)
            TQ_SCORE_CHUNK(2, 4)
            TQ_SCORE_CHUNK(3, 6)
            if constexpr (NCH == 8) {
                TQ_SCORE_CHUNK(4, 0)
                TQ_SCORE_CHUNK(5, 2)
                TQ_SCORE_CHUNK(6, 4)
                TQ_SCORE_CHUNK(7, 6)
            }
#undef TQ_SCORE_CHUNK
        }
        // piece sums -> scores (log2 units) of tokens gq, gq+8 for head tq
        float pk0, pk1, pq0, pq1;
        if constexpr (NT == 2) {
            pk0 = ck[0][0] + ck[0][1] * 0.0625f + ck[1][0] * 0.00390625f + ck[1][1] * 0.000244140625f;
            pk1 = ck[0][2] + ck[0][3] * 0.0625f + ck[1][2] * 0.00390625f + ck[1][3] * 0.000244140625f;
            pq0 = cq[0][0] + cq[0][1] * 0.0625f + cq[1][0] * 0.00390625f + cq[1][1] * 0.000244140625f;
            pq1 = cq[0][2] + cq[0][3] * 0.0625f + cq[1][2] * 0.00390625f + cq[1][3] * 0.000244140625f;
        } else {
            const float w0 = (tq & 1) ? 0.00390625f : 1.f, w1 = (tq & 1) ? 0.000244140625f : 0.0625f;
            pk0 = ck[0][0] * w0 + ck[0][1] * w1;
            pk1 = ck[0][2] * w0 + ck[0][3] * w1;
            pq0 = cq[0][0] * w0 + cq[0][1] * w1;
            pq1 = cq[0][2] * w0 + cq[0][3] * w1;
            pk0 += __shfl_xor_sync(0xffffffffu, pk0, 1);
            pk1 += __shfl_xor_sync(0xffffffffu, pk1, 1);
            pq0 += __shfl_xor_sync(0xffffffffu, pq0, 1);
            pq1 += __shfl_xor_sync(0xffffffffu, pq1, 1);
            // lanes 2h, 2h+1 of a quad hold head h; lane h takes it
            const int src = (lane & ~3) | ((2 * tq) & 3);
            pk0 = __shfl_sync(0xffffffffu, pk0, src);
            pk1 = __shfl_sync(0xffffffffu, pk1, src);
            pq0 = __shfl_sync(0xffffffffu, pq0, src);
            pq1 = __shfl_sync(0xffffffffu, pq1, src);
        }
        const __half* kn = reinterpret_cast<const __half*>(pg + L.k_norm);
        const float n0 = __half2float(kn[gq]), n1 = __half2float(kn[gq + 8]);
        float r0 = 0.f, r1 = 0.f;
        if (qjl) {
            const __half* rn = reinterpret_cast<const __half*>(pg + L.k_rnorm);
            r0 = __half2float(rn[gq]);
            r1 = __half2float(rn[gq + 8]);
        }
        const float s0 = (v0 && head_ok) ? n0 * (C + pk0 * scK) + r0 * (Qc + pq0 * scQ) : -INFINITY;
        const float s1 = (v1 && head_ok) ? n1 * (C + pk1 * scK) + r1 * (Qc + pq1 * scQ) : -INFINITY;

        // ---------------- online softmax (the 8 lanes sharing tq hold one head)
        float mx = fmaxf(s0, s1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float m_new = fmaxf(m_run, mx);
        const float alpha = m_run == -INFINITY ? 0.f : exp2f(m_run - m_new);
        const float p0 = s0 == -INFINITY ? 0.f : exp2f(s0 - m_new);
        const float p1 = s1 == -INFINITY ? 0.f : exp2f(s1 - m_new);
        l_part = l_part * alpha + p0 + p1;
        m_run = m_new;
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) pv[mt][i] *= alpha;
#pragma unroll
        for (int i = 0; i < NZ; ++i) zacc[i] *= alpha;

        // ---------------- probability operands: pbuf[set][head][piece][token]
        // (set = value group for group-32, value plane for MSE; hi + lo fp16)
        auto put = [&](int set, int tok, float x) {
            const __half hi = __float2half_rn(x);
            const __half lo = __float2half_rn(x - __half2float(hi));
            pbuf[((set * 4 + tq) * 2 + 0) * 16 + tok] = hi;
            pbuf[((set * 4 + tq) * 2 + 1) * 16 + tok] = lo;
        };
        if constexpr (G32) {
            const __half* meta0 = reinterpret_cast<const __half*>(pg + L.v_meta + gq * L.v_meta_row);
            const __half* meta1 = reinterpret_cast<const __half*>(pg + L.v_meta + (gq + 8) * L.v_meta_row);
#pragma unroll
            for (int gr = 0; gr < D / 32; ++gr) {
                const float sc0 = __half2float(meta0[2 * gr]), z0 = __half2float(meta0[2 * gr + 1]);
                const float sc1 = __half2float(meta1[2 * gr]), z1 = __half2float(meta1[2 * gr + 1]);
                if (head_ok) {
                    put(gr, gq, p0 * sc0);
                    put(gr, gq + 8, p1 * sc1);
                }
                zacc[gr] = fmaf(p0, z0, fmaf(p1, z1, zacc[gr]));
            }
        } else {
            const __half* vn = reinterpret_cast<const __half*>(pg + L.v_meta);
            const float nv0 = __half2float(vn[gq]), nv1 = __half2float(vn[gq + 8]);
            if (head_ok)
#pragma unroll
                for (int P = 0; P < NPV; ++P) {
                    put(P, gq, p0 * nv0 * v_beta[P]);
                    put(P, gq + 8, p1 * nv1 * v_beta[P]);
                }
            zacc[0] = fmaf(v_alpha, fmaf(p0, nv0, p1 * nv1), zacc[0]);
        }
        __syncwarp();

        // ---------------- values: code operands x probability operands
        {
            const int bh = gq >> 1, bpc = gq & 1;  // B column gq -> (head, piece)
            if constexpr (G32) {
                constexpr int TB = D * VB / 64;  // bytes of a token row per thread role
                constexpr int TW = TB / 4;
                uint32_t va[TW], vb2[TW], vc[TW], vd[TW];
                const uint8_t* vrow = pg + L.v_codes + TB * gq;
#pragma unroll
                for (int w = 0; w < TW; ++w) {
                    va[w] = *reinterpret_cast<const uint32_t*>(vrow + (2 * tq) * L.v_code_row + 4 * w);
                    vb2[w] = *reinterpret_cast<const uint32_t*>(vrow + (2 * tq + 1) * L.v_code_row + 4 * w);
                    vc[w] = *reinterpret_cast<const uint32_t*>(vrow + (2 * tq + 8) * L.v_code_row + 4 * w);
                    vd[w] = *reinterpret_cast<const uint32_t*>(vrow + (2 * tq + 9) * L.v_code_row + 4 * w);
                }
#pragma unroll
                for (int mt = 0; mt < NMT; ++mt) {
                    const int gr = mt >> 1;
                    const __half* bp = &pbuf[((gr * 4 + bh) * 2 + bpc) * 16 + 2 * tq];
                    const uint32_t b0 = *reinterpret_cast<const uint32_t*>(bp);
                    const uint32_t b1 = *reinterpret_cast<const uint32_t*>(bp + 8);
                    const int byte = VB == 4 ? mt : (mt >> 1);
                    const uint32_t sb = byte & 3;
                    const uint32_t sel = sb | (sb << 4) | ((4 + sb) << 8) | ((4 + sb) << 12);
                    const uint32_t r01 = prmt(va[byte >> 2], vb2[byte >> 2], sel);
                    const uint32_t r89 = prmt(vc[byte >> 2], vd[byte >> 2], sel);
                    uint32_t a0, a1, a2, a3;
                    if constexpr (VB == 4) {
                        a0 = r01 & 0x000F000Fu;
                        a1 = r01 & 0x00F000F0u;
                        a2 = r89 & 0x000F000Fu;
                        a3 = r89 & 0x00F000F0u;
                    } else {
                        const int sh = 4 * (mt & 1);
                        a0 = r01 & (0x00030003u << sh);
                        a1 = r01 & (0x000C000Cu << sh);
                        a2 = r89 & (0x00030003u << sh);
                        a3 = r89 & (0x000C000Cu << sh);
                    }
                    mma_f16(pv[mt], a0, a1, a2, a3, b0, b1);
                }
            } else {
                // value bit-planes: thread role gq owns coordinates (D/8)*gq ... + D/8 - 1
                constexpr int CB = D / 64;  // bytes of a plane row per thread role (2 or 4)
                uint32_t wlo[VB][2], whi[VB][2];  // token pairs (2tq, 2tq+1) and (2tq+8, 2tq+9)
#pragma unroll
                for (int p = 0; p < VB; ++p) {
                    const uint8_t* base = pg + L.v_codes + p * kBlock * (D / 8) + CB * gq;
                    if constexpr (CB == 2) {
                        const uint32_t ra = *reinterpret_cast<const uint16_t*>(base + (2 * tq) * (D / 8));
                        const uint32_t rb = *reinterpret_cast<const uint16_t*>(base + (2 * tq + 1) * (D / 8));
                        const uint32_t rc = *reinterpret_cast<const uint16_t*>(base + (2 * tq + 8) * (D / 8));
                        const uint32_t rd = *reinterpret_cast<const uint16_t*>(base + (2 * tq + 9) * (D / 8));
                        wlo[p][0] = ra | (rb << 16);
                        whi[p][0] = rc | (rd << 16);
                        wlo[p][1] = whi[p][1] = 0;
                    } else {
                        const uint32_t ra = *reinterpret_cast<const uint32_t*>(base + (2 * tq) * (D / 8));
                        const uint32_t rb = *reinterpret_cast<const uint32_t*>(base + (2 * tq + 1) * (D / 8));
                        const uint32_t rc = *reinterpret_cast<const uint32_t*>(base + (2 * tq + 8) * (D / 8));
                        const uint32_t rd = *reinterpret_cast<const uint32_t*>(base + (2 * tq + 9) * (D / 8));
                        wlo[p][0] = (ra & 0xFFFFu) | (rb << 16);
                        wlo[p][1] = (ra >> 16) | (rb & 0xFFFF0000u);
                        whi[p][0] = (rc & 0xFFFFu) | (rd << 16);
                        whi[p][1] = (rc >> 16) | (rd & 0xFFFF0000u);
                    }
                }
#pragma unroll
                for (int P = 0; P < NPV; ++P) {
                    uint32_t ul[2] = {0, 0}, uh[2] = {0, 0};
#pragma unroll
                    for (int p = 0; p < VB; ++p)
                        if ((plane_subset(VB, P) >> p) & 1) {
                            ul[0] ^= wlo[p][0];
                            ul[1] ^= wlo[p][1];
                            uh[0] ^= whi[p][0];
                            uh[1] ^= whi[p][1];
                        }
                    const __half* bp = &pbuf[((P * 4 + bh) * 2 + bpc) * 16 + 2 * tq];
                    const uint32_t b0 = *reinterpret_cast<const uint32_t*>(bp);
                    const uint32_t b1 = *reinterpret_cast<const uint32_t*>(bp + 8);
#pragma unroll
                    for (int mt = 0; mt < NMT; ++mt) {
                        const int wsel = mt >> 3, sh = 2 * (mt & 7);
                        const uint32_t a0 = (ul[wsel] >> sh) & 0x00010001u;
                        const uint32_t a1 = (ul[wsel] >> (sh + 1)) & 0x00010001u;
                        const uint32_t a2 = (uh[wsel] >> sh) & 0x00010001u;
                        const uint32_t a3 = (uh[wsel] >> (sh + 1)) & 0x00010001u;
                        mma_f16(pv[mt], a0, a1, a2, a3, b0, b1);
                    }
                }
            }
        }
        __syncwarp();
        // refill this stage with page j + kStages
        if (j + kStages < my_pages) {
            if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            issue(pw + kWarpsPerGroup * (j + kStages), s);
        }
    }
    // a wait that gave up leaves copies in flight: drain them (bounded) before
    // the shared memory is released
    for (int j = consumed; j < my_pages && j < consumed + kStages; ++j) {
        const int s = j % kStages;
        if (!((invalid >> s) & 1)) {
            mbar_wait(smem_u32(&bars[s]), (phase >> s) & 1, a.dp.err);
            phase ^= 1u << s;
        }
    }

    // ---------------- per-warp partial -> smem -> merged split partial
    l_part += __shfl_xor_sync(0xffffffffu, l_part, 4);
    l_part += __shfl_xor_sync(0xffffffffu, l_part, 8);
    l_part += __shfl_xor_sync(0xffffffffu, l_part, 16);
#pragma unroll
    for (int i = 0; i < NZ; ++i) {
        zacc[i] += __shfl_xor_sync(0xffffffffu, zacc[i], 4);
        zacc[i] += __shfl_xor_sync(0xffffffffu, zacc[i], 8);
        zacc[i] += __shfl_xor_sync(0xffffffffu, zacc[i], 16);
    }
    // red[pw][head][0..D-1: acc | D: m | D+1: l]
    float* my = red + (pw * 4 + tq) * (D + 2);
    if (head_ok) {
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) {
            float v0v = pv[mt][0] + pv[mt][1], v1v = pv[mt][2] + pv[mt][3];
            int c0;
            if constexpr (G32) {
                // operand scales: 4-bit q*2^-24 (even slot), q*2^-20 (odd slot);
                // 2-bit q*2^(4(mt%2)-24), q*2^(4(mt%2)-22)
                const float s0 = VB == 4 ? 16777216.f : ((mt & 1) ? 1048576.f : 16777216.f);
                const float s1 = VB == 4 ? 1048576.f : ((mt & 1) ? 262144.f : 4194304.f);
                c0 = 32 * (mt >> 1) + 4 * gq + 2 * (mt & 1);
                v0v = fmaf(v0v, s0, zacc[mt >> 1]);
                v1v = fmaf(v1v, s1, zacc[mt >> 1]);
            } else {
                c0 = (D / 8) * gq + 2 * mt;
                v0v = fmaf(v0v, 16777216.f, zacc[0]);
                v1v = fmaf(v1v, 16777216.f, zacc[0]);
            }
            my[c0] = v0v;
            my[c0 + 1] = v1v;
        }
        if (gq == 0) {
            my[D] = m_run;
            my[D + 1] = l_part;
        }
    }
    __syncthreads();
    // merge the page workers of the head group; write (m, l, acc)
    for (int e = threadIdx.x; e < HG * D; e += blockDim.x) {
        const int h = e / D, i = e % D;
        float M = -INFINITY;
        for (int w = 0; w < kWarpsPerGroup; ++w) M = fmaxf(M, red[(w * 4 + h) * (D + 2) + D]);
        float acc = 0.f, l = 0.f;
        for (int w = 0; w < kWarpsPerGroup; ++w) {
            const float* r = red + (w * 4 + h) * (D + 2);
            if (r[D] == -INFINITY) continue;
            const float wt = exp2f(r[D] - M);
            acc = fmaf(wt, r[i], acc);
            l = fmaf(wt, r[D + 1], l);
        }
        const int64_t idx = ((int64_t)b * a.q_heads + g * a.group + hg * 4 + h) * a.sp.n_splits + chunk;
        a.ws_acc[idx * D + i] = acc;
        if (i == 0) {
            a.ws_ml[idx * 2] = M;
            a.ws_ml[idx * 2 + 1] = l;
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
            for (int p = 0; p < kPerThread; ++p)
                acc[p] = fmaf(w, a.ws_acc[(base + s) * D + threadIdx.x + 128 * p], acc[p]);
        }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
    for (int p = 0; p < kPerThread; ++p) o[threadIdx.x + 128 * p] = acc[p] * inv;
    __syncthreads();
    const int64_t ob = ((int64_t)b * a.q_heads + h) * D;
    if (a.lay.v_mode == TQ_V_MSE) {
        // out = R^T o = D H o / sqrt(d): in-warp Hadamard transform, warp 0
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            float x[D / 32];
#pragma unroll
            for (int k = 0; k < D / 32; ++k) x[k] = o[lane + 32 * k];
            fwht_warp<D / 32>(x, lane);
#pragma unroll
            for (int k = 0; k < D / 32; ++k) {
                const int i = lane + 32 * k;
                const float v = x[k] * a.dp.signs[i] * rsqrtf((float)D);
                if (a.out_dtype == TQ_DTYPE_F32)
                    static_cast<float*>(a.out)[ob + i] = v;
                else
                    static_cast<__nv_bfloat16*>(a.out)[ob + i] = __float2bfloat16_rn(v);
            }
        }
        return;
    }
#pragma unroll
    for (int p = 0; p < kPerThread; ++p) {
        const int i = threadIdx.x + 128 * p;
        if (a.out_dtype == TQ_DTYPE_F32)
            static_cast<float*>(a.out)[ob + i] = o[i];
        else
            static_cast<__nv_bfloat16*>(a.out)[ob + i] = __float2bfloat16_rn(o[i]);
    }
}

// ------------------------------------------------------- split dispatch
template <int D, int KB, int NT, bool G32, int VB>
inline tq_status launch_split(const DecodeArgs& a, cudaStream_t s, size_t smem) {
    auto kern = split_kernel<D, KB, NT, G32, VB>;
    static bool attr_set = false;  // once per kernel instance, before any capture
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess)
            return TQ_ERR_CUDA;
        attr_set = true;
    }
    kern<<<dim3(a.sp.n_splits, a.heads * a.gm.nhg, a.batch), 32 * kWarpsPerGroup, smem, s>>>(a);
    return TQ_OK;
}

template <int D, int KB, int NT>
inline tq_status dispatch_v(const DecodeArgs& a, cudaStream_t s, size_t smem) {
    if (a.lay.v_mode == TQ_V_G32)
        return a.lay.v_bits == 4 ? launch_split<D, KB, NT, true, 4>(a, s, smem)
                                 : launch_split<D, KB, NT, true, 2>(a, s, smem);
    switch (a.lay.v_bits) {
        case 2: return launch_split<D, KB, NT, false, 2>(a, s, smem);
        case 3: return launch_split<D, KB, NT, false, 3>(a, s, smem);
        default: return launch_split<D, KB, NT, false, 4>(a, s, smem);
    }
}

template <int D, int KB>
inline tq_status dispatch_nt(const DecodeArgs& a, cudaStream_t s, size_t smem) {
    return a.gm.nt == 2 ? dispatch_v<D, KB, 2>(a, s, smem) : dispatch_v<D, KB, 1>(a, s, smem);
}

// split-kernel launch for one (head dim, key bits); each pair is compiled in
// its own translation unit
template <int D, int KB>
tq_status dispatch_split(const DecodeArgs& a, cudaStream_t s, size_t smem);

}  // namespace tq
