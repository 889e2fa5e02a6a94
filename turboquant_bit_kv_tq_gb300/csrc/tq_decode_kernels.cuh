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
//            pre-scaled by scale*log2(e); per-head constants and the score
//            operand image (fp8 pieces in the tensor-core shared-memory layout)
//   split    per (split, KV head x head group, b): 128-token tiles of pages
//            staged by bulk async copies; scores are fp8 tcgen05 contractions
//            (key code bit-planes x R q, QJL sign plane x S q) accumulated in
//            tensor memory, then online exp2 softmax, then the value
//            contraction on fp16 tensor cores; the newest exact tokens (hybrid
//            tail) are one extra split on CUDA cores -> (m, l, acc) partials
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
// fp8 pieces (~20 significant bits) as extra matrix rows (N = 5 per head).
//
// Value contraction.  Group-32 codes become exact fp16 subnormals (q * 2^-24,
// q * 2^-20 by nibble position); the per-(token, group) scale multiplies the
// probabilities (hi + lo fp16 pieces), the zero points add on CUDA cores.
// MSE values use the XOR bit-planes of their codes as +-1 operands, so that the
// codebook's constant term (which the inverse rotation would put entirely into
// output coordinate 0) vanishes for a symmetric codebook instead of cancelling.
#pragma once

#include <cuda_fp8.h>

#include <algorithm>
#include <type_traits>

#include "tq_device.cuh"

namespace tq {

constexpr int kTile = 128;  // tail split: tokens per smem tile
constexpr int kMaxG = 16;
constexpr int kTailV = 64;  // tail split: value rows staged in shared memory at a time
// shared memory of the exact tail split: scaled queries, scores, maxima and
// the staged value rows (bf16)
template <int D>
__host__ __device__ constexpr size_t tail_smem_bytes(int G) {
    return (size_t)G * D * 4 + (size_t)G * kTile * 4 + kMaxG * 4 + (size_t)kTailV * D * 2;
}
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
    bool out_rotated;  // MSE values: leave the output in the rotated space (no R^T)
    bool k_uniform;    // the key codebook is a uniform grid
    // extend attention: batch entry b is one new token; row_of[b] is its
    // sequence's block-table row, and its exact tail tokens are rows
    // tail_base[b] + i of a token-major [tokens][H_kv][d] buffer.  Both null
    // for decode (row b; tail [B][H_kv][tail_cap][d]).
    const int32_t* row_of = nullptr;
    const int32_t* tail_base = nullptr;
    bool chunk_attn = false;  // the tail partials come from chunk_attn_kernel
    // extend: query blocks {first entry, entries, sequence, index of the
    // block's first prefix work item} and {block count, item count} for
    // extend_prefix_kernel (null otherwise)
    const int4* xblocks = nullptr;
    const int32_t* xcounts = nullptr;
    int xblocks_max = 0;  // the plan's capacity (an upper bound of the block count)
    int prep_entries = 1;  // batch entries per query-prep CTA
    // the query prep releases its dependents at its end rather than at its
    // start (before the extend prefix kernel, which takes a whole SM)
    bool prep_late_release = false;
    // the query prep's predecessor is a store kernel launched without the
    // programmatic attribute, so everything that wrote the queries finished
    // before it began: the prep loads its queries and computes R q and S q
    // before its wait (which still comes before any write; its completion
    // then implies the store's, which the split kernel relies on)
    bool q_early = false;
    float scale_log2e;  // softmax scale * log2(e)
    int batch;
    int64_t num_blocks;
    int heads, q_heads, group;
    int max_blocks, split_blocks, tail_cap;
    int stages;  // split ring depth (tiles)
    bool pdl;    // split and combine launch programmatically (no profiling events between them)
    Splits sp;
    Layout lay;
    DeviceParams dp;
    DecodeGeom gm;
    uint8_t* ws_bimg;
    float* ws_cst;
    float* ws_acc;
    float* ws_ml;
};

// ------------------------------------------------------------ helpers
__device__ __forceinline__ void mma_e4m3(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm(
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

// 2^x for x <= 0 (softmax weights; approximate to ~2 ulp)
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// lazy softmax rescaling: the running reference maximum only moves when a new
// score exceeds it by more than this many log2 units (weights stay <= 2^8)
constexpr float kRescaleSlack = 8.f;

// sum of the kPieces piece accumulators of one head (fp32 bit patterns)
__device__ __forceinline__ float piece_sum(const uint32_t* c) {
    float x = __uint_as_float(c[kPieces - 1]);
#pragma unroll
    for (int k = kPieces - 2; k >= 0; --k) x = fmaf(x, 0.0625f, __uint_as_float(c[k]));
    return x;
}

// Instruction descriptor of a dense fp8 (e4m3 x e4m3) MMA with fp32
// accumulation, both operands K-major, M = 128.
__host__ __device__ constexpr uint32_t fp8_idesc(int n) { return (1u << 4) | ((uint32_t)(n >> 3) << 17) | (8u << 24); }

// D[128 x N] (+)= A[128 x 32] * B[N x 32]^T with A in tensor memory, B in
// shared memory; issued by one thread
__device__ __forceinline__ void mma_fp8_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}
// ------------------------------------------------------------------ prep
__device__ __forceinline__ void mma_bf16f32(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two 8x8 b16 matrices from shared memory, transposed: lanes 0-7 give the row
// addresses (16 bytes each, 16-byte aligned) of the first, lanes 8-15 of the
// second; r0/r1 then hold a k-major [16 x 8] block as an mma B fragment.
__device__ __forceinline__ void ldsm_x2_trans(uint32_t& r0, uint32_t& r1, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}
// f = scale*log2(e); R q * f
// and S q * f * sqrt(pi/2)/d stay in shared memory for what follows:
// ws_cst[b][h] = { C_h, Q_h, 2^-sigmaK, 2^-sigmaQ } with
//   C_h = alpha sum_i (Rq)_i + 1/2 sum_P beta_P sum_{i%8=7} (Rq)_i
//   Q_h = -sum_j (Sq)_j + sum_{j%8=7} (Sq)_j
// (the i%8=7 terms undo the +-1 form of byte-bit 7, see bit_operand), and the
// score operand image of every head group: row n = kPieces*head + piece, K index
// kk = P*d + 4*col + e holds piece `piece` of
//   beta_P * (R q)_c * bit_weight(c%8) * 2^sigmaK   (key plane P < npk)
//   2 * (S q)_c * bit_weight(c%8) * 2^sigmaQ        (sign plane P = npk)
// for coordinate c = 32*(col/8) + 8*e + col%8: the coordinate that byte e of
// tensor-memory column col of plane P holds in the split kernel.
// One CTA serves prep_entries consecutive batch entries of one KV head (1 for
// decode; a block of extend's new tokens): their E x G query heads are handled
// as "virtual heads" v = e G + h, with S^T staged once.  Every head's
// arithmetic is the same for any entry count.
constexpr int kPrepMaxV = 32;  // virtual heads per CTA at most
// the staged queries' row pitch is D + kPrepQPad floats, so that the eight
// rows of an mma A fragment fall on different banks
constexpr int kPrepQPad = 8;
template <int D>
__host__ __device__ constexpr size_t prep_smem_bytes(int GV) {
    return (size_t)D * D * 2 + (size_t)3 * GV * D * 4 + (size_t)GV * kPrepQPad * 4 + 2 * kPrepMaxV * 4 + 16;
}

constexpr int kPrepThreads = 512;  // its phases are short serial chains
template <int D>
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(DecodeArgs a) {
    // launched programmatically: the preceding kernel (the step's store, or
    // whatever wrote the queries) must be complete before anything is read,
    // unless q_early says the queries were complete before that kernel began
    if (!a.q_early) pdl_wait();
    // the split kernel's prologue may start (with q_early once the store is
    // done: its CTAs would otherwise sit beside the store's)
    if (!a.prep_late_release && !a.q_early) pdl_launch_dependents();
    const int g = blockIdx.x, E = a.prep_entries, b0 = blockIdx.y * E;
    const int ne = min(E, a.batch - b0);
    if (ne <= 0) {
        if (a.q_early) pdl_wait();
        return;
    }
    // an extend entry with no compressed prefix uses none of this (its exact
    // part reads the raw queries)
    if (a.chunk_attn) {
        bool any = false;
        for (int e = 0; e < ne; ++e) any |= a.seq_lens[b0 + e] > 0;
        if (!any) {
            if (a.q_early) pdl_wait();
            return;
        }
    }
    const int G = a.group, GV = ne * G, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5,
              nwarps = blockDim.x >> 5;
    // global query-head row of virtual head v
    auto hrow = [&](int v) { return (int64_t)(b0 + v / G) * a.q_heads + (int64_t)g * G + v % G; };
    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t* st = reinterpret_cast<uint16_t*>(smem);           // S^T bf16 [D][D]
    constexpr int QS = D + kPrepQPad;                           // row pitch of qv
    float* qv = reinterpret_cast<float*>(smem + (size_t)D * D * 2);  // [GV][QS]
    float* rq = qv + GV * QS;                                   // [GV][D]
    float* sq = rq + GV * D;                                    // [GV][D]
    float* sig = sq + GV * D;                                   // [kPrepMaxV][2] = 2^sigmaK, 2^sigmaQ
    uint64_t* bar = reinterpret_cast<uint64_t*>(sig + 2 * kMaxG);
    if (tid == 0) {
        mbar_init(smem_u32(bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_expect_tx(smem_u32(bar), D * D * 2);
        bulk_copy(smem_u32(st), a.dp.st_bf16, D * D * 2, smem_u32(bar));
    }
    // the queries, the rotation signs and the key codebook's Walsh terms load
    // together (one memory latency), the S^T copy meanwhile
    __shared__ float s_signs[D], s_kw[9];
    for (int e = tid; e < GV * D; e += blockDim.x) {
        const int64_t src = hrow(e / D) * D + e % D;
        qv[(e / D) * QS + e % D] = a.q_dtype == TQ_DTYPE_F32 ? static_cast<const float*>(a.q)[src]
                                          : bf16_bits_to_float(static_cast<const uint16_t*>(a.q)[src]);
    }
    for (int e = tid; e < D; e += blockDim.x) s_signs[e] = a.dp.signs[e];
    if (tid < 9) s_kw[tid] = a.dp.k_walsh[tid];
    __syncthreads();
    const float f = a.scale_log2e;
    // per-head sums and maxima for the constants below: [head][0..2] sum, sum
    // over i % 8 = 7, max of |v| bit_weight(i % 8) of R q (one entry per head)
    // and of S q (one entry per warp of the head, on the one-pass S q path;
    // the tensor-core path takes them in the constants phase)
    constexpr int kSqWarps = D / 64;  // warps per head in the one-pass S q
    __shared__ float red_r[kPrepMaxV][3], red_s[kPrepMaxV][kSqWarps][3];
    // R q by an in-warp Hadamard transform (one warp per head)
    for (int h = warp; h < GV; h += nwarps) {
        float x[D / 32];
#pragma unroll
        for (int k = 0; k < D / 32; ++k) x[k] = qv[h * QS + lane + 32 * k] * s_signs[lane + 32 * k];
        fwht_warp<D / 32>(x, lane);
        const float bw = fabsf(bit_weight(lane & 7));  // i % 8 = lane % 8 for i = lane + 32 k
        float s0 = 0.f, m0 = 0.f;
#pragma unroll
        for (int k = 0; k < D / 32; ++k) {
            const float r = x[k] * rsqrtf((float)D) * f;
            rq[h * D + lane + 32 * k] = r;
            s0 += r;
            m0 = fmaxf(m0, fabsf(r) * bw);
        }
        const float s7 = warp_sum((lane & 7) == 7 ? s0 : 0.f);
        s0 = warp_sum(s0);
        m0 = warp_max(m0);
        if (lane == 0) {
            red_r[h][0] = s0;
            red_r[h][1] = s7;
            red_r[h][2] = m0;
        }
    }
    // S q.  When one pass of single heads covers the CTA's heads (decode's
    // head groups at d = 128): thread (column pair j, j + 1; head), 32-bit
    // loads of S^T pairs and 128-bit loads of four query elements, with the
    // head's sums taken in the same pass.  Otherwise (more heads, d = 256)
    // on the tensor cores, sums in the constants phase.
    bool s_ok = mbar_wait(smem_u32(bar), 0, a.dp.err);
    const float kq = f * sqrtf(1.5707963267948966f) / (float)D;
    const bool sq_tc = GV > kPrepThreads / (D / 2);
    auto sq_pass = [&](auto hpt_c) {
        constexpr int HPT = decltype(hpt_c)::value;
        constexpr int NP = D / 2;                 // column pairs
        constexpr int HS = kPrepThreads / NP;     // head blocks covered per pass
        const int jp = tid % NP, b0h = tid / NP;  // (warp-uniform b0h)
        for (int hb = b0h; hb * HPT < GV; hb += HS) {
            float s0[HPT][2], s1[HPT][2];  // two partial sums per column and head
#pragma unroll
            for (int hh = 0; hh < HPT; ++hh) s0[hh][0] = s0[hh][1] = s1[hh][0] = s1[hh][1] = 0.f;
            if (s_ok) {
#pragma unroll 2
                for (int i4 = 0; i4 < D / 4; ++i4) {
                    uint32_t pr[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) pr[u] = *reinterpret_cast<const uint32_t*>(st + (4 * i4 + u) * D + 2 * jp);
#pragma unroll
                    for (int hh = 0; hh < HPT; ++hh) {
                        const int h = hb * HPT + hh;
                        if (h < GV) {
                            const float4 qq = reinterpret_cast<const float4*>(qv + h * QS)[i4];
                            const float qa[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                s0[hh][u & 1] = fmaf(__uint_as_float(pr[u] << 16), qa[u], s0[hh][u & 1]);
                                s1[hh][u & 1] = fmaf(__uint_as_float(pr[u] & 0xFFFF0000u), qa[u], s1[hh][u & 1]);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int hh = 0; hh < HPT; ++hh) {
                const int h = hb * HPT + hh;
                if (h >= GV) break;
                const float v0 = (s0[hh][0] + s0[hh][1]) * kq, v1 = (s1[hh][0] + s1[hh][1]) * kq;
                sq[h * D + 2 * jp] = v0;
                sq[h * D + 2 * jp + 1] = v1;
                // columns 2jp (i % 8 even) and 2jp + 1 (i % 8 = 7 when jp % 4 = 3)
                float sum = warp_sum(v0 + v1);
                float s7 = warp_sum((jp & 3) == 3 ? v1 : 0.f);
                float mx = warp_max(fmaxf(fabsf(v0) * fabsf(bit_weight((2 * jp) & 7)),
                                          fabsf(v1) * fabsf(bit_weight((2 * jp + 1) & 7))));
                if (lane == 0) {
                    const int wh = (jp >> 5);  // this warp's place among the head's warps
                    red_s[h][wh][0] = sum;
                    red_s[h][wh][1] = s7;
                    red_s[h][wh][2] = mx;
                }
            }
        }
    };
    if (!sq_tc) sq_pass(std::integral_constant<int, 1>{});
    if (sq_tc && s_ok) {
        // tensor cores: sq[h][j] = kq sum_i q[h][i] S^T[i][j] with bf16 operands
        // and fp32 accumulation (a bf16 query is exact in one part, an fp32
        // query is split into three bf16 parts); warp w takes the 8-column
        // blocks nt = w, w + nwarps, ... of every head
        const int g8 = lane >> 2, t4 = lane & 3;
        const int nparts = a.q_dtype == TQ_DTYPE_F32 ? 3 : 1;
        static_assert(kPrepMaxV <= 32, "two 16-head row tiles at most");
        for (int nt = warp; nt < D / 8; nt += nwarps) {
            float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 2
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t b0, b1;
                ldsm_x2_trans(b0, b1, smem_u32(st + (16 * ks + (lane & 15)) * D + 8 * nt));
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    if (16 * mt >= GV) break;
                    // A rows: heads 16 mt + g8 and 16 mt + g8 + 8; columns
                    // 16 ks + 2 t4 (+1, +8, +9)
                    float xa[2][4];
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int h = 16 * mt + g8 + 8 * r;
                        const float* qr = qv + h * QS + 16 * ks + 2 * t4;
                        const bool in = h < GV;
                        xa[r][0] = in ? qr[0] : 0.f;
                        xa[r][1] = in ? qr[1] : 0.f;
                        xa[r][2] = in ? qr[8] : 0.f;
                        xa[r][3] = in ? qr[9] : 0.f;
                    }
                    for (int part = 0; part < nparts; ++part) {
                        const uint32_t af[4] = {pack_bf16x2(xa[0][0], xa[0][1]), pack_bf16x2(xa[1][0], xa[1][1]),
                                                pack_bf16x2(xa[0][2], xa[0][3]), pack_bf16x2(xa[1][2], xa[1][3])};
                        mma_bf16f32(c[mt], af, b0, b1);
                        if (part + 1 < nparts) {
                            // the remainders for the next part
#pragma unroll
                            for (int r = 0; r < 2; ++r)
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    const uint32_t w2 = af[2 * e + r];
                                    xa[r][2 * e] -= __uint_as_float(w2 << 16);
                                    xa[r][2 * e + 1] -= __uint_as_float(w2 & 0xFFFF0000u);
                                }
                        }
                    }
                }
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int h = 16 * mt + g8 + 8 * r;
                    if (h < GV) {
                        sq[h * D + 8 * nt + 2 * t4] = c[mt][2 * r] * kq;
                        sq[h * D + 8 * nt + 2 * t4 + 1] = c[mt][2 * r + 1] * kq;
                    }
                }
        }
    }
    // a copy that never completed must land before the block exits
    if (!s_ok) mbar_wait(smem_u32(bar), 0, a.dp.err);
    __syncthreads();
    if (a.q_early) {
        pdl_wait();  // the store, before any write
        if (!a.prep_late_release) pdl_launch_dependents();
    }
    // per-head constants and operand scales (one warp per head)
    const DecodeGeom gm = a.gm;
    const float* kw = s_kw;
    float bmax = 0.f, bsum = 0.f;
    for (int p = 0; p < gm.npk; ++p) {
        bmax = fmaxf(bmax, fabsf(kw[1 + p]));
        bsum += kw[1 + p];
    }
    for (int h = warp; h < GV; h += nwarps) {
        // S q's sum, sum over j % 8 = 7 and max of |v| bit_weight(j % 8)
        float s_sq = 0.f, s_sq7 = 0.f, m_sq = 0.f;
        if (sq_tc) {
#pragma unroll
            for (int k = 0; k < D / 32; ++k) {
                const float v = sq[h * D + lane + 32 * k];  // j % 8 = lane % 8
                s_sq += v;
                m_sq = fmaxf(m_sq, fabsf(v) * fabsf(bit_weight(lane & 7)));
            }
            s_sq7 = warp_sum((lane & 7) == 7 ? s_sq : 0.f);
            s_sq = warp_sum(s_sq);
            m_sq = warp_max(m_sq);
        } else {
#pragma unroll
            for (int w = 0; w < kSqWarps; ++w) {
                s_sq += red_s[h][w][0];
                s_sq7 += red_s[h][w][1];
                m_sq = fmaxf(m_sq, red_s[h][w][2]);
            }
        }
        if (lane != 0) continue;
        const float s_rq = red_r[h][0], s_rq7 = red_r[h][1], m_rq = red_r[h][2] * bmax;
        m_sq *= 2.f;
        {
            // operand scales 2^e with 2^e m <= 224 (e4m3 holds up to 448): e is
            // the binary exponent of 224 / m, read from its float bits
            auto scale_exp = [](float m) {
                return m > 0.f ? (int)((__float_as_uint(224.f / m) >> 23) & 0xFF) - 127 : 0;
            };
            auto pow2 = [](int e) { return __uint_as_float((uint32_t)(127 + e) << 23); };
            const int ek = max(-120, min(120, scale_exp(m_rq))), eq = max(-120, min(120, scale_exp(m_sq)));
            float* c = a.ws_cst + hrow(h) * 4;
            c[0] = kw[0] * s_rq + 0.5f * bsum * s_rq7;
            c[1] = -s_sq + s_sq7;
            c[2] = pow2(-ek);
            c[3] = pow2(-eq);
            sig[2 * h] = pow2(ek);
            sig[2 * h + 1] = pow2(eq);
        }
    }
    __syncthreads();
    // score operand images: a work unit is (head group, head row block, plane,
    // tensor-memory column); it writes the kPieces words (4 K indices each) of
    // the rows kPieces*hl + piece, computing the pieces of each value in one pass
    const int kt = gm.npl * D;           // K extent (bytes per row)
    const uint32_t sbo = 8u * kt;        // byte step between 8-row groups
    const int hrows = (gm.n_cols + kPieces - 1) / kPieces;  // head row blocks (incl. padding)
    // a work unit is (entry, head group, 16-byte K chunk j, head row block hl,
    // fastest): the kPieces rows of head hl over K bytes 16j .. 16j + 15 are
    // 64 contiguous bytes of the image, and consecutive units fill whole lines
    const int nchunk = kt / 16;
    const int units = ne * gm.nhg * nchunk * hrows;
    for (int u = tid; u < units; u += blockDim.x) {
        int x = u;
        const int hl = x % hrows;
        x /= hrows;
        const int j = x % nchunk;
        x /= nchunk;
        const int hgi = x % gm.nhg, ent = x / gm.nhg;
        const int P = (16 * j) / D, col0 = ((16 * j) % D) / 4;
        uint32_t word[kPieces][4];
#pragma unroll
        for (int k = 0; k < kPieces; ++k)
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) word[k][cc] = 0;
        if (hl < gm.hc) {
            const int h = ent * G + hgi * gm.hc + hl;  // virtual head
            const bool sign_plane = P == gm.npk;
            const float beta = sign_plane ? 2.f : kw[1 + P];
            const float* src = sign_plane ? sq + h * D : rq + h * D;
            const float sc = sig[2 * h + (sign_plane ? 1 : 0)];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int col = col0 + cc;
                const float bw = bit_weight(col & 7);
                float y[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) y[e] = beta * src[32 * (col >> 3) + 8 * e + (col & 7)] * bw * sc;
                // the pieces of bytes (0, 1) and (2, 3) in packed conversions:
                // the same roundings as one value at a time
#pragma unroll
                for (int k = 0; k < kPieces; ++k) {
                    uint32_t w = 0;
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const __nv_fp8x2_storage_t pk =
                            __nv_cvt_float2_to_fp8x2(make_float2(y[e], y[e + 1]), __NV_SATFINITE, __NV_E4M3);
                        w |= (uint32_t)pk << (8 * e);
                        const float2 back = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pk, __NV_E4M3)));
                        y[e] = (y[e] - back.x) * 16.f;
                        y[e + 1] = (y[e + 1] - back.y) * 16.f;
                    }
                    word[k][cc] = w;
                }
            }
        }
        uint8_t* img = a.ws_bimg + (((int64_t)(b0 + ent) * a.heads + g) * gm.nhg + hgi) * gm.bimg_bytes;
#pragma unroll
        for (int k = 0; k < kPieces; ++k) {
            const int n = kPieces * hl + k;
            if (n < gm.n_cols)
                *reinterpret_cast<uint4*>(img + (n & 7) * 16 + (n >> 3) * sbo + j * 128) =
                    make_uint4(word[k][0], word[k][1], word[k][2], word[k][3]);
        }
    }
    if (a.prep_late_release) pdl_launch_dependents();
}

// ------------------------------------------------- extend: exact chunk part
// Extend attention's exact causal part at d = 128, written as the tail split
// partial of every new token.  A CTA takes 16 consecutive token rows t0.. of
// one KV head; warp w takes query head w (then w + warps, ...).  Token t's
// keys are rows tail_base[t] .. tail_base[t] + min(tail_len[t], tail_cap) - 1
// of the token-major new-token buffers.  Those key tiles (64 rows) are staged
// in shared memory once for all 16 rows and all heads:
//   S = Q K^T    bf16 tensor-core products, fp32 accumulation (an fp32 query
//                is split into bf16 high and low parts, two products)
//   P V          probabilities as fp16 high and low parts times the values
//                converted to fp16 (exact for bf16 values of normal
//                magnitude), fp32 accumulation
// with an online exp2 softmax per row.  MSE values leave in the rotated space
// (R acc = H D acc / sqrt(d), butterflies across the quad's lanes and the
// thread's registers), as the combine expects of every split.
constexpr int kChunkRows = 16;
constexpr int kChunkKeys = 64;
constexpr int kChunkMaxWarps = 8;

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// (x, y) as fp16 high parts and fp16 roundings of the remainders
__device__ __forceinline__ void split_f16x2(float x, float y, uint32_t& hi, uint32_t& lo) {
    const __half2 h = __floats2half2_rn(x, y);
    const float2 hf = __half22float2(h);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = pack_f16x2(x - hf.x, y - hf.y);
}

// bf16 pair (element c, c+1) of query row t, head hq: the high parts and,
// for an fp32 query, the low parts
__device__ __forceinline__ void chunk_q_pair(const DecodeArgs& a, int t, int hq, int c, uint32_t& hi, uint32_t& lo) {
    hi = lo = 0u;
    if (t >= a.batch) return;
    const int64_t off = ((int64_t)t * a.q_heads + hq) * 128 + c;
    if (a.q_dtype == TQ_DTYPE_BF16) {
        hi = *reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(a.q) + off);
    } else {
        const float2 x = *reinterpret_cast<const float2*>(static_cast<const float*>(a.q) + off);
        const __nv_bfloat162 h = __floats2bfloat162_rn(x.x, x.y);
        const float2 hf = __bfloat1622float2(h);
        const __nv_bfloat162 l = __floats2bfloat162_rn(x.x - hf.x, x.y - hf.y);
        hi = *reinterpret_cast<const uint32_t*>(&h);
        lo = *reinterpret_cast<const uint32_t*>(&l);
    }
}

__host__ __device__ constexpr size_t chunk_smem_bytes() {
    return (size_t)2 * kChunkKeys * (128 * 2 + 16) + 2 * kChunkRows * 4 + 16;
}

template <int D>
__global__ void __launch_bounds__(32 * kChunkMaxWarps) chunk_attn_kernel(DecodeArgs a) {
    static_assert(D == 128, "the chunk kernel holds a 128-wide output row in registers");
    // launched in plain stream order; the query prep after it (q_early) may
    // compute beside it and waits for it before its first write
    pdl_launch_dependents();
    constexpr int KP = D * 2 + 16;  // staged row pitch (bytes): conflict-free fragment loads
    constexpr int NKS = D / 16, NSB = kChunkKeys / 8, NOB = D / 8;
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t* ks = smem;                    // [kChunkKeys][KP] keys, bf16
    uint8_t* vs = smem + kChunkKeys * KP;  // [kChunkKeys][KP] values, fp16
    int* rlo = reinterpret_cast<int*>(vs + kChunkKeys * KP);
    int* rhi = rlo + kChunkRows;
    __shared__ int s_range[2];
    const int g = blockIdx.y, t0 = blockIdx.x * kChunkRows;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
    const int G = a.group, gr = lane >> 2, q4 = lane & 3;
    if (tid < kChunkRows) {
        const int t = t0 + tid;
        int lo = 0x7fffffff, hi = -1;
        if (t < a.batch) {
            int tl = a.tail_lens[t];
            if (tl > a.tail_cap) {
                if (g == 0) set_error(a.dp.err, TQ_DEVERR_TAIL);
                tl = a.tail_cap;
            }
            if (tl > 0) {
                lo = a.tail_base[t];
                hi = lo + tl - 1;
            }
        }
        rlo[tid] = lo;
        rhi[tid] = hi;
    }
    __syncthreads();
    if (tid == 0) {
        int lo = 0x7fffffff, hi = -1;
        for (int r = 0; r < kChunkRows; ++r) {
            lo = min(lo, rlo[r]);
            hi = max(hi, rhi[r]);
        }
        s_range[0] = lo;
        s_range[1] = hi;
    }
    __syncthreads();
    const int kmin = s_range[0], kmax = s_range[1];
    const float f = a.scale_log2e;
    const bool qf32 = a.q_dtype != TQ_DTYPE_BF16;
    const int lo0 = rlo[gr], hi0 = rhi[gr], lo1 = rlo[gr + 8], hi1 = rhi[gr + 8];
    for (int hb = 0; hb < G; hb += nwarps) {
        const int h = hb + warp;
        const bool active = h < G;
        const int hq = g * G + (active ? h : 0);
        uint32_t qh[NKS][4], ql[NKS][4];
#pragma unroll
        for (int k = 0; k < NKS; ++k) {
            const int c = 16 * k + 2 * q4;
            chunk_q_pair(a, active ? t0 + gr : a.batch, hq, c, qh[k][0], ql[k][0]);
            chunk_q_pair(a, active ? t0 + gr + 8 : a.batch, hq, c, qh[k][1], ql[k][1]);
            chunk_q_pair(a, active ? t0 + gr : a.batch, hq, c + 8, qh[k][2], ql[k][2]);
            chunk_q_pair(a, active ? t0 + gr + 8 : a.batch, hq, c + 8, qh[k][3], ql[k][3]);
        }
        float o[NOB][4];
#pragma unroll
        for (int n = 0; n < NOB; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        for (int k0 = kmin; k0 <= kmax; k0 += kChunkKeys) {
            __syncthreads();  // the previous tile is consumed
            for (int e = tid; e < kChunkKeys * (D / 8); e += blockDim.x) {
                const int row = e / (D / 8), c8 = e % (D / 8), k = k0 + row;
                uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = make_uint4(0u, 0u, 0u, 0u);
                if (k <= kmax) {
                    const int64_t off = ((int64_t)k * a.heads + g) * D + 8 * c8;
                    kv = __ldg(reinterpret_cast<const uint4*>(a.tail_k + off));
                    const uint4 vb = __ldg(reinterpret_cast<const uint4*>(a.tail_v + off));
                    const uint32_t w[4] = {vb.x, vb.y, vb.z, vb.w};
                    uint32_t hw[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        hw[i] = pack_f16x2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
                    vv = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                }
                *reinterpret_cast<uint4*>(ks + row * KP + 16 * c8) = kv;
                *reinterpret_cast<uint4*>(vs + row * KP + 16 * c8) = vv;
            }
            __syncthreads();
            if (!active) continue;
            float sc[NSB][4];
#pragma unroll
            for (int n = 0; n < NSB; ++n) {
                sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
                const uint8_t* krow = ks + (8 * n + gr) * KP + 4 * q4;
#pragma unroll
                for (int k = 0; k < NKS; ++k) {
                    const uint32_t b0 = *reinterpret_cast<const uint32_t*>(krow + 32 * k);
                    const uint32_t b1 = *reinterpret_cast<const uint32_t*>(krow + 32 * k + 16);
                    mma_bf16f32(sc[n], qh[k], b0, b1);
                    if (qf32) mma_bf16f32(sc[n], ql[k], b0, b1);
                }
            }
            // scale, causal mask, running maxima of the two rows
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int n = 0; n < NSB; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = k0 + 8 * n + 2 * q4 + (e & 1);
                    const bool ok = e < 2 ? (key >= lo0 && key <= hi0) : (key >= lo1 && key <= hi1);
                    const float v = ok ? sc[n][e] * f : -INFINITY;
                    sc[n][e] = v;
                    if (e < 2) mx0 = fmaxf(mx0, v);
                    else mx1 = fmaxf(mx1, v);
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
            const float al0 = m0 == -INFINITY ? 0.f : exp2f(m0 - n0);
            const float al1 = m1 == -INFINITY ? 0.f : exp2f(m1 - n1);
            m0 = n0;
            m1 = n1;
            l0 *= al0;
            l1 *= al1;
#pragma unroll
            for (int n = 0; n < NOB; ++n) {
                o[n][0] *= al0;
                o[n][1] *= al0;
                o[n][2] *= al1;
                o[n][3] *= al1;
            }
#pragma unroll
            for (int n = 0; n < NSB; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float mr = e < 2 ? n0 : n1;
                    const float p = sc[n][e] == -INFINITY ? 0.f : exp2f(sc[n][e] - mr);
                    sc[n][e] = p;
                    if (e < 2) l0 += p;
                    else l1 += p;
                }
            // O += P V: the score fragments of key blocks 2j, 2j+1 are the
            // A fragment of the j-th 16-key step; P goes in as an fp16 high
            // part and the fp16 rounding of its remainder (two products)
#pragma unroll
            for (int j = 0; j < kChunkKeys / 16; ++j) {
                uint32_t pa[4], pl[4];
                split_f16x2(sc[2 * j][0], sc[2 * j][1], pa[0], pl[0]);
                split_f16x2(sc[2 * j][2], sc[2 * j][3], pa[1], pl[1]);
                split_f16x2(sc[2 * j + 1][0], sc[2 * j + 1][1], pa[2], pl[2]);
                split_f16x2(sc[2 * j + 1][2], sc[2 * j + 1][3], pa[3], pl[3]);
                const uint8_t* v0 = vs + (16 * j + 2 * q4) * KP + 2 * gr;
#pragma unroll
                for (int n = 0; n < NOB; ++n) {
                    const uint8_t* vp = v0 + 16 * n;
                    const uint32_t b0 = (uint32_t)*reinterpret_cast<const uint16_t*>(vp) |
                                        ((uint32_t)*reinterpret_cast<const uint16_t*>(vp + KP) << 16);
                    const uint32_t b1 = (uint32_t)*reinterpret_cast<const uint16_t*>(vp + 8 * KP) |
                                        ((uint32_t)*reinterpret_cast<const uint16_t*>(vp + 9 * KP) << 16);
                    mma_f16(o[n], pa[0], pa[1], pa[2], pa[3], b0, b1);
                    mma_f16(o[n], pl[0], pl[1], pl[2], pl[3], b0, b1);
                }
            }
        }
        if (!active) continue;
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        if (a.lay.v_mode == TQ_V_MSE) {
            // R o = H D o / sqrt(d) on each row; column c = 8n + 2*q4 + (e & 1)
#pragma unroll
            for (int n = 0; n < NOB; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[n][e] *= a.dp.signs[8 * n + 2 * q4 + (e & 1)];
#pragma unroll
            for (int n = 0; n < NOB; ++n)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const float x = o[n][e], y = o[n][e + 1];
                    o[n][e] = x + y;
                    o[n][e + 1] = x - y;
                }
#pragma unroll
            for (int bit = 1; bit <= 2; bit <<= 1)
#pragma unroll
                for (int n = 0; n < NOB; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float x = o[n][e], other = __shfl_xor_sync(0xffffffffu, x, bit);
                        o[n][e] = (q4 & bit) ? other - x : x + other;
                    }
#pragma unroll
            for (int hbit = 1; hbit < NOB; hbit <<= 1)
#pragma unroll
                for (int n = 0; n < NOB; ++n)
                    if (!(n & hbit))
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float x = o[n][e], y = o[n + hbit][e];
                            o[n][e] = x + y;
                            o[n + hbit][e] = x - y;
                        }
            const float inv = rsqrtf((float)D);
#pragma unroll
            for (int n = 0; n < NOB; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[n][e] *= inv;
        }
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int t = t0 + gr + 8 * rr;
            if (t >= a.batch) continue;
            const int64_t idx = ((int64_t)t * a.q_heads + hq) * a.sp.n_splits + a.sp.n_chunks;
#pragma unroll
            for (int n = 0; n < NOB; ++n)
                *reinterpret_cast<float2*>(a.ws_acc + idx * D + 8 * n + 2 * q4) =
                    make_float2(o[n][2 * rr], o[n][2 * rr + 1]);
            if (q4 == 0) {
                a.ws_ml[idx * 2] = rr ? m1 : m0;
                a.ws_ml[idx * 2 + 1] = rr ? l1 : l0;
            }
        }
    }
}

// ----------------------------------------------------------- tail split
// Exact bf16 tail tokens on CUDA cores (scores by (token, head), values by
// coordinate); partial in the same form as the compressed splits.
template <int D>
__device__ void tail_split(const DecodeArgs& a, int g, int b, uint8_t* smem, int h0, int NH) {
    constexpr int kPerThread = D / 128;
    // query heads h0 .. h0 + NH - 1 of the group
    const int G = a.group, tid = threadIdx.x;
    const int chunk = a.sp.n_chunks;
    float* qs = reinterpret_cast<float*>(smem);  // [NH][D] = q * f
    float* pr = qs + NH * D;                     // [NH][kTile]
    float* sm_m = pr + NH * kTile;               // [NH]
    uint16_t* vst = reinterpret_cast<uint16_t*>(sm_m + kMaxG);  // [kTailV][D] staged values (bf16)
    // the query times f, read from the caller's queries (the same product
    // as the query prep's, which this kernel does not wait for)
    for (int e = tid; e < NH * D; e += blockDim.x) {
        const int64_t src = ((int64_t)b * a.q_heads + g * G + h0 + e / D) * D + e % D;
        qs[e] = (a.q_dtype == TQ_DTYPE_F32 ? static_cast<const float*>(a.q)[src]
                                           : bf16_bits_to_float(static_cast<const uint16_t*>(a.q)[src])) *
                a.scale_log2e;
    }
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
    // element offset of tail token i of (entry b, KV head g)
    const int64_t row0 = a.tail_base ? (int64_t)a.tail_base[b] : 0;
    auto tail_off = [&](int i) -> int64_t {
        return a.tail_base ? ((row0 + i) * a.heads + g) * D : (((int64_t)b * a.heads + g) * a.tail_cap + i) * D;
    };
    for (int tt = 0; tt < tl; tt += kTile) {
        const int n_tok = min(kTile, tl - tt);
        for (int e = tid; e < NH * kTile; e += blockDim.x) pr[e] = -INFINITY;
        __syncthreads();
        // a thread per token: one pass over its key row (16-byte loads) for
        // every head of the group
        for (int t = tid; t < n_tok; t += blockDim.x) {
            const uint4* krow = reinterpret_cast<const uint4*>(a.tail_k + tail_off(tt + t));
            float s[kMaxG];
#pragma unroll
            for (int h = 0; h < kMaxG; ++h) s[h] = 0.f;
            // (unrolled: the row's loads issue together)
#pragma unroll
            for (int i8 = 0; i8 < D / 8; ++i8) {
                const uint4 u = __ldg(krow + i8);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
                float kf[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    kf[2 * e] = __uint_as_float(w[e] << 16);
                    kf[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
                }
#pragma unroll
                for (int h = 0; h < kMaxG; ++h) {
                    if (h < NH) {
                        const float* qh = qs + h * D + 8 * i8;
#pragma unroll
                        for (int e = 0; e < 8; ++e) s[h] = fmaf(qh[e], kf[e], s[h]);
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < kMaxG; ++h)
                if (h < NH) pr[h * kTile + t] = s[h];
        }
        __syncthreads();
        {
            const int lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
            for (int h = warp; h < NH; h += nw) {
                float mx = -INFINITY;
                for (int t = lane; t < kTile; t += 32) mx = fmaxf(mx, pr[h * kTile + t]);
                mx = warp_max(mx);
                if (lane == 0) sm_m[h] = fmaxf(mx, m_run[h]);
            }
        }
        __syncthreads();
        for (int e = tid; e < NH * kTile; e += blockDim.x) {
            const float sv = pr[e];
            pr[e] = sv == -INFINITY ? 0.f : exp2f(sv - sm_m[e / kTile]);
        }
        __syncthreads();
        // (head loops unrolled to kMaxG with a guard keep the running
        // state in registers)
#pragma unroll
        for (int h = 0; h < kMaxG; ++h) {
            if (h >= NH) continue;
            const float m_new = sm_m[h];
            const float alpha = m_run[h] == -INFINITY ? 0.f : exp2f(m_run[h] - m_new);
            float psum = 0.f;
            for (int t = 0; t < n_tok; ++t) psum += pr[h * kTile + t];
            l_run[h] = l_run[h] * alpha + psum;
            m_run[h] = m_new;
#pragma unroll
            for (int p = 0; p < kPerThread; ++p) acc[h][p] *= alpha;
        }
        // values, a thread per coordinate, from kTailV-row chunks staged in
        // shared memory with 16-byte loads (one memory latency per chunk)
        for (int c0 = 0; c0 < n_tok; c0 += kTailV) {
            const int nc = min(kTailV, n_tok - c0);
            for (int e = tid; e < nc * (D / 8); e += blockDim.x) {
                const int t = e / (D / 8), c8 = e % (D / 8);
                reinterpret_cast<uint4*>(vst)[e] =
                    __ldg(reinterpret_cast<const uint4*>(a.tail_v + tail_off(tt + c0 + t)) + c8);
            }
            __syncthreads();
            if (tid < 128) {
#pragma unroll
                for (int p = 0; p < kPerThread; ++p) {
                    const int i = tid + 128 * p;
                    for (int t = 0; t < nc; ++t) {
                        const float v = bf16_bits_to_float(vst[t * D + i]);
#pragma unroll
                        for (int h = 0; h < kMaxG; ++h)
                            if (h < NH) acc[h][p] = fmaf(pr[h * kTile + c0 + t], v, acc[h][p]);
                    }
                }
            }
            __syncthreads();  // the staged rows are consumed
        }
    }
    // MSE values are combined in the rotated space: acc <- R acc = H D acc / sqrt(d)
    if (a.lay.v_mode == TQ_V_MSE) {
        float* buf = qs;
        __syncthreads();
        if (tid < 128)
#pragma unroll
            for (int h = 0; h < kMaxG; ++h)
                if (h < NH)
#pragma unroll
                    for (int p = 0; p < kPerThread; ++p)
                        buf[h * D + tid + 128 * p] = acc[h][p] * a.dp.signs[tid + 128 * p];
        __syncthreads();
        if (tid < 128)
#pragma unroll
            for (int h = 0; h < kMaxG; ++h)
                if (h < NH)
#pragma unroll
                    for (int p = 0; p < kPerThread; ++p) {
                        const int i = tid + 128 * p;
                        float s = 0.f;
                        for (int j = 0; j < D; ++j) s += (__popc(i & j) & 1) ? -buf[h * D + j] : buf[h * D + j];
                        acc[h][p] = s * rsqrtf((float)D);
                    }
    }
    if (tid < 128)
#pragma unroll
        for (int h = 0; h < kMaxG; ++h) {
            if (h >= NH) continue;
            const int64_t idx = ((int64_t)b * a.q_heads + g * G + h0 + h) * a.sp.n_splits + chunk;
#pragma unroll
            for (int p = 0; p < kPerThread; ++p) a.ws_acc[idx * D + tid + 128 * p] = acc[h][p];
            if (tid == 0) {
                a.ws_ml[idx * 2] = m_run[h];
                a.ws_ml[idx * 2 + 1] = l_run[h];
            }
        }
}

// -------------------------------------------------------------- split
// One CTA = one split (split_blocks pages) of one KV head for a head group of
// hc query heads; four warps walk the split in 128-token tiles (8 pages):
//   * the tile's pages arrive by bulk async copies into a ring of tiles
//   * thread t owns token t: it expands the token's key planes into fp8 score
//     operands in tensor-memory lane t (one AND per 4 coordinates)
//   * one thread issues the fp8 MMAs D[token][head, piece] += A * B^T against
//     the query operand image in shared memory (tcgen05, fp32 accumulators in
//     tensor memory); each thread reads its token's scores back
//   * online exp2 softmax per warp; the probabilities, times the group-32 scale
//     or the MSE norm and plane weight, go to a per-warp buffer as fp16 hi + lo
//   * each warp contracts the values of its two pages on fp16 tensor cores
//     (mma.sync); the token order inside the contraction is permuted so that a
//     B register is one buffer word holding tokens (t, t+8).
constexpr int kTilePages = 8;
constexpr int kTileTokens = kTilePages * kBlock;  // 128 = MMA M
constexpr int kTmemCols = 256;  // per CTA; two CTAs per SM share the 512 columns

// score accumulator columns (kPieces per head, whole multiples of 16) and the
// first A operand column (after both accumulators) for nth n-tiles of heads
__host__ __device__ constexpr int score_cols(int nth) { return (kPieces * 4 * nth + 15) / 16 * 16; }
__host__ __device__ constexpr int tmem_a_col(int nth) { return (2 * score_cols(nth) + 31) / 32 * 32; }

struct SplitLayout {
    size_t tile, ring, bimg, pbuf, cst, zsm, bars, tslot, total;
    int pls, pbuf_words;  // probability buffer: words per page, per warp
};

// nsets: probability operand sets (group-32: d/32 groups; MSE: value planes)
template <int D>
__host__ __device__ inline SplitLayout split_layout(int page_bytes, const DecodeGeom& gm, int nsets, int stages) {
    auto up = [](size_t x) { return (x + 127) & ~(size_t)127; };
    const int h4 = 4 * gm.nth;
    SplitLayout l;
    l.tile = up((size_t)kTilePages * page_bytes);
    l.pls = nsets * h4 * 24 + 16;
    l.pbuf_words = 2 * l.pls;
    size_t off = 0;
    l.ring = off;
    off = up(off + (size_t)stages * l.tile);
    l.bimg = off;
    off = up(off + (size_t)gm.bimg_bytes);
    l.pbuf = off;
    off = up(off + (size_t)kWarpsPerGroup * l.pbuf_words * 4);
    l.cst = off;
    off = up(off + (size_t)h4 * 4 * 4);
    l.zsm = off;
    off = up(off + (size_t)kWarpsPerGroup * h4 * (D / 32) * 4);
    l.bars = off;
    off = up(off + (size_t)(stages + 2) * 8);
    l.tslot = off;
    off = up(off + 4);
    l.total = off;
    return l;
}
// per-warp partials merged at the end, placed over the ring
template <int D>
__host__ __device__ constexpr size_t split_red_bytes(int h4) {
    return (size_t)kWarpsPerGroup * h4 * (D + 2) * 4;
}

template <int D, int KB, bool G32, int VB, int NTH>
__global__ void __launch_bounds__(128, 2) split_kernel(DecodeArgs a) {
    pdl_launch_dependents();
    pdl_wait();  // the query prep's results
    constexpr int NPK = 1 << (KB - 1);  // key code planes
    constexpr int NW = D / 32;          // 32-bit words of a plane row
    constexpr int NCOL = D / 4;         // tensor-memory columns of one plane
    constexpr int NMT = D / 16;         // value m-tiles (16 coordinates)
    constexpr int NPV = G32 ? 1 : (1 << (VB - 1));
    constexpr int NSET = G32 ? D / 32 : NPV;
    constexpr int NZ = G32 ? D / 32 : 1;
    constexpr int H4 = 4 * NTH;         // heads of the CTA, padded to whole n-tiles
    constexpr int NCOLS = score_cols(NTH);  // score accumulator columns (head, piece)
    constexpr int TA = tmem_a_col(NTH);     // first A operand column
    constexpr int PCH = (kTmemCols - TA) / NCOL;  // planes per tensor-memory chunk
    const DecodeGeom gm = a.gm;
    const int chunk = blockIdx.x, g = blockIdx.y / gm.nhg, hgi = blockIdx.y % gm.nhg, b = blockIdx.z;
    if (b >= a.batch) return;
    extern __shared__ __align__(16) uint8_t smem[];
    if (a.tail_cap > 0 && chunk == a.sp.n_chunks) {
        // all G heads of the tail in one CTA (extend's chunk kernel may have
        // written it already)
        if (hgi == 0 && !a.chunk_attn) tail_split<D>(a, g, b, smem, 0, a.group);
        return;
    }
    const Layout& L = a.lay;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const int hc = gm.hc, npl = gm.npl, S = a.stages;
    const bool qjl = L.k_qjl;
    const SplitLayout sl = split_layout<D>(L.page_bytes, gm, NSET, S);
    uint8_t* ring = smem + sl.ring;
    const uint8_t* bimg = smem + sl.bimg;
    uint32_t* pbw = reinterpret_cast<uint32_t*>(smem + sl.pbuf) + warp * sl.pbuf_words;
    float* cst = reinterpret_cast<float*>(smem + sl.cst);
    float* zsm = reinterpret_cast<float*>(smem + sl.zsm) + warp * H4 * (D / 32);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + sl.bars);  // [S] ring, [S] image, [S+1] MMA
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + sl.tslot);
    float* red = reinterpret_cast<float*>(smem + sl.ring);

    // this split's token range
    int len = a.seq_lens[b];
    if (len < 0 || len > a.max_blocks * kBlock) {
        if (tid == 0 && g == 0 && chunk == 0 && hgi == 0) set_error(a.dp.err, TQ_DEVERR_SEQLEN);
        len = max(0, min(len, a.max_blocks * kBlock));
    }
    const int t0 = chunk * a.split_blocks * kBlock;
    const int t1 = min(len, t0 + a.split_blocks * kBlock);
    const int n_pages = t1 > t0 ? (t1 - t0 + kBlock - 1) / kBlock : 0;
    const int n_tiles = (n_pages + kTilePages - 1) / kTilePages;

    for (int e = tid; e < H4 * 4; e += blockDim.x) {
        const int h = e >> 2;
        cst[e] = h < hc ? a.ws_cst[((int64_t)b * a.q_heads + g * a.group + hgi * hc + h) * 4 + (e & 3)] : 0.f;
    }
    for (int e = lane; e < sl.pbuf_words; e += 32) pbw[e] = 0u;
    // MSE values: with sigma_P = 1 - 2 u_P (+-1 operands, no constant offset to
    // cancel later), c = (alpha + sum_P beta_P / 2) - sum_P (beta_P / 2) sigma_P
    float v_dc = 0.f, v_beta[NPV];
    if constexpr (!G32) {
        v_dc = a.dp.v_walsh[0];
#pragma unroll
        for (int P = 0; P < NPV; ++P) {
            v_beta[P] = -0.5f * a.dp.v_walsh[1 + P];
            v_dc += 0.5f * a.dp.v_walsh[1 + P];
        }
    }

    const int32_t* btab = a.block_table + (int64_t)(a.row_of ? a.row_of[b] : b) * a.max_blocks + t0 / kBlock;
    if (tid == 0) {
        for (int i = 0; i < S + 2; ++i) mbar_init(smem_u32(&bars[i]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // (thread 0) bulk copies of tile i's pages into stage s; bad block ids are
    // flagged and not copied, their tokens are masked
    auto issue_tile = [&](int i, int s) {
        const int p0 = i * kTilePages, np = min(kTilePages, n_pages - p0);
        uint32_t bytes = 0;
        for (int j = 0; j < np; ++j) {
            const int blk = btab[p0 + j];
            if (blk >= 0 && blk < a.num_blocks)
                bytes += L.page_bytes;
            else
                set_error(a.dp.err, TQ_DEVERR_BLOCK);
        }
        const uint32_t bar = smem_u32(&bars[s]);
        mbar_expect_tx(bar, bytes);
        for (int j = 0; j < np; ++j) {
            const int blk = btab[p0 + j];
            if (blk >= 0 && blk < a.num_blocks)
                bulk_copy(smem_u32(ring + s * sl.tile + (size_t)j * L.page_bytes),
                          a.cache + ((int64_t)blk * a.heads + g) * L.page_bytes, L.page_bytes, bar);
        }
    };
    int issued = 0;  // tiles issued so far (thread 0)
    uint32_t tmem = 0;
    if (n_tiles > 0) {
        if (warp == 0) tmem_alloc(tslot, kTmemCols);
        if (tid == 0) {
            const uint32_t bb = smem_u32(&bars[S]);
            mbar_expect_tx(bb, gm.bimg_bytes);
            bulk_copy(smem_u32(bimg), a.ws_bimg + (((int64_t)b * a.heads + g) * gm.nhg + hgi) * gm.bimg_bytes,
                      gm.bimg_bytes, bb);
            for (; issued < S && issued < n_tiles; ++issued) issue_tile(issued, issued);
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        tmem = *tslot;
    }

    float m_ref[H4], l_part[H4], zacc[H4][NZ];
    float pv[NTH][NMT][4];
#pragma unroll
    for (int h = 0; h < H4; ++h) {
        m_ref[h] = -INFINITY;
        l_part[h] = 0.f;
#pragma unroll
        for (int z = 0; z < NZ; ++z) zacc[h][z] = 0.f;
    }
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt)
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) pv[nt][mt][0] = pv[nt][mt][1] = pv[nt][mt][2] = pv[nt][mt][3] = 0.f;

    bool ok = n_tiles > 0 ? mbar_wait(smem_u32(&bars[S]), 0, a.dp.err) : true;
    bool mma_ok = true;
    uint32_t ring_phase = 0, mma_phase = 0;
    int consumed = 0;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const uint32_t idesc = fp8_idesc(NCOLS);
    const uint32_t sbo = 8u * (uint32_t)(npl * D);
    const int pj = tid >> 4, r = tid & 15;  // this thread's page and row in the tile
    const int pl = pj & 1, pair = r & 7, hf = r >> 3;

    for (int i = 0; i < n_tiles; ++i) {
        const int s = i % S;
        ok = mbar_wait(smem_u32(&bars[s]), (ring_phase >> s) & 1, a.dp.err) && ok;
        ring_phase ^= 1u << s;
        consumed = i + 1;
        const int p0 = i * kTilePages, np = min(kTilePages, n_pages - p0);
        const uint8_t* tile = ring + s * sl.tile;
        const int pos = t0 + (p0 + pj) * kBlock + r;
        bool valid = pj < np && pos < t1;
        if (valid) {
            const int blk = btab[p0 + pj];
            valid = blk >= 0 && blk < a.num_blocks;
        }
        const uint8_t* pg = tile + pj * L.page_bytes;

        // ---------------- score operands of this token, chunks of planes
        uint32_t kw[KB][NW], sw[NW];
#pragma unroll
        for (int p = 0; p < KB; ++p)
#pragma unroll
            for (int w4 = 0; w4 < NW; w4 += 4) {
                const uint4 u = *reinterpret_cast<const uint4*>(pg + L.k_codes + (p * kBlock + r) * (D / 8) + 4 * w4);
                kw[p][w4] = u.x;
                kw[p][w4 + 1] = u.y;
                kw[p][w4 + 2] = u.z;
                kw[p][w4 + 3] = u.w;
            }
#pragma unroll
        for (int w4 = 0; w4 < NW; w4 += 4) {
            uint4 u = make_uint4(0u, 0u, 0u, 0u);
            if (qjl) u = *reinterpret_cast<const uint4*>(pg + L.k_signs + r * (D / 8) + 4 * w4);
            sw[w4] = u.x;
            sw[w4 + 1] = u.y;
            sw[w4 + 2] = u.z;
            sw[w4 + 3] = u.w;
        }
        bool stop = false;
        for (int c0 = 0; c0 < npl; c0 += PCH) {
            const int c1 = min(npl, c0 + PCH);
#pragma unroll
            for (int P = 0; P <= NPK; ++P) {
                if (P < c0 || P >= c1) continue;
                uint32_t wv[NW];
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    uint32_t x = 0;
                    if (P < NPK) {
#pragma unroll
                        for (int p = 0; p < KB; ++p)
                            if ((plane_subset(KB, P) >> p) & 1) x ^= kw[p][w];
                    } else {
                        x = sw[w];
                    }
                    wv[w] = x;
                }
#pragma unroll
                for (int q = 0; q < NW / 4; ++q) {
                    // the empty volatile asm orders this chunk after the previous
                    // store, so that only 32 operand registers are live at a time
                    asm volatile("" : "+r"(wv[4 * q]), "+r"(wv[4 * q + 1]), "+r"(wv[4 * q + 2]), "+r"(wv[4 * q + 3]));
                    uint32_t a32[32];
#pragma unroll
                    for (int w4 = 0; w4 < 4; ++w4) {
                        const uint32_t x = wv[4 * q + w4];
                        a32[8 * w4 + 0] = bit_operand<0>(x);
                        a32[8 * w4 + 1] = bit_operand<1>(x);
                        a32[8 * w4 + 2] = bit_operand<2>(x);
                        a32[8 * w4 + 3] = bit_operand<3>(x);
                        a32[8 * w4 + 4] = bit_operand<4>(x);
                        a32[8 * w4 + 5] = bit_operand<5>(x);
                        a32[8 * w4 + 6] = bit_operand<6>(x);
                        a32[8 * w4 + 7] = bit_operand<7>(x);
                    }
                    tmem_st32(tmem + lane_base + TA + (P - c0) * NCOL + 32 * q, a32);
                }
            }
            tc_wait_st();
            tc_fence_before();
            const bool all_ok = __syncthreads_and(ok && mma_ok);
            tc_fence_after();
            if (!all_ok) {
                stop = true;
                break;
            }
            if (tid == 0) {
                // every warp is past tile i-1: its stage takes the next tile
                if (c0 == 0 && i >= 1 && issued < n_tiles) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue_tile(issued, (i - 1) % S);
                    ++issued;
                }
                for (int P = c0; P < c1; ++P)
                    for (int kb = 0; kb < NW; ++kb) {
                        const uint32_t d_addr = tmem + (P < NPK ? 0u : (uint32_t)NCOLS);
                        const uint32_t a_addr = tmem + TA + (P - c0) * NCOL + 8 * kb;
                        const uint64_t bd = smem_desc(smem_u32(bimg) + (P * (D / 16) + 2 * kb) * 128, 128, sbo);
                        const uint32_t acc = P < NPK ? (P > 0 || kb > 0) : (kb > 0);
                        mma_fp8_ts(d_addr, a_addr, bd, idesc, acc);
                    }
                tc_commit(smem_u32(&bars[S + 1]));
            }
            mma_ok = mbar_wait(smem_u32(&bars[S + 1]), mma_phase, a.dp.err);
            mma_phase ^= 1;
            tc_fence_after();
        }
        if (stop) break;

        // ---------------- scores of this token (log2 units)
        const float n16 = __half2float(*reinterpret_cast<const __half*>(pg + L.k_norm + 2 * r));
        const float rho = qjl ? __half2float(*reinterpret_cast<const __half*>(pg + L.k_rnorm + 2 * r)) : 0.f;
        float sc[H4];
        {
            uint32_t acc[NCOLS];
            float sk[H4];
#pragma unroll
            for (int q = 0; q < NCOLS / 16; ++q) tmem_ld16(tmem + lane_base + 16 * q, *reinterpret_cast<uint32_t(*)[16]>(&acc[16 * q]));
            tc_wait_ld();
#pragma unroll
            for (int h = 0; h < H4; ++h) sk[h] = piece_sum(&acc[kPieces * h]);
            if (qjl) {
#pragma unroll
                for (int q = 0; q < NCOLS / 16; ++q)
                    tmem_ld16(tmem + lane_base + NCOLS + 16 * q, *reinterpret_cast<uint32_t(*)[16]>(&acc[16 * q]));
                tc_wait_ld();
            }
#pragma unroll
            for (int h = 0; h < H4; ++h) {
                float v = n16 * (cst[4 * h] + sk[h] * cst[4 * h + 2]);
                if (qjl) v += rho * (cst[4 * h + 1] + piece_sum(&acc[kPieces * h]) * cst[4 * h + 3]);
                sc[h] = (valid && h < hc) ? v : -INFINITY;
            }
        }

        // ---------------- online softmax per warp: m_ref is a reference
        // maximum that moves (with a rescale) only when a score passes it by
        // more than kRescaleSlack
        float p[H4];
#pragma unroll
        for (int h = 0; h < H4; ++h) {
            const bool mv = sc[h] > m_ref[h] + kRescaleSlack;
            if (__any_sync(0xffffffffu, mv)) {
                const float mx = warp_max(sc[h]);
                const float alpha = m_ref[h] == -INFINITY ? 0.f : fast_exp2(m_ref[h] - mx);
                l_part[h] *= alpha;
#pragma unroll
                for (int z = 0; z < NZ; ++z) zacc[h][z] *= alpha;
                // value accumulators: thread (gq, tq) of n-tile nt holds head 4 nt + tq
                if (tq == (h & 3)) {
#pragma unroll
                    for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) pv[h >> 2][mt][e] *= alpha;
                }
                m_ref[h] = mx;
            }
            p[h] = sc[h] == -INFINITY ? 0.f : fast_exp2(sc[h] - m_ref[h]);
            l_part[h] += p[h];
        }

        // ---------------- probability operands: word (set, head, pair, piece)
        // of page pl holds tokens (pair, pair + 8) as fp16 halves
        {
            __half* pb = reinterpret_cast<__half*>(pbw + pl * sl.pls) + hf;
            auto put = [&](int set, int h, float x) {
                const __half hi = __float2half_rn(x);
                const __half lo = __float2half_rn(x - __half2float(hi));
                const int wd = (set * H4 + h) * 24 + pair * 2;
                pb[2 * wd] = hi;
                pb[2 * wd + 2] = lo;
            };
            if constexpr (G32) {
                constexpr int MW = D / 32;  // {fp16 scale, fp16 zero} per group
                uint32_t mw[MW];
#pragma unroll
                for (int w4 = 0; w4 < MW; w4 += 4) {
                    const uint4 u = *reinterpret_cast<const uint4*>(pg + L.v_meta + r * L.v_meta_row + 4 * w4);
                    mw[w4] = u.x;
                    mw[w4 + 1] = u.y;
                    mw[w4 + 2] = u.z;
                    mw[w4 + 3] = u.w;
                }
#pragma unroll
                for (int gr = 0; gr < MW; ++gr) {
                    const float2 sz = __half22float2(*reinterpret_cast<const __half2*>(&mw[gr]));
                    const float sv = valid ? sz.x : 0.f, zv = valid ? sz.y : 0.f;
#pragma unroll
                    for (int h = 0; h < H4; ++h) {
                        if (h < hc) put(gr, h, p[h] * sv);
                        zacc[h][gr] = fmaf(p[h], zv, zacc[h][gr]);
                    }
                }
            } else {
                const float nv = valid ? __half2float(*reinterpret_cast<const __half*>(pg + L.v_meta + 2 * r)) : 0.f;
#pragma unroll
                for (int h = 0; h < H4; ++h) {
                    const float pn = p[h] * nv;
                    if (h < hc)
#pragma unroll
                        for (int P = 0; P < NPV; ++P) put(P, h, pn * v_beta[P]);
                    zacc[h][0] = fmaf(v_dc, pn, zacc[h][0]);
                }
            }
        }
        __syncwarp();

        // ---------------- values of this warp's two pages
#pragma unroll
        for (int pl2 = 0; pl2 < 2; ++pl2) {
            const int pjw = 2 * warp + pl2;
            if (pjw >= np) break;
            const uint8_t* pgw = tile + pjw * L.page_bytes;
            const uint32_t* pbr = pbw + pl2 * sl.pls + (gq >> 1) * 24 + (gq & 1) + 2 * tq;  // + (set*H4 + 4 nt)*24
            if constexpr (G32) {
                constexpr int TB = D * VB / 64;  // bytes of a token row per thread role
                constexpr int TW = TB / 4;
                uint32_t va[TW], vb2[TW], vc[TW], vd[TW];
                const uint8_t* vrow = pgw + L.v_codes + TB * gq;
#pragma unroll
                for (int w = 0; w < TW; ++w) {
                    va[w] = *reinterpret_cast<const uint32_t*>(vrow + tq * L.v_code_row + 4 * w);
                    vb2[w] = *reinterpret_cast<const uint32_t*>(vrow + (tq + 8) * L.v_code_row + 4 * w);
                    vc[w] = *reinterpret_cast<const uint32_t*>(vrow + (tq + 4) * L.v_code_row + 4 * w);
                    vd[w] = *reinterpret_cast<const uint32_t*>(vrow + (tq + 12) * L.v_code_row + 4 * w);
                }
#pragma unroll
                for (int mt = 0; mt < NMT; ++mt) {
                    const int gr = mt >> 1;
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
#pragma unroll
                    for (int nt = 0; nt < NTH; ++nt) {
                        const uint32_t* bp = pbr + (gr * H4 + 4 * nt) * 24;
                        mma_f16(pv[nt][mt], a0, a1, a2, a3, bp[0], bp[8]);
                    }
                }
            } else {
                // value bit-planes: thread role gq owns coordinates (D/8)*gq ... + D/8 - 1
                constexpr int CB = D / 64;  // bytes of a plane row per thread role (2 or 4)
                uint32_t wlo[VB][2], whi[VB][2];  // token pairs (tq, tq+8) and (tq+4, tq+12)
#pragma unroll
                for (int pp = 0; pp < VB; ++pp) {
                    const uint8_t* base = pgw + L.v_codes + pp * kBlock * (D / 8) + CB * gq;
                    if constexpr (CB == 2) {
                        const uint32_t ra = *reinterpret_cast<const uint16_t*>(base + tq * (D / 8));
                        const uint32_t rb = *reinterpret_cast<const uint16_t*>(base + (tq + 8) * (D / 8));
                        const uint32_t rc = *reinterpret_cast<const uint16_t*>(base + (tq + 4) * (D / 8));
                        const uint32_t rd = *reinterpret_cast<const uint16_t*>(base + (tq + 12) * (D / 8));
                        wlo[pp][0] = ra | (rb << 16);
                        whi[pp][0] = rc | (rd << 16);
                        wlo[pp][1] = whi[pp][1] = 0;
                    } else {
                        const uint32_t ra = *reinterpret_cast<const uint32_t*>(base + tq * (D / 8));
                        const uint32_t rb = *reinterpret_cast<const uint32_t*>(base + (tq + 8) * (D / 8));
                        const uint32_t rc = *reinterpret_cast<const uint32_t*>(base + (tq + 4) * (D / 8));
                        const uint32_t rd = *reinterpret_cast<const uint32_t*>(base + (tq + 12) * (D / 8));
                        wlo[pp][0] = (ra & 0xFFFFu) | (rb << 16);
                        wlo[pp][1] = (ra >> 16) | (rb & 0xFFFF0000u);
                        whi[pp][0] = (rc & 0xFFFFu) | (rd << 16);
                        whi[pp][1] = (rc >> 16) | (rd & 0xFFFF0000u);
                    }
                }
#pragma unroll
                for (int P = 0; P < NPV; ++P) {
                    uint32_t ul[2] = {0, 0}, uh[2] = {0, 0};
#pragma unroll
                    for (int pp = 0; pp < VB; ++pp)
                        if ((plane_subset(VB, P) >> pp) & 1) {
                            ul[0] ^= wlo[pp][0];
                            ul[1] ^= wlo[pp][1];
                            uh[0] ^= whi[pp][0];
                            uh[1] ^= whi[pp][1];
                        }
#pragma unroll
                    for (int mt = 0; mt < NMT; ++mt) {
                        // bit k of each half moved to the fp16 sign: 1.0 or -1.0
                        const int wsel = mt >> 3, sh = 2 * (mt & 7);
                        const uint32_t a0 = ((ul[wsel] << (15 - sh)) & 0x80008000u) | 0x3C003C00u;
                        const uint32_t a1 = ((ul[wsel] << (14 - sh)) & 0x80008000u) | 0x3C003C00u;
                        const uint32_t a2 = ((uh[wsel] << (15 - sh)) & 0x80008000u) | 0x3C003C00u;
                        const uint32_t a3 = ((uh[wsel] << (14 - sh)) & 0x80008000u) | 0x3C003C00u;
#pragma unroll
                        for (int nt = 0; nt < NTH; ++nt) {
                            const uint32_t* bp = pbr + (P * H4 + 4 * nt) * 24;
                            mma_f16(pv[nt][mt], a0, a1, a2, a3, bp[0], bp[8]);
                        }
                    }
                }
            }
        }
        __syncwarp();
    }
    // copies issued but not consumed (a wait gave up) must land before the
    // shared memory is released
    if (tid == 0)
        for (int t = consumed; t < issued; ++t) {
            const int s = t % S;
            mbar_wait(smem_u32(&bars[s]), (ring_phase >> s) & 1, a.dp.err);
            ring_phase ^= 1u << s;
        }
    if (!mma_ok) mbar_wait(smem_u32(&bars[S + 1]), mma_phase ^ 1, a.dp.err);
    tc_fence_before();
    __syncthreads();
    if (n_tiles > 0 && warp == 0) tmem_dealloc(tmem, kTmemCols);

    // ---------------- per-warp partials -> shared memory -> merged split partial
#pragma unroll
    for (int h = 0; h < H4; ++h) {
        l_part[h] = warp_sum(l_part[h]);
#pragma unroll
        for (int z = 0; z < NZ; ++z) zacc[h][z] = warp_sum(zacc[h][z]);
    }
    if (lane == 0)
#pragma unroll
        for (int h = 0; h < H4; ++h) {
#pragma unroll
            for (int z = 0; z < NZ; ++z) zsm[h * NZ + z] = zacc[h][z];
            red[(warp * H4 + h) * (D + 2) + D] = m_ref[h];
            red[(warp * H4 + h) * (D + 2) + D + 1] = l_part[h];
        }
    __syncwarp();
#pragma unroll
    for (int nt = 0; nt < NTH; ++nt) {
        const int head = 4 * nt + tq;
        float* my = red + (warp * H4 + head) * (D + 2);
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) {
            float v0v = pv[nt][mt][0] + pv[nt][mt][1], v1v = pv[nt][mt][2] + pv[nt][mt][3];
            int c0;
            if constexpr (G32) {
                // operand scales: 4-bit q*2^-24 (even slot), q*2^-20 (odd slot);
                // 2-bit q*2^(4(mt%2)-24), q*2^(4(mt%2)-22)
                const float s0 = VB == 4 ? 16777216.f : ((mt & 1) ? 1048576.f : 16777216.f);
                const float s1 = VB == 4 ? 1048576.f : ((mt & 1) ? 262144.f : 4194304.f);
                const float zv = zsm[head * NZ + (mt >> 1)];
                c0 = 32 * (mt >> 1) + 4 * gq + 2 * (mt & 1);
                v0v = fmaf(v0v, s0, zv);
                v1v = fmaf(v1v, s1, zv);
            } else {
                const float zv = zsm[head * NZ];
                c0 = (D / 8) * gq + 2 * mt;
                v0v += zv;
                v1v += zv;
            }
            my[c0] = v0v;
            my[c0 + 1] = v1v;
        }
    }
    __syncthreads();
    // merge the four warps; write (m, l, acc) of this split
    for (int e = threadIdx.x; e < hc * D; e += blockDim.x) {
        const int h = e / D, i = e % D;
        float M = -INFINITY;
        for (int w = 0; w < kWarpsPerGroup; ++w) M = fmaxf(M, red[(w * H4 + h) * (D + 2) + D]);
        float acc = 0.f, l = 0.f;
        for (int w = 0; w < kWarpsPerGroup; ++w) {
            const float* rr = red + (w * H4 + h) * (D + 2);
            if (rr[D] == -INFINITY) continue;
            const float wt = exp2f(rr[D] - M);
            acc = fmaf(wt, rr[i], acc);
            l = fmaf(wt, rr[D + 1], l);
        }
        const int64_t idx = ((int64_t)b * a.q_heads + g * a.group + hgi * hc + h) * a.sp.n_splits + chunk;
        a.ws_acc[idx * D + i] = acc;
        if (i == 0) {
            a.ws_ml[idx * 2] = M;
            a.ws_ml[idx * 2 + 1] = l;
        }
    }
}

// --------------------------------------------------------------- combine
// kPre: splits whose partials load beside the (m, l) pairs (8 when a row has
// at most 8 splits: fewer registers, more CTAs per SM; else 32)
template <int D, int kPre>
__global__ void __launch_bounds__(128) combine_kernel(DecodeArgs a) {
    pdl_launch_dependents();
    pdl_wait();  // the split partials
    constexpr int kPerThread = D / 128;
    const int h = blockIdx.x, b = blockIdx.y;
    if (b >= a.batch) return;
    const int S = a.sp.n_splits;
    const int64_t base = ((int64_t)b * a.q_heads + h) * S;
    __shared__ float o[D];
    __shared__ float red[2][4];
    extern __shared__ float wgt[];  // [S] split weights 2^(m_s - M)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the first kPre splits' partials load now, beside the (m, l) pairs,
    // instead of after the two reductions below
    const float* src = a.ws_acc + base * D + tid;
    float pre[kPre][kPerThread];
#pragma unroll
    for (int s = 0; s < kPre; ++s)
#pragma unroll
        for (int p = 0; p < kPerThread; ++p) pre[s][p] = s < S ? src[(int64_t)s * D + 128 * p] : 0.f;
    // every split's (m, l) at once; M = max m.  Compressed splits past the
    // sequence's length are empty and need not have been written.
    const int len = max(0, min(a.seq_lens[b], a.max_blocks * kBlock));
    const int nch = (len + a.split_blocks * kBlock - 1) / (a.split_blocks * kBlock);
    float lsum;
    float acc[kPerThread];
#pragma unroll
    for (int p = 0; p < kPerThread; ++p) acc[p] = 0.f;
    if (S <= 32) {
        // one split per lane: every warp finds M, the weights and their sum
        // itself, with no barrier (the same arithmetic as below)
        float m = -INFINITY, l = 0.f;
        if (lane < S && !(lane < a.sp.n_chunks && lane >= nch)) {
            m = a.ws_ml[(base + lane) * 2];
            l = a.ws_ml[(base + lane) * 2 + 1];
        }
        const float M = warp_max(m);
        const float w = (m == -INFINITY || M == -INFINITY) ? 0.f : exp2f(m - M);  // empty split: 0
        lsum = warp_sum(w > 0.f ? fmaf(w, l, 0.f) : 0.f);
        // an empty split (weight 0) may leave its partial unwritten: skip it
#pragma unroll
        for (int s = 0; s < kPre; ++s) {
            const float ws = __shfl_sync(0xffffffffu, w, s);
#pragma unroll
            for (int p = 0; p < kPerThread; ++p) acc[p] = ws > 0.f ? fmaf(ws, pre[s][p], acc[p]) : acc[p];
        }
        for (int s = kPre; s < S; ++s) {
            const float ws = __shfl_sync(0xffffffffu, w, s);
#pragma unroll
            for (int p = 0; p < kPerThread; ++p)
                if (ws > 0.f) acc[p] = fmaf(ws, src[(int64_t)s * D + 128 * p], acc[p]);
        }
    } else {
        float M = -INFINITY;
        for (int s = tid; s < S; s += 128) {
            const float m = (s < a.sp.n_chunks && s >= nch) ? -INFINITY : a.ws_ml[(base + s) * 2];
            wgt[s] = m;
            M = fmaxf(M, m);
        }
        M = warp_max(M);
        if (lane == 0) red[0][warp] = M;
        __syncthreads();
        M = fmaxf(fmaxf(red[0][0], red[0][1]), fmaxf(red[0][2], red[0][3]));
        float lpart = 0.f;
        for (int s = tid; s < S; s += 128) {
            const float m = wgt[s];
            const float w = (m == -INFINITY || M == -INFINITY) ? 0.f : exp2f(m - M);  // empty split: 0
            wgt[s] = w;
            if (w > 0.f) lpart = fmaf(w, a.ws_ml[(base + s) * 2 + 1], lpart);
        }
        lpart = warp_sum(lpart);
        if (lane == 0) red[1][warp] = lpart;
        __syncthreads();
        lsum = (red[1][0] + red[1][1]) + (red[1][2] + red[1][3]);
        // an empty split (weight 0) may leave its partial unwritten: skip it
#pragma unroll
        for (int s = 0; s < kPre; ++s) {
            const float w = wgt[s];
#pragma unroll
            for (int p = 0; p < kPerThread; ++p) acc[p] = w > 0.f ? fmaf(w, pre[s][p], acc[p]) : acc[p];
        }
#pragma unroll 8
        for (int s = kPre; s < S; ++s) {
            const float w = wgt[s];
#pragma unroll
            for (int p = 0; p < kPerThread; ++p) {
                const float v = src[(int64_t)s * D + 128 * p];
                acc[p] = w > 0.f ? fmaf(w, v, acc[p]) : acc[p];
            }
        }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
    for (int p = 0; p < kPerThread; ++p) o[threadIdx.x + 128 * p] = acc[p] * inv;
    __syncthreads();
    const int64_t ob = ((int64_t)b * a.q_heads + h) * D;
    if (a.lay.v_mode == TQ_V_MSE && !a.out_rotated) {
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
template <int D, int KB, bool G32, int VB, int NTH>
inline tq_status launch_split(const DecodeArgs& a, cudaStream_t s, size_t smem) {
    auto kern = split_kernel<D, KB, G32, VB, NTH>;
    {
        const tq_status fs = ensure_dynamic_smem((const void*)kern, 227 * 1024, "split_kernel");
        if (fs != TQ_OK) return fs;
    }
    {
        const cudaError_t e =
            launch_pdl(a.pdl, kern, dim3(a.sp.n_splits, a.heads * a.gm.nhg, a.batch), dim3(32 * kWarpsPerGroup), smem,
                       s, a);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return cuda_status(cudaGetLastError());
}

template <int D, int KB, int NTH>
inline tq_status dispatch_v(const DecodeArgs& a, cudaStream_t s, size_t smem) {
    if (a.lay.v_mode == TQ_V_G32)
        return a.lay.v_bits == 4 ? launch_split<D, KB, true, 4, NTH>(a, s, smem)
                                 : launch_split<D, KB, true, 2, NTH>(a, s, smem);
    switch (a.lay.v_bits) {
        case 2: return launch_split<D, KB, false, 2, NTH>(a, s, smem);
        case 3: return launch_split<D, KB, false, 3, NTH>(a, s, smem);
        default: return launch_split<D, KB, false, 4, NTH>(a, s, smem);
    }
}

template <int D, int KB>
inline tq_status dispatch_nth(const DecodeArgs& a, cudaStream_t s, size_t smem) {
    if constexpr (D == 128)
        if (a.gm.nth == 2) return dispatch_v<D, KB, 2>(a, s, smem);
    return dispatch_v<D, KB, 1>(a, s, smem);
}

// split-kernel launch for one (head dim, key bits); each pair is compiled in
// its own translation unit.  grid > 0: the warp-specialized persistent kernel
// (tq_decode_ws.cuh) on `grid` CTAs; grid == 0: split_kernel.
template <int D, int KB>
tq_status dispatch_split(const DecodeArgs& a, cudaStream_t s, size_t smem, int grid);

// Ring depth and dynamic shared memory of the split launch: the deepest ring
// (4..2 tiles) that keeps two CTAs per SM, else the deepest that fits one.
// At least 80 KB is requested so that no third CTA competes for tensor memory.
template <int D>
inline tq_status split_config(const DecodeArgs& a, int* stages, size_t* smem) {
    const int nsets = a.lay.v_mode == TQ_V_G32 ? D / 32 : (1 << (a.lay.v_bits - 1));
    const size_t tail_smem = tail_smem_bytes<D>(a.group);
    const size_t limits[2] = {112 * 1024, 226 * 1024};
    for (size_t lim : limits)
        for (int st = 4; st >= 2; --st) {
            const SplitLayout sl = split_layout<D>(a.lay.page_bytes, a.gm, nsets, st);
            size_t need = std::max(sl.total, a.tail_cap > 0 ? tail_smem : (size_t)0);
            if (need > lim || (size_t)st * sl.tile < split_red_bytes<D>(4 * a.gm.nth)) continue;
            *stages = st;
            *smem = std::max(need, (size_t)80 * 1024);
            return TQ_OK;
        }
    return TQ_ERR_UNSUPPORTED;
}

// prep -> split (optionally bracketed by profiling events) -> combine on the
// caller's stream.  Defined in tq_decode.cu, the one translation unit that
// instantiates the prep and combine kernels.
tq_status launch_decode(const DecodeArgs& a, cudaStream_t s, void* ev0, void* ev1);

// The argument checks of tq_decode_attention (TQ_ERR_INVALID_ARG or
// TQ_ERR_MISALIGNED, launching nothing) and the DecodeArgs they describe, with
// the scratch pointers of the handle's workspace.  Defined in tq_decode.cu; the
// allocation-free entry point uses it too and then points the scratch
// elsewhere.
tq_status decode_args(const tq_cache* c, const void* q, int q_dtype, const void* cache_buf,
                      const int32_t* block_table, const int32_t* seq_lens, const void* tail_k, const void* tail_v,
                      const int32_t* tail_lens, float scale, int batch, void* out, int out_dtype, DecodeArgs* a);

}  // namespace tq
