// Fused TurboQuant KV-cache store: norm, rotation, Lloyd-Max codes, key
// residual + QJL signs, value codes, bit packing and the scattered write into
// the paged cache, in one launch ([Roadmap] §3.1 "rotation fused into the
// quantise kernel"; [Paged] "Which path vLLM takes": the store kernel
// quantises, packs and writes the paged KV cache).
//
// One warp encodes one (token, KV head) vector at a time; lane l holds
// coordinates l + 32k.  In bulk the QJL projection S r of eight vectors at a
// time runs on tensor cores (mma.sync bf16, S as the A operand from shared
// memory); for a few vectors, on CUDA cores from S rows in L2.

#include <algorithm>
#include <atomic>
#include <type_traits>

#include "tq_store.cuh"

namespace tq {



// Pack codes[0..d) (one byte each, b bits used) into the row's LSB-first
// bitstream; lanes write whole 32-bit words.
__device__ __forceinline__ void pack_row(const uint8_t* codes, int d, int b, uint8_t* dst, int lane) {
    const int words = d * b / 32;
    for (int w = lane; w < words; w += 32) {
        const int bit0 = w * 32;
        uint32_t word = 0;
        for (int i = bit0 / b; i * b < bit0 + 32; ++i) {
            const int sh = i * b - bit0;
            const uint32_t c = codes[i];
            word |= sh >= 0 ? (c << sh) : (c >> -sh);
        }
        reinterpret_cast<uint32_t*>(dst)[w] = word;
    }
}

// Bit-sliced code planes: plane p, bit c of the row = bit p of the code of
// coordinate c.  Lane l holds coordinates l + 32k, so word k of a plane row is
// one warp ballot.
template <int D>
__device__ __forceinline__ void write_bit_planes(const int (&idx)[D / 32], int bits, uint8_t* planes, int row,
                                                 int lane) {
    for (int p = 0; p < bits; ++p) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(planes + (p * kBlock + row) * (D / 8));
#pragma unroll
        for (int k = 0; k < D / 32; ++k) {
            const uint32_t word = __ballot_sync(0xffffffffu, (idx[k] >> p) & 1);
            if (lane == k) dst[k] = word;
        }
    }
}

// Group-32 value field slot of coordinate c: group gr = c/32, offset o = c%32
// -> slot (D/8)*(o/4) + 2*(2*gr + (o%4)/2) + o%2 (inverse of the slot map in
// the page layout).
template <int D>
__device__ __forceinline__ int g32_slot(int c) {
    const int gr = c >> 5, o = c & 31;
    return (D / 8) * (o >> 2) + 2 * (2 * gr + ((o & 3) >> 1)) + (o & 1);
}

// TurboQuant-MSE code of one vector ([Explainer] steps 1-2): returns the fp32
// norm; idx[k] is the code of coordinate lane + 32k.
template <int D>
__device__ __forceinline__ float mse_codes(const float (&v)[D / 32], const float* signs, const float* bound, int nb,
                                           int lane, int (&idx)[D / 32]) {
    constexpr int PER = D / 32;
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < PER; ++k) ss = fmaf(v[k], v[k], ss);
    const float n = sqrtf(warp_sum(ss));
    float y[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) y[k] = v[k] * signs[lane + 32 * k];
    fwht_warp<PER>(y, lane);
    // y = H D v / (n sqrt(d)); a zero vector maps to y = 0
    const float inv = n > 0.f ? rsqrtf((float)D) / n : 0.f;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const float yk = y[k] * inv;
        // number of boundaries strictly below yk: a binary search over the
        // sorted boundaries (nb = 2^b - 1, b steps)
        int c = 0;
        for (int step = (nb + 1) >> 1; step > 0; step >>= 1)
            if (yk > bound[c + step - 1]) c += step;
        idx[k] = c;
    }
    return n;
}

// Bulk store (bulk appends): each warp encodes its vectors NB = 8 at a time.
// Phase A encodes one (token, KV head) vector at a time (lane l holds
// coordinates l + 32k), up to the key residual r, which it leaves in shared
// memory as three bf16 pieces (r = hi + mid + lo to ~24 significant bits).
// Phase B projects the eight residuals at once on tensor cores: z = S [r_0 ..
// r_7] as (d/16)^2 m16n8k16 tiles per piece, with S (bf16, exact) as the A
// operand from a padded shared copy; bit j of vector v is [z_jv >= 0], and
// lane (v, w) assembles sign word w of vector v from the tiles' ballots.
constexpr int kStoreNB = 8;  // vectors per warp batch (the MMA's N)

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// bits 4g (g = 0..7) of x -> bits g
__device__ __forceinline__ uint32_t gather_nibble_bits(uint32_t x) {
    x &= 0x11111111u;
    x = (x | (x >> 3)) & 0x03030303u;
    x = (x | (x >> 6)) & 0x000F000Fu;
    return (x | (x >> 12)) & 0xFFu;
}

template <int D>
struct StoreBulkLayout {
    static constexpr int kWarps = D == 128 ? 24 : 4;
    static constexpr int SP = 2 * D + 16;             // padded S row (bytes)
    static constexpr int VS = 3 * 2 * D + 16;         // one vector's residual pieces (bytes, padded)
    static constexpr size_t s_off = 0;
    static constexpr size_t rp_off = s_off + (size_t)D * SP;
    static constexpr size_t sg_off = rp_off + (size_t)kWarps * kStoreNB * VS;
    static constexpr size_t cw_off = sg_off + (size_t)kWarps * kStoreNB * 8;
    static constexpr size_t tab_off = cw_off + (size_t)kWarps * D;
    static constexpr size_t total = tab_off + (size_t)(D + 4 * kMaxLevels) * 4;
};

template <int D, typename Tin>
__global__ void __launch_bounds__(StoreBulkLayout<D>::kWarps * 32) store_kernel(StoreArgs a) {
    using SL = StoreBulkLayout<D>;
    constexpr int PER = D / 32;
    constexpr int kWarps = SL::kWarps;
    constexpr int NT = D / 16;  // m16n8k16 tiles per dimension
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t* s_rows = smem + SL::s_off;                                   // S, bf16 [D][D], padded rows
    uint8_t* rp_all = smem + SL::rp_off;                                  // [warp][NB] residual pieces
    uint8_t** sg_all = reinterpret_cast<uint8_t**>(smem + SL::sg_off);    // [warp][NB] sign rows (or null)
    uint8_t* codes = smem + SL::cw_off;                                   // [warp][D]
    float* tables = reinterpret_cast<float*>(smem + SL::tab_off);
    float* s_signs = tables;
    float* s_kc = tables + D;
    float* s_kb = s_kc + kMaxLevels;
    float* s_vc = s_kb + kMaxLevels;
    float* s_vb = s_vc + kMaxLevels;

    const Layout& L = a.lay;
    // S (row-major bf16) into padded rows: 16-byte chunks
    for (int e = threadIdx.x; e < D * D / 8; e += blockDim.x) {
        const int row = e / (D / 8), ch = e % (D / 8);
        *reinterpret_cast<uint4*>(s_rows + row * SL::SP + 16 * ch) =
            __ldg(reinterpret_cast<const uint4*>(a.dp.s_bf16) + e);
    }
    for (int e = threadIdx.x; e < D; e += blockDim.x) s_signs[e] = a.dp.signs[e];
    for (int e = threadIdx.x; e < kMaxLevels; e += blockDim.x) {
        s_kc[e] = a.dp.k_cent[e];
        s_kb[e] = a.dp.k_bound[e];
        s_vc[e] = a.dp.v_cent[e];
        s_vb[e] = a.dp.v_bound[e];
    }
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gq = lane >> 2, tq = lane & 3;
    uint8_t* rp = rp_all + (size_t)warp * kStoreNB * SL::VS;
    uint8_t** sg = sg_all + warp * kStoreNB;
    uint8_t* cw = codes + warp * D;
    const float rsd = rsqrtf((float)D);
    const bool qjl = L.k_qjl;
    const int64_t nvec = a.num_tokens * a.heads;
    const int64_t wstep = (int64_t)gridDim.x * kWarps * kStoreNB;
    // the next vector's key, value and slot load while the current one is
    // encoded (one vector ahead, across batches)
    float nxk[PER], nxv[PER];
    int64_t nslot = -1;
    auto prefetch = [&](int64_t w) {
        if (w < nvec) {
            const Tin* kin = static_cast<const Tin*>(a.k) + w * D;
            const Tin* vin = static_cast<const Tin*>(a.v) + w * D;
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                nxk[k] = load_as_float(kin + lane + 32 * k);
                nxv[k] = load_as_float(vin + lane + 32 * k);
            }
            nslot = a.slots[w / a.heads];
        }
    };
    prefetch(((int64_t)blockIdx.x * kWarps + warp) * kStoreNB);
    for (int64_t w0 = ((int64_t)blockIdx.x * kWarps + warp) * kStoreNB; w0 < nvec; w0 += wstep) {
        // ---------------------------------------------- phase A: per vector
#pragma unroll 1
        for (int v = 0; v < kStoreNB; ++v) {
            const int64_t w = w0 + v;
            uint8_t* srow = nullptr;  // this vector's sign row, if it is written
            __nv_bfloat16* pv = reinterpret_cast<__nv_bfloat16*>(rp + v * SL::VS);
            float x[PER], xv[PER];
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                x[k] = nxk[k];
                xv[k] = nxv[k];
            }
            const int64_t slot = nslot;
            prefetch(v + 1 < kStoreNB ? w + 1 : w0 + wstep);
            if (w < nvec) {
                const int64_t t = nvec < (int64_t)1 << 31 ? (int64_t)((uint32_t)w / (uint32_t)a.heads) : w / a.heads;
                const int h = (int)(w - t * a.heads);
                if (slot < 0 || slot >= a.num_slots) {
                    if (slot != -1 && lane == 0 && h == 0) set_error(a.dp.err, TQ_DEVERR_SLOT);
                } else {
                    const int row = (int)(slot & 15);
                    uint8_t* page = a.cache + ((slot >> 4) * a.heads + h) * (int64_t)L.page_bytes;

                    // -------------------------------------------------- key
                    int idx[PER];
                    const float n = mse_codes<D>(x, s_signs, s_kb, (1 << L.k_bits) - 1, lane, idx);
                    const __half n16 = __float2half_rn(n);
                    write_bit_planes<D>(idx, L.k_bits, page + L.k_codes, row, lane);
                    if (lane == 0) reinterpret_cast<__half*>(page + L.k_norm)[row] = n16;
                    if (qjl) {
                        // residual r = k - n16 R^T c[idx] as three bf16 pieces
                        float c[PER];
#pragma unroll
                        for (int k = 0; k < PER; ++k) c[k] = s_kc[idx[k]];
                        fwht_warp<PER>(c, lane);
                        const float n16f = __half2float(n16);
                        float rr = 0.f;
#pragma unroll
                        for (int k = 0; k < PER; ++k) {
                            const int i = lane + 32 * k;
                            const float res = x[k] - n16f * (c[k] * s_signs[i] * rsd);
                            rr = fmaf(res, res, rr);
                            const __nv_bfloat16 p0 = __float2bfloat16_rn(res);
                            const float r1 = res - __bfloat162float(p0);
                            const __nv_bfloat16 p1 = __float2bfloat16_rn(r1);
                            const __nv_bfloat16 p2 = __float2bfloat16_rn(r1 - __bfloat162float(p1));
                            pv[i] = p0;
                            pv[D + i] = p1;
                            pv[2 * D + i] = p2;
                        }
                        const float rho = sqrtf(warp_sum(rr));
                        if (lane == 0) reinterpret_cast<__half*>(page + L.k_rnorm)[row] = __float2half_rn(rho);
                        srow = page + L.k_signs + row * (D / 8);
                    }

                    // ------------------------------------------------ value
#pragma unroll
                    for (int k = 0; k < PER; ++k) x[k] = xv[k];
                    if (L.v_mode == TQ_V_MSE) {
                        const float vn = mse_codes<D>(x, s_signs, s_vb, (1 << L.v_bits) - 1, lane, idx);
                        write_bit_planes<D>(idx, L.v_bits, page + L.v_codes, row, lane);
                        if (lane == 0) reinterpret_cast<__half*>(page + L.v_meta)[row] = __float2half_rn(vn);
                    } else {
                        // group g = coordinates [32g, 32g+32) = slot k of every lane
                        const int top = (1 << L.v_bits) - 1;
                        uint32_t* meta = reinterpret_cast<uint32_t*>(page + L.v_meta + row * L.v_meta_row);
#pragma unroll
                        for (int k = 0; k < PER; ++k) {
                            const float lo = warp_min(x[k]), hi = warp_max(x[k]);
                            const __half z16 = __float2half_rn(lo);
                            const __half s16 = __float2half_rn((hi - lo) / (float)top);
                            const float zf = __half2float(z16), sf = __half2float(s16);
                            int q = 0;
                            if (sf > 0.f) {
                                const float tqv = (x[k] - zf) / sf;
                                const float fl = floorf(tqv);
                                q = (int)fl + ((tqv - fl) >= 0.5f ? 1 : 0);
                                q = min(max(q, 0), top);
                            }
                            cw[g32_slot<D>(lane + 32 * k)] = (uint8_t)q;
                            if (lane == k)
                                meta[k] = (uint32_t)__half_as_ushort(s16) | ((uint32_t)__half_as_ushort(z16) << 16);
                        }
                        __syncwarp();
                        pack_row(cw, D, L.v_bits, page + L.v_codes + row * L.v_code_row, lane);
                    }
                }
            }
            if (srow == nullptr && qjl) {
                // a vector with no sign row still feeds the batch: zero residual
#pragma unroll
                for (int k = 0; k < PER; ++k) {
                    const int i = lane + 32 * k;
                    pv[i] = pv[D + i] = pv[2 * D + i] = __float2bfloat16_rn(0.f);
                }
            }
            if (lane == 0) sg[v] = srow;
            __syncwarp();
        }
        if (!qjl) continue;

        // ------------------------------------- phase B: z = S [r_0 .. r_7]
        // lane (v, w) writes sign words w = (lane & 3) + 4 q of vector v = lane >> 2
        constexpr int NWQ = D / 128;  // sign words per lane
        uint32_t word[NWQ];
#pragma unroll
        for (int q = 0; q < NWQ; ++q) word[q] = 0u;
        const uint32_t s_base = smem_u32(s_rows) + (uint32_t)(((lane & 7) + ((lane >> 3) & 1) * 8) * SL::SP +
                                                              ((lane >> 4) * 8) * 2);
        const uint8_t* rv = rp + gq * SL::VS;  // B operand: vector n = gq
#pragma unroll 1
        for (int mt = 0; mt < NT; ++mt) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int kt = 0; kt < NT; ++kt) {
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4(s_base + (uint32_t)(16 * mt * SL::SP + 32 * kt), a0, a1, a2, a3);
#pragma unroll
                for (int p = 0; p < 3; ++p) {
                    const uint8_t* bp = rv + p * 2 * D + (16 * kt + 2 * tq) * 2;
                    const uint32_t b0 = *reinterpret_cast<const uint32_t*>(bp);
                    const uint32_t b1 = *reinterpret_cast<const uint32_t*>(bp + 16);
                    mma_bf16(acc, a0, a1, a2, a3, b0, b1);
                }
            }
            // acc: z(16 mt + gq, 2 tq), z(.., 2 tq + 1), z(16 mt + gq + 8, 2 tq), z(.., 2 tq + 1)
            const uint32_t bl0 = __ballot_sync(0xffffffffu, acc[0] >= 0.f);
            const uint32_t bl1 = __ballot_sync(0xffffffffu, acc[1] >= 0.f);
            const uint32_t bl2 = __ballot_sync(0xffffffffu, acc[2] >= 0.f);
            const uint32_t bl3 = __ballot_sync(0xffffffffu, acc[3] >= 0.f);
            // vector v = gq of this lane: column 2 tq' + e with tq' = v >> 1, e = v & 1
            const int v = gq, sh = v >> 1;
            const uint32_t lo8 = gather_nibble_bits(((v & 1) ? bl1 : bl0) >> sh);  // rows 16 mt + 0..7
            const uint32_t hi8 = gather_nibble_bits(((v & 1) ? bl3 : bl2) >> sh);  // rows 16 mt + 8..15
            const int wsel = mt >> 1;  // word of rows 32 wsel .. 32 wsel + 31
            const uint32_t bits16 = (lo8 | (hi8 << 8)) << (16 * (mt & 1));
#pragma unroll
            for (int q = 0; q < NWQ; ++q)
                if (wsel == tq + 4 * q) word[q] |= bits16;
        }
        uint8_t* dst = sg[gq];
        if (dst != nullptr) {
#pragma unroll
            for (int q = 0; q < NWQ; ++q) reinterpret_cast<uint32_t*>(dst)[tq + 4 * q] = word[q];
        }
        __syncwarp();
    }
}

// Few vectors (a decode step's new tokens): one CTA of d threads per
// (token, KV head).  Warp 0 encodes the key and the residual, warp 1 the
// value, then warp w projects the residual onto rows 32w .. 32w+31 of S
// (row-major bf16, read straight from L2) and writes that word of sign bits.
// The sums run over i in the same order as store_kernel's.
template <int D, typename Tin>
__global__ void __launch_bounds__(D) store_small_kernel(StoreArgs a) {
    // a programmatically launched successor (the decode's query prep) may be
    // scheduled now; it waits for this grid to finish before it reads anything
    pdl_launch_dependents();
    constexpr int PER = D / 32;
    constexpr int kChunk = 16;  // uint4 (8 bf16) loads of an S row held at once
    __shared__ __align__(16) float r_s[D];
    __shared__ float s_signs[D], s_kb[kMaxLevels], s_kc[kMaxLevels], s_vb[kMaxLevels];
    __shared__ float rho_s;
    __shared__ uint8_t cw_s[D];
    const Layout& L = a.lay;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t w = blockIdx.x;
    const int64_t t = w / a.heads;
    const int h = (int)(w - t * a.heads);
    const int64_t slot = a.slots[t];
    const bool qjl = L.k_qjl;
    // every load of the encoding at once, the slot's among them (none of the
    // others depends on it): the input vector (warp 0: key, warp 1: value),
    // the tables, and this warp's first S rows
    float x[PER];
    if (warp < 2) {
        const Tin* in = static_cast<const Tin*>(warp == 0 ? a.k : a.v) + w * D;
#pragma unroll
        for (int k = 0; k < PER; ++k) x[k] = load_as_float(in + lane + 32 * k);
    }
    s_signs[threadIdx.x] = __ldg(a.dp.signs + threadIdx.x);
    if (threadIdx.x < kMaxLevels) {
        s_kb[threadIdx.x] = __ldg(a.dp.k_bound + threadIdx.x);
        s_kc[threadIdx.x] = __ldg(a.dp.k_cent + threadIdx.x);
        s_vb[threadIdx.x] = __ldg(a.dp.v_bound + threadIdx.x);
    }
    const uint4* srow = reinterpret_cast<const uint4*>(a.dp.s_bf16 + (size_t)(32 * warp + lane) * D);
    uint4 sv[kChunk];
    if (qjl) {
#pragma unroll
        for (int q = 0; q < kChunk; ++q) sv[q] = __ldg(srow + q);
    }
    // a skipped or bad slot ends the block (uniformly: the slot is per block)
    if (slot < 0 || slot >= a.num_slots) {
        if (slot != -1 && threadIdx.x == 0 && h == 0) set_error(a.dp.err, TQ_DEVERR_SLOT);
        return;
    }
    const int row = (int)(slot & 15);
    uint8_t* page = a.cache + ((slot >> 4) * a.heads + h) * (int64_t)L.page_bytes;
    __syncthreads();
    if (warp == 0) {
        // ------------------------------------------------------------ key
        int idx[PER];
        const float n = mse_codes<D>(x, s_signs, s_kb, (1 << L.k_bits) - 1, lane, idx);
        const __half n16 = __float2half_rn(n);
        write_bit_planes<D>(idx, L.k_bits, page + L.k_codes, row, lane);
        if (lane == 0) reinterpret_cast<__half*>(page + L.k_norm)[row] = n16;
        if (qjl) {
            float c[PER];
#pragma unroll
            for (int k = 0; k < PER; ++k) c[k] = s_kc[idx[k]];
            fwht_warp<PER>(c, lane);
            const float n16f = __half2float(n16), rsd = rsqrtf((float)D);
            float rr = 0.f;
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int i = lane + 32 * k;
                const float res = x[k] - n16f * (c[k] * s_signs[i] * rsd);
                r_s[i] = res;
                rr = fmaf(res, res, rr);
            }
            const float rho = sqrtf(warp_sum(rr));
            if (lane == 0) rho_s = rho;
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- value
        if (L.v_mode == TQ_V_MSE) {
            int idx[PER];
            const float vn = mse_codes<D>(x, s_signs, s_vb, (1 << L.v_bits) - 1, lane, idx);
            write_bit_planes<D>(idx, L.v_bits, page + L.v_codes, row, lane);
            if (lane == 0) reinterpret_cast<__half*>(page + L.v_meta)[row] = __float2half_rn(vn);
        } else {
            const int top = (1 << L.v_bits) - 1;
            uint32_t* meta = reinterpret_cast<uint32_t*>(page + L.v_meta + row * L.v_meta_row);
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const float lo = warp_min(x[k]), hi = warp_max(x[k]);
                const __half z16 = __float2half_rn(lo);
                const __half s16 = __float2half_rn((hi - lo) / (float)top);
                const float zf = __half2float(z16), sf = __half2float(s16);
                int q = 0;
                if (sf > 0.f) {
                    const float tq = (x[k] - zf) / sf;
                    const float fl = floorf(tq);
                    q = (int)fl + ((tq - fl) >= 0.5f ? 1 : 0);
                    q = min(max(q, 0), top);
                }
                cw_s[g32_slot<D>(lane + 32 * k)] = (uint8_t)q;
                if (lane == k)
                    meta[k] = (uint32_t)__half_as_ushort(s16) | ((uint32_t)__half_as_ushort(z16) << 16);
            }
            __syncwarp();
            pack_row(cw_s, D, L.v_bits, page + L.v_codes + row * L.v_code_row, lane);
        }
    }
    if (!qjl) return;
    __syncthreads();
    // z_j = sum_i S[j][i] r_i for j = 32 warp + lane; bit j = [z_j >= 0]
    // (four partial sums: four short dependency chains instead of one of d)
    float z4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int q0 = 0; q0 < D / 8; q0 += kChunk) {
        if (q0 > 0) {
#pragma unroll
            for (int q = 0; q < kChunk; ++q) sv[q] = __ldg(srow + q0 + q);
        }
#pragma unroll
        for (int q = 0; q < kChunk; ++q) {
            const float4 ra = *reinterpret_cast<const float4*>(&r_s[8 * (q0 + q)]);
            const float4 rb = *reinterpret_cast<const float4*>(&r_s[8 * (q0 + q) + 4]);
            const uint4 u = sv[q];
            z4[0] = fmaf(__uint_as_float(u.x << 16), ra.x, z4[0]);
            z4[0] = fmaf(__uint_as_float(u.x & 0xFFFF0000u), ra.y, z4[0]);
            z4[1] = fmaf(__uint_as_float(u.y << 16), ra.z, z4[1]);
            z4[1] = fmaf(__uint_as_float(u.y & 0xFFFF0000u), ra.w, z4[1]);
            z4[2] = fmaf(__uint_as_float(u.z << 16), rb.x, z4[2]);
            z4[2] = fmaf(__uint_as_float(u.z & 0xFFFF0000u), rb.y, z4[2]);
            z4[3] = fmaf(__uint_as_float(u.w << 16), rb.z, z4[3]);
            z4[3] = fmaf(__uint_as_float(u.w & 0xFFFF0000u), rb.w, z4[3]);
        }
    }
    const float z = (z4[0] + z4[1]) + (z4[2] + z4[3]);
    const uint32_t bits = __ballot_sync(0xffffffffu, z >= 0.f);
    if (lane == 0) reinterpret_cast<uint32_t*>(page + L.k_signs + row * (D / 8))[warp] = bits;
    if (threadIdx.x == 0) reinterpret_cast<__half*>(page + L.k_rnorm)[row] = __float2half_rn(rho_s);
}

// largest vector count for store_small_kernel; negative: 16 x the SM count
static std::atomic<int64_t> g_small_max{-1};

template <int D, typename Tin>
static tq_status launch(const StoreArgs& a, cudaStream_t s, void* ev0, void* ev1) {
    const size_t smem = StoreBulkLayout<D>::total;
    auto kern = store_kernel<D, Tin>;
    // per-device set-up (the first call on a device does it; before any capture)
    int sms = 0;
    {
        tq_status fs = device_sms(&sms);
        if (fs == TQ_OK) fs = ensure_dynamic_smem((const void*)kern, (int)smem, "store_kernel");
        if (fs != TQ_OK) return fs;
    }
    const int64_t nvec = a.num_tokens * a.heads;
    const int64_t small_max = g_small_max.load(std::memory_order_relaxed);
    if (ev0) cudaEventRecord((cudaEvent_t)ev0, s);
    if (nvec <= (small_max < 0 ? (int64_t)sms * 16 : small_max)) {
        // few vectors: one CTA each (no shared copy of S to stage)
        store_small_kernel<D, Tin><<<(unsigned)nvec, D, 0, s>>>(a);
    } else if (store_tc_supported(a, std::is_same<Tin, float>::value ? TQ_DTYPE_F32 : TQ_DTYPE_BF16)) {
        // bulk appends at d = 128 from bf16: tiles of 128 vectors on the tensor cores
        const tq_status st = launch_store_tc(a, s, sms);
        if (st != TQ_OK) return st;
    } else {
        constexpr int kPerCta = StoreBulkLayout<D>::kWarps * kStoreNB;  // vectors per CTA pass
        const int grid = (int)std::min<int64_t>((nvec + kPerCta - 1) / kPerCta, (int64_t)sms);
        kern<<<grid, StoreBulkLayout<D>::kWarps * 32, smem, s>>>(a);
    }
    if (ev1) cudaEventRecord((cudaEvent_t)ev1, s);
    return cuda_status(cudaGetLastError());
}

}  // namespace tq

using namespace tq;

extern "C" tq_status tq_set_store_small_max(int64_t max_vectors) {
    g_small_max.store(max_vectors < 0 ? -1 : max_vectors, std::memory_order_relaxed);
    return TQ_OK;
}

extern "C" tq_status tq_store(const tq_cache* c, const void* k, const void* v, int in_dtype, int64_t num_tokens,
                              const int64_t* slot_mapping, void* cache_buf, void* stream) {
    if (!c || num_tokens < 0) return TQ_ERR_INVALID_ARG;
    if (num_tokens == 0) return TQ_OK;
    if (!k || !v || !slot_mapping || !cache_buf) return TQ_ERR_INVALID_ARG;
    if (in_dtype != TQ_DTYPE_F32 && in_dtype != TQ_DTYPE_BF16) return TQ_ERR_INVALID_ARG;
    if (((uintptr_t)cache_buf & 15) || ((uintptr_t)k & 3) || ((uintptr_t)v & 3)) return TQ_ERR_MISALIGNED;
    StoreArgs a;
    a.k = k;
    a.v = v;
    a.slots = slot_mapping;
    a.cache = static_cast<uint8_t*>(cache_buf);
    a.num_tokens = num_tokens;
    a.num_slots = c->cfg.num_blocks * kBlock;
    a.heads = c->cfg.num_kv_heads;
    a.lay = c->lay;
    a.dp = c->dp;
    cudaStream_t s = (cudaStream_t)stream;
    const int d = c->cfg.head_dim;
    void *e0 = c->prof_start[TQ_PROF_STORE], *e1 = c->prof_stop[TQ_PROF_STORE];
    if (in_dtype == TQ_DTYPE_F32)
        return d == 128 ? launch<128, float>(a, s, e0, e1) : launch<256, float>(a, s, e0, e1);
    return d == 128 ? launch<128, __nv_bfloat16>(a, s, e0, e1) : launch<256, __nv_bfloat16>(a, s, e0, e1);
}
