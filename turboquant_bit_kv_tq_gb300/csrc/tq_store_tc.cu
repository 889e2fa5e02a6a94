// Bulk KV-cache store on the tensor cores (d = 128, bf16 inputs): the same
// bytes as store_kernel, for appends of many vectors ([Roadmap] §3.1: the WHT
// rotation and the quantisation fused into the store; [Hub] "Technical
// principle" steps 1-5; [Paged] "Which path vLLM takes").
//
// A tile is 128 consecutive (token, KV head) vectors.  Per tile:
//   1. the tile's K and V rows land in shared memory by bulk-tensor copies
//      (16 boxes of 8 elements x 128 rows each) in the tensor cores' K-major
//      layout, issued by the MMA warp as soon as the last tile's rotation
//      MMAs have read the buffer;
//   2. tcgen05 MMAs rotate them: Y = X (D H)^T, i.e. y = H D x for every row
//      (the input is bf16 and D H is +-1, so every product is exact; the sums
//      accumulate in fp32 in tensor memory);
//   3. one thread per vector reads its row of Y: the norm n = ||y|| / sqrt(d),
//      the codes (the number of Lloyd-Max boundaries below y / (n sqrt(d)),
//      found by comparing |y| against the positive boundaries scaled by
//      n sqrt(d)), the bit planes, and for keys the rotated residual
//        r~ = R k - n16 c[idx] = y / sqrt(d) - n16 c[idx]   (= R r)
//      scaled by a power of two and split into fp16 high and low parts;
//   4. for keys with QJL, tcgen05 MMAs project it word by word (32
//      coordinates, as the threads finish them): z = T r~ with
//      T = S R^T = S D H / sqrt(d) (so z = S r), as T_hi r~_hi + T_hi r~_lo +
//      T_lo r~_hi (T_hi, T_lo: T's fp16 parts from the cache parameters);
//      bit j = [z_j >= 0];
//   5. the thread writes its vector's page rows.
// Group-32 values skip the rotation: their thread reads its row from shared
// memory.  Two warpgroups of four warps take alternate tiles, each with its
// own MMA-issue warp, so one tile's CUDA-core work overlaps the other's MMAs.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <dlfcn.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "tq_store.cuh"

namespace tq {

constexpr int kTcWG = 2;                                  // compute warpgroups per CTA
constexpr int kTcThreads = 32 * (4 * kTcWG + kTcWG);      // + one MMA-issue warp each
constexpr float kTcRsd = 0.08838834764831845f;            // 1 / sqrt(128)
constexpr int kTcBars = 10;                               // mbarriers per warpgroup

struct TcLayout {
    static constexpr uint32_t x_bytes = 65536;            // per warpgroup: X_k (32 KB) then X_v (32 KB)
    static constexpr uint32_t mt = kTcWG * x_bytes;       // rotation operand (D H)^T, bf16
    static constexpr uint32_t th = mt + 32768;            // T high part, fp16
    static constexpr uint32_t tl = th + 32768;            // T low part, fp16
    static constexpr uint32_t tab = tl + 32768;           // float tables
    static constexpr uint32_t bars = tab + 256;           // kTcBars mbarriers per warpgroup
    static constexpr uint32_t tslot = bars + 8 * kTcBars * kTcWG;
    static constexpr uint32_t total = tslot + 16;
};
static_assert(TcLayout::total <= 227 * 1024, "shared memory");

// Byte offset of the 16-byte chunk j (elements 8j .. 8j+7) of row r in the
// no-swizzle K-major layout: 8-row x 16-byte core matrices, 8-row groups 128 B
// apart, chunk columns 2048 B apart.  A thread's row is 16 B per chunk and a
// warp's 32 rows are 512 contiguous bytes.
__device__ __forceinline__ uint32_t tc_chunk(int r, int j) {
    return (uint32_t)j * 2048u + ((uint32_t)r >> 3) * 128u + ((uint32_t)r & 7u) * 16u;
}

// D[128 x 128] (+)= A[128 x 16] B[128 x 16]^T, both operands in shared memory
// (kind::f16: fp16 or bf16 inputs, fp32 accumulation), issued by one thread
__device__ __forceinline__ void mma_f16_ss(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}
// the same with A (fp16 pairs per 32-bit column) from tensor memory
__device__ __forceinline__ void mma_f16_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}
// instruction descriptor: fp32 accumulate, A and B bf16 (or fp16), K-major,
// M = 128, N = 128
__host__ __device__ constexpr uint32_t f16kind_idesc(bool bf16) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((128u >> 3) << 17) |
           ((128u >> 4) << 24);
}
__device__ __forceinline__ uint64_t tc_desc(uint32_t addr) { return smem_desc(addr, 2048, 128); }

// (w << 1) | top bit of m
__device__ __forceinline__ uint32_t push_bit(uint32_t w, uint32_t m) { return __funnelshift_l(m, w, 1); }
// a * b + c on the integer multiply-add pipe (the FMA pipe): with b01 in
// {0, 1}, imad(b01, A - B, B) selects A or B and imad(w, 2, b01) pushes a bit,
// leaving the ALU pipe (logic, shifts, integer adds) to what only it does
__device__ __forceinline__ uint32_t imad(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// 1 if x is negative (its sign bit), else 0
__device__ __forceinline__ uint32_t neg01(float x) { return __float_as_uint(x) >> 31; }

// The cells of |y| against a symmetric codebook's sorted positive boundaries
// T_0 < ... < T_{2^NB - 2} (scaled by n sqrt(d)) and positive centroids G_c:
// cnt = #{T below |y|} by a binary search whose steps are the signs of
// T - |y| (fp32 subtraction without flush-to-zero: the computed difference is
// negative iff |y| > T, and +0 when they are equal), the threshold of each
// step chosen by bit-weighted multiply-adds on T's bit patterns; G_cnt by the
// same multiply-adds over the bits of cnt.
template <int NB>
struct Cells {
    float tf;          // the first step's threshold: T_{2^(NB-1) - 1}
    uint32_t tb[4];    // the later steps' base patterns and differences
    uint32_t gb[8];    // G_0 and the bit-weighted differences of the centroids
    __device__ __forceinline__ void init(const float* T, const float* G) {
        auto u = [](float x) { return __float_as_uint(x); };
        if constexpr (NB == 1) {
            tf = T[0];
            gb[0] = u(G[0]);
            gb[1] = u(G[1]) - u(G[0]);
        } else if constexpr (NB == 2) {
            tf = T[1];
            tb[0] = u(T[0]);
            tb[1] = u(T[2]) - u(T[0]);
            gb[0] = u(G[0]);
            gb[1] = u(G[1]) - u(G[0]);
            gb[2] = u(G[2]) - u(G[0]);
            gb[3] = u(G[3]) - u(G[2]) - u(G[1]) + u(G[0]);
        } else {
            tf = T[3];
            tb[0] = u(T[1]);                              // second step: T_1 or T_5
            tb[1] = u(T[5]) - u(T[1]);
            tb[2] = u(T[2]) - u(T[0]);                    // third step: T_{4 b2 + 2 b1}
            tb[3] = u(T[6]) - u(T[4]) - u(T[2]) + u(T[0]);
            gb[0] = u(G[0]);                              // G_{b0 + 2 b1} and G_{4 + b0 + 2 b1}
            gb[1] = u(G[1]) - u(G[0]);
            gb[2] = u(G[2]) - u(G[0]);
            gb[3] = u(G[3]) - u(G[2]) - u(G[1]) + u(G[0]);
            gb[4] = u(G[4]);
            gb[5] = u(G[5]) - u(G[4]);
            gb[6] = u(G[6]) - u(G[4]);
            gb[7] = u(G[7]) - u(G[6]) - u(G[5]) + u(G[4]);
            t0 = u(T[0]);
            t40 = u(T[4]) - u(T[0]);
        }
    }
    uint32_t t0 = 0, t40 = 0;  // NB = 3: T_0 and T_4 - T_0
    // bits b[q] (0/1) of cnt for a = |y|
    __device__ __forceinline__ void bits(float a, uint32_t (&b)[3]) const {
        if constexpr (NB == 1) {
            b[0] = neg01(tf - a);
        } else if constexpr (NB == 2) {
            b[1] = neg01(tf - a);
            b[0] = neg01(__uint_as_float(imad(b[1], tb[1], tb[0])) - a);
        } else {
            b[2] = neg01(tf - a);
            b[1] = neg01(__uint_as_float(imad(b[2], tb[1], tb[0])) - a);
            const uint32_t p = imad(b[1], b[2], 0u);
            uint32_t t = imad(b[1], tb[2], t0);
            t = imad(b[2], t40, t);
            t = imad(p, tb[3], t);
            b[0] = neg01(__uint_as_float(t) - a);
        }
    }
    // G_cnt (float bits)
    __device__ __forceinline__ uint32_t centroid(const uint32_t (&b)[3]) const {
        if constexpr (NB == 1) {
            return imad(b[0], gb[1], gb[0]);
        } else {
            const uint32_t p = imad(b[0], b[1], 0u);
            uint32_t lo = imad(b[0], gb[1], gb[0]);
            lo = imad(b[1], gb[2], lo);
            lo = imad(p, gb[3], lo);
            if constexpr (NB == 2) {
                return lo;
            } else {
                uint32_t hi = imad(b[0], gb[5], gb[4]);
                hi = imad(b[1], gb[6], hi);
                hi = imad(p, gb[7], hi);
                return imad(b[2], hi - lo, lo);
            }
        }
    }
};

// Plane words of 32 coordinates are built from four 8-bit accumulators
// (coordinates 8q+7 .. 8q pushed, highest first, into accumulator q), joined
// as bytes: four short dependency chains instead of one of 32.
struct Bits32 {
    uint32_t q[4] = {0u, 0u, 0u, 0u};
    // the top bit of m (a shift on the ALU pipe)
    __device__ __forceinline__ void push(int i, uint32_t m) { q[i >> 3] = push_bit(q[i >> 3], m); }
    // a 0/1 bit (a multiply-add on the FMA pipe)
    __device__ __forceinline__ void push01(int i, uint32_t b) { q[i >> 3] = imad(q[i >> 3], 2u, b); }
    __device__ __forceinline__ uint32_t word() const {
        return __byte_perm(__byte_perm(q[0], q[1], 0x0040), __byte_perm(q[2], q[3], 0x0040), 0x5410);
    }
};

// Codes of a symmetric codebook with B bits: idx = 2^(B-1) + cnt for y > 0,
// 2^(B-1) - 1 - cnt otherwise (cnt = #{positive boundaries below |y|}), i.e.
// plane B-1 = [y > 0] and plane q < B-1 = bit q of cnt XOR [y <= 0].  [y > 0]
// is taken as "sign bit clear" on a non-zero row (a coordinate exactly +0 of a
// non-zero row is a boundary case; an all-zero row gets [y > 0] = 0 and so
// the middle-low code, as the definition gives).

// 32 consecutive fp32 columns of this thread's lane of tensor memory
__device__ __forceinline__ void tmem_row32(uint32_t taddr, float (&y)[32]) {
    uint32_t r[32];
    tmem_ld32(taddr, r);
    tc_wait_ld();
#pragma unroll
    for (int c = 0; c < 32; ++c) y[c] = __uint_as_float(r[c]);
}

// ||y|| / sqrt(128) of the 128 columns at taddr: four loads, eight running
// sums of 16 squares, then a tree
__device__ __forceinline__ float row_norm128(uint32_t taddr) {
    float s[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) s[k] = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t r[2][32];
        tmem_ld32(taddr + 64 * h, r[0]);
        tmem_ld32(taddr + 64 * h + 32, r[1]);
        tc_wait_ld();
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float y = __uint_as_float(r[q][c]);
                s[c & 7] = fmaf(y, y, s[c & 7]);
            }
    }
    return sqrtf((((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]))) * (1.f / 128.f));
}

// MSE codes of the rotated row at taddr (values): the fp32 norm; the plane
// words go straight to the page's rows (planes at `planes`, row `row`) when
// `planes` is not null.  PB: the codebook's positive boundaries (2^(B-1) - 1).
template <int B>
__device__ __forceinline__ float mse_planes(uint32_t taddr, const float* PB, uint8_t* planes, int row) {
    constexpr int NB = B - 1;
    const float n = row_norm128(taddr);
    const uint32_t nz = n > 0.f ? 0xFFFFFFFFu : 0u;
    float T[7], G[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const float sc = n * 11.313708498984761f;  // n sqrt(d)
#pragma unroll
    for (int k = 0; k < (1 << NB) - 1; ++k) T[k] = PB[k] * sc;
    Cells<NB> cells;
    cells.init(T, G);
    uint32_t W[B][4];
    // word wd + 1 loads from tensor memory while word wd is encoded
    uint32_t ybuf[32];
    tmem_ld32(taddr, ybuf);
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
        float y[32];
        tc_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) y[c] = __uint_as_float(ybuf[c]);
        if (wd < 3) tmem_ld32(taddr + 32 * (wd + 1), ybuf);
        Bits32 S, C[NB];
#pragma unroll
        for (int i = 31; i >= 0; --i) {
            uint32_t b[3];
            cells.bits(fabsf(y[i]), b);
            S.push(i, __float_as_uint(y[i]));  // the sign bit
#pragma unroll
            for (int q = 0; q < NB; ++q) C[q].push01(i, b[q]);
        }
        const uint32_t pos = ~S.word() & nz;  // [y > 0]
        W[B - 1][wd] = pos;
#pragma unroll
        for (int q = 0; q < NB; ++q) W[q][wd] = C[q].word() ^ ~pos;
    }
    if (planes) {
#pragma unroll
        for (int p = 0; p < B; ++p)
            *reinterpret_cast<uint4*>(planes + (p * kBlock + row) * 16) = make_uint4(W[p][0], W[p][1], W[p][2], W[p][3]);
    }
    return n;
}

// Group-32 value fields of one row read from shared memory (bf16, canonical
// layout): zero = fp16(min), scale = fp16((max - min)/(2^VB - 1)),
// q = clamp(floor((v - zero)/scale + 1/2)); fields in the page's slot order.
template <int VB>
__device__ __forceinline__ void g32_row(const uint8_t* xrow_base, int v, uint8_t* codes, uint8_t* meta) {
    constexpr int top = (1 << VB) - 1;
    uint32_t words[VB * 4];  // the 128 x VB-bit row: 16 (VB = 4) or 8 (VB = 2) words
#pragma unroll
    for (int k = 0; k < VB * 4; ++k) words[k] = 0u;
    uint32_t mw[4];
#pragma unroll
    for (int gr = 0; gr < 4; ++gr) {
        float x[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 u = *reinterpret_cast<const uint4*>(xrow_base + tc_chunk(v, 4 * gr + j));
            const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[8 * j + 2 * e] = __uint_as_float(ww[e] << 16);
                x[8 * j + 2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
            }
        }
        float lo = x[0], hi = x[0];
#pragma unroll
        for (int i = 1; i < 32; ++i) {
            lo = fminf(lo, x[i]);
            hi = fmaxf(hi, x[i]);
        }
        const __half z16 = __float2half_rn(lo);
        const __half s16 = __float2half_rn((hi - lo) / (float)top);
        const float zf = __half2float(z16), sf = __half2float(s16);
        mw[gr] = (uint32_t)__half_as_ushort(s16) | ((uint32_t)__half_as_ushort(z16) << 16);
        // t = (v - zero) / scale from the correctly rounded reciprocal and one
        // fma correction (the quotient correctly rounded but for ties of the
        // rounding itself, one ulp -- below 1e-6 at t <= 15 -- away at most);
        // a zero scale gives t = 0 and so q = 0
        const float rs = sf > 0.f ? __frcp_rn(sf) : 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float num = x[i] - zf;
            const float q0 = num * rs;
            const float t = fmaf(fmaf(-q0, sf, num), rs, q0);
            // floor(t + 1/2), exactly, by two round-down additions (the second
            // against 1.5 * 2^23 leaves the integer in the low bits), clamped
            // in float: no conversion instructions
            float y = __fadd_rd(__fadd_rd(t, 0.5f), 12582912.f);
            y = fminf(fmaxf(y, 12582912.f), 12582912.f + (float)top);
            const uint32_t q = __float_as_uint(y) & (uint32_t)top;
            // coordinate c = 32 gr + i = 32 (m >> 1) + 4 g + 2 (m & 1) + e
            const int g = (i >> 2) & 7, m = 2 * gr + ((i >> 1) & 1), e = i & 1;
            const int slot = 16 * g + 2 * m + e;
            words[(slot * VB) >> 5] |= q << ((slot * VB) & 31);
        }
    }
#pragma unroll
    for (int k = 0; k < VB; ++k)
        *reinterpret_cast<uint4*>(codes + 16 * k) =
            make_uint4(words[4 * k], words[4 * k + 1], words[4 * k + 2], words[4 * k + 3]);
    *reinterpret_cast<uint4*>(meta) = make_uint4(mw[0], mw[1], mw[2], mw[3]);
}

// 2-D tiled bulk-tensor load: the box at (x, y) of the map into shared memory
// at dst, completing on the mbarrier bar (transaction bytes)
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// KB: key bits; VG: group-32 values (else MSE); VB: value bits.  mk, mv: the
// K and V rows ([vectors][128] bf16) as 2-D maps with 8 x 128 boxes, so that
// box j of a tile lands as chunk column j of the K-major layout.
template <int KB, bool VG, int VB>
__global__ void __launch_bounds__(kTcThreads, 1)
    store_tc_kernel(StoreArgs a, const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Layout& L = a.lay;
    const bool qjl = L.k_qjl;
    const int64_t nvec = a.num_tokens * a.heads;
    const int64_t ntiles = (nvec + 127) / 128;
    float* tab = reinterpret_cast<float*>(smem + TcLayout::tab);
    float* kpb = tab;        // [7] key positive boundaries
    float* kpc = tab + 8;    // [8] key positive centroids
    float* vpb = tab + 16;   // [7] value positive boundaries
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + TcLayout::bars);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + TcLayout::tslot);
    uint32_t* err = a.dp.err;

    // ---- set-up: tables, the rotation operand, T's parts; barriers; tensor memory
    constexpr int kh = 1 << (KB - 1), vh = 1 << (VB - 1);
    if (tid < kh - 1) kpb[tid] = a.dp.k_bound[kh + tid];
    if (tid < kh) kpc[tid] = a.dp.k_cent[kh + tid];
    if (!VG && tid < vh - 1) vpb[tid] = a.dp.v_bound[vh + tid];
    for (int e = tid; e < 2048; e += blockDim.x) {
        // (D H)^T as the B operand of the rotation: row i (output), column j:
        // D_j H_ij, bf16 +-1; T parts: row i (output), column j8.., fp16
        const int i = e & 127, j8 = e >> 7;
        uint32_t wd[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            uint32_t pr = 0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j = 8 * j8 + 2 * u + h;
                const bool neg = (a.dp.signs[j] < 0.f) != (bool)(__popc(i & j) & 1);
                pr |= (uint32_t)(neg ? 0xBF80u : 0x3F80u) << (16 * h);
            }
            wd[u] = pr;
        }
        *reinterpret_cast<uint4*>(smem + TcLayout::mt + tc_chunk(i, j8)) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        if (qjl) {
            *reinterpret_cast<uint4*>(smem + TcLayout::th + tc_chunk(i, j8)) =
                __ldg(reinterpret_cast<const uint4*>(a.dp.t_hi + i * 128 + 8 * j8));
            *reinterpret_cast<uint4*>(smem + TcLayout::tl + tc_chunk(i, j8)) =
                __ldg(reinterpret_cast<const uint4*>(a.dp.t_lo + i * 128 + 8 * j8));
        }
    }
    if (tid == 0) {
        for (int g = 0; g < kTcWG; ++g) {
            uint64_t* b = &bars[kTcBars * g];
            for (int k = 0; k < 4; ++k) mbar_init(smem_u32(&b[k]), 1);  // xfull, ydone, zdone, vdone
            for (int k = 4; k < kTcBars; ++k) mbar_init(smem_u32(&b[k]), 4);  // xfree, tfree, rready[4]
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(tslot, 512);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int g = warp < 4 * kTcWG ? warp >> 2 : warp - 4 * kTcWG;  // this thread's warpgroup
    uint64_t* wb = &bars[kTcBars * g];
    const uint32_t xfull = smem_u32(&wb[0]);   // tile's K and V rows landed (transaction bytes)
    const uint32_t ydone = smem_u32(&wb[1]);   // key rotation MMAs done (commit)
    const uint32_t zdone = smem_u32(&wb[2]);   // projection MMAs done (commit)
    const uint32_t vdone = smem_u32(&wb[3]);   // value rotation MMAs done (commit; MSE values)
    const uint32_t xfree = smem_u32(&wb[4]);   // X_v read by the compute warps (group-32 values; one arrival per warp)
    const uint32_t tfree = smem_u32(&wb[5]);   // tile's tensor memory read (one arrival per warp)
    const uint32_t rready0 = smem_u32(&wb[6]); // + 8 wd: residual parts of word wd in tensor memory (per warp)
    const uint32_t xk_s = smem_u32(smem) + g * TcLayout::x_bytes;
    const uint32_t xv_s = xk_s + 32768;
    // tensor memory of the warpgroup: Y_k in columns 0..127, Y_v in 128..255;
    // word wd of the key residual's fp16 parts (the projection's A operand)
    // goes over Y_k's columns 32 wd .. 32 wd + 31 once they are read (high
    // half first), and the projection z over Y_v
    const uint32_t tcol = tmem + 256u * g;
    const int64_t tstep = (int64_t)gridDim.x * kTcWG;
    bool dead = false;

    if (warp >= 4 * kTcWG) {
        // ------------------------------------------------ MMA and copy issue (lane 0)
        if (lane == 0) {
            const uint32_t id_bf = f16kind_idesc(true), id_h = f16kind_idesc(false);
            const uint32_t mt_s = smem_u32(smem) + TcLayout::mt, th_s = smem_u32(smem) + TcLayout::th,
                           tl_s = smem_u32(smem) + TcLayout::tl;
            int nx = 0, it = 0, ny = 0, nz = 0, nvd = 0;  // loads issued; tiles begun; commits on ydone, zdone, vdone
            auto load_x = [&](int64_t tile) {
                const int y = (int)(tile * 128);
                mbar_expect_tx(xfull, 65536u);
#pragma unroll 1
                for (int j = 0; j < 16; ++j) {
                    tma_load_2d(xk_s + 2048 * j, &mk, 8 * j, y, xfull);
                    tma_load_2d(xv_s + 2048 * j, &mv, 8 * j, y, xfull);
                }
                ++nx;
            };
            int64_t tile = (int64_t)blockIdx.x * kTcWG + g;
            if (tile < ntiles) load_x(tile);
            for (; tile < ntiles && !dead; tile += tstep, ++it) {
                // the compute warps are done with the last tile's tensor memory
                if (it > 0 && (dead = !mbar_wait(tfree, (it - 1) & 1, err))) break;
                if ((dead = !mbar_wait(xfull, it & 1, err))) break;
                tc_fence_after();
                // values first (their encoding starts while the keys rotate)
                if constexpr (!VG) {
#pragma unroll 1
                    for (int s = 0; s < 8; ++s)
                        mma_f16_ss(tcol + 128, tc_desc(xv_s + 4096 * s), tc_desc(mt_s + 4096 * s), id_bf, s > 0);
                    tc_commit(vdone);
                    ++nvd;
                }
#pragma unroll 1
                for (int s = 0; s < 8; ++s)
                    mma_f16_ss(tcol, tc_desc(xk_s + 4096 * s), tc_desc(mt_s + 4096 * s), id_bf, s > 0);
                tc_commit(ydone);
                ++ny;
                // the next tile's rows load once the MMAs (and, for group-32
                // values, the compute warps) have read this one's
                if ((dead = !mbar_wait(ydone, it & 1, err))) break;
                if (VG && (dead = !mbar_wait(xfree, it & 1, err))) break;
                if (tile + tstep < ntiles) load_x(tile + tstep);
                if (!qjl) continue;
                // z = T_hi r_hi + T_hi r_lo + T_lo r_hi, word by word as the
                // compute warps leave the residual's parts in tensor memory
                // (fp16 pairs: K = 16 is 8 columns)
#pragma unroll 1
                for (int wd = 0; wd < 4 && !dead; ++wd) {
                    if ((dead = !mbar_wait(rready0 + 8 * wd, it & 1, err))) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int u = 0; u < 6; ++u) {
                        const int s = 2 * wd + (u & 1), p = u >> 1;  // k-block; product hi.hi, hi.lo, lo.hi
                        const uint32_t acol = tcol + 32 * wd + 8 * (s & 1) + (p == 1 ? 16 : 0);
                        const uint32_t bs = (p < 2 ? th_s : tl_s) + 4096 * s;
                        mma_f16_ts(tcol + 128, acol, tc_desc(bs), id_h, (wd | u) ? 1u : 0u);
                    }
                }
                if (dead) break;
                tc_commit(zdone);
                ++nz;
            }
            // the last commits and copies must land before the CTA's memory is
            // freed (bounded waits, also after a wait above gave up)
            if (nvd > 0) mbar_wait(vdone, (nvd - 1) & 1, err);
            if (ny > 0) mbar_wait(ydone, (ny - 1) & 1, err);
            if (nz > 0) mbar_wait(zdone, (nz - 1) & 1, err);
            if (nx > it) mbar_wait(xfull, (nx - 1) & 1, err);
        }
    } else {
        // --------------------------------------------- compute (thread = row)
        const int v = tid & 127;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t yk = tcol + lane_base, yv = tcol + 128 + lane_base;
        const uint8_t* xv = smem + g * TcLayout::x_bytes + 32768;
        // this row's (slot, head) in tile `tile` (slot -2: no such row), loaded
        // a tile ahead
        auto row_slot = [&](int64_t tile, int& h) -> int64_t {
            const int64_t w = tile * 128 + v;
            h = 0;
            if (w >= nvec) return -2;
            const int64_t t = nvec < ((int64_t)1 << 31) ? (int64_t)((uint32_t)w / (uint32_t)a.heads) : w / a.heads;
            h = (int)(w - t * a.heads);
            return a.slots[t];
        };
        int64_t tile = (int64_t)blockIdx.x * kTcWG + g;
        int h_next = 0;
        int64_t slot_next = tile < ntiles ? row_slot(tile, h_next) : -2;
        for (int it = 0; tile < ntiles; tile += tstep, ++it) {
            const int64_t slot = slot_next;
            const int h = h_next;
            if (tile + tstep < ntiles) slot_next = row_slot(tile + tstep, h_next);
            const bool live = slot != -2;
            const bool ok = live && slot >= 0 && slot < a.num_slots;
            if (live && slot != -1 && !ok && h == 0) set_error(err, TQ_DEVERR_SLOT);
            const int row = (int)(slot & 15);
            uint8_t* page = ok ? a.cache + ((slot >> 4) * a.heads + h) * (int64_t)L.page_bytes : nullptr;

            // ---------------------------------------------------------- value
            if constexpr (VG) {
                // (from shared memory, while the keys rotate)
                if (!dead) dead = !mbar_wait(xfull, it & 1, err);
                if (ok && !dead) g32_row<VB>(xv, v, page + L.v_codes + row * L.v_code_row, page + L.v_meta + row * 16);
                __syncwarp();
                if (lane == 0) mbar_arrive(xfree);
            } else {
                if (!dead) dead = !mbar_wait(vdone, it & 1, err);
                tc_fence_after();
                const float n = mse_planes<VB>(yv, vpb, ok && !dead ? page + L.v_codes : nullptr, row);
                if (ok && !dead) reinterpret_cast<__half*>(page + L.v_meta)[row] = __float2half_rn(n);
            }
            if (!dead) dead = !mbar_wait(ydone, it & 1, err);
            tc_fence_after();

            // ------------------------------------------------------------ key
            {
                constexpr int NB = KB - 1;
                const float n = row_norm128(yk);
                const __half n16 = __float2half_rn(n);
                float T[7], G[8];
                const float sc = n * 11.313708498984761f;
#pragma unroll
                for (int k = 0; k < (1 << NB) - 1; ++k) T[k] = kpb[k] * sc;
                // residual scale 2^(7 - e) for n in [2^(e-1), 2^e): the scaled
                // residual's entries stay well inside fp16's normal range
                int e2 = 0;
                frexpf(n, &e2);
                const float rs = ldexpf(1.f, 7 - e2);
                const float s1 = rs * kTcRsd;
                const float cs = __half2float(n16) * rs;
#pragma unroll
                for (int k = 0; k < (1 << NB); ++k) G[k] = kpc[k] * cs;
                uint8_t* kplanes = ok && !dead ? page + L.k_codes : nullptr;
                const uint32_t nz = n > 0.f ? 0xFFFFFFFFu : 0u;
                Cells<NB> cells;
                cells.init(T, G);
                float rr4[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t KW[KB][4];
                // word wd + 1 loads from tensor memory while word wd is encoded
                uint32_t ybuf[32];
                tmem_ld32(yk, ybuf);
#pragma unroll
                for (int wd = 0; wd < 4; ++wd) {
                    float y[32];
                    tc_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) y[c] = __uint_as_float(ybuf[c]);
                    if (wd < 3) tmem_ld32(yk + 32 * (wd + 1), ybuf);
                    Bits32 S, C[NB];
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int i = 31; i >= 0; --i) {
                        const uint32_t yb = __float_as_uint(y[i]);
                        uint32_t b[3];
                        cells.bits(fabsf(y[i]), b);
                        S.push(i, yb);
#pragma unroll
                        for (int q = 0; q < NB; ++q) C[q].push01(i, b[q]);
                        // -n16 rs c[idx]: c[idx] = +G[cnt] for y > 0, -G[cnt]
                        // otherwise, i.e. -c takes the sign bit of y flipped
                        const float cneg = __uint_as_float(cells.centroid(b) ^ (~yb & 0x80000000u));
                        y[i] = fmaf(y[i], s1, cneg);  // the scaled rotated residual
                        rr4[i & 3] = fmaf(y[i], y[i], rr4[i & 3]);
                    }
                    if (qjl) {
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const __half2 hh = __floats2half2_rn(y[2 * u], y[2 * u + 1]);
                            const float2 hf = __half22float2(hh);
                            const __half2 ll = __floats2half2_rn(y[2 * u] - hf.x, y[2 * u + 1] - hf.y);
                            hi[u] = *reinterpret_cast<const uint32_t*>(&hh);
                            lo[u] = *reinterpret_cast<const uint32_t*>(&ll);
                        }
                        tmem_st16(yk + 32 * wd, hi);
                        tmem_st16(yk + 32 * wd + 16, lo);
                        tc_wait_st();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(rready0 + 8 * wd);  // this warp's rows of word wd
                    }
                    const uint32_t pos = ~S.word() & nz;  // [y > 0]
                    KW[KB - 1][wd] = pos;
#pragma unroll
                    for (int q = 0; q < NB; ++q) KW[q][wd] = C[q].word() ^ ~pos;
                }
                if (kplanes) {
#pragma unroll
                    for (int p = 0; p < KB; ++p)
                        *reinterpret_cast<uint4*>(kplanes + (p * kBlock + row) * 16) =
                            make_uint4(KW[p][0], KW[p][1], KW[p][2], KW[p][3]);
                }
                if (ok && !dead) reinterpret_cast<__half*>(page + L.k_norm)[row] = n16;
                if (qjl) {
                    if (!dead) dead = !mbar_wait(zdone, it & 1, err);
                    tc_fence_after();
                    uint32_t sw[4];
                    uint32_t zbuf[32];
                    tmem_ld32(yv, zbuf);
#pragma unroll
                    for (int wd = 0; wd < 4; ++wd) {
                        uint32_t z[32];
                        tc_wait_ld();
#pragma unroll
                        for (int c = 0; c < 32; ++c) z[c] = zbuf[c];
                        if (wd < 3) tmem_ld32(yv + 32 * (wd + 1), zbuf);
                        Bits32 neg;
#pragma unroll
                        for (int i = 31; i >= 0; --i) neg.push(i, z[i]);
                        sw[wd] = ~neg.word();  // bit j = [z_j >= 0]
                    }
                    if (ok && !dead) {
                        *reinterpret_cast<uint4*>(page + L.k_signs + row * 16) = make_uint4(sw[0], sw[1], sw[2], sw[3]);
                        const float rr = (rr4[0] + rr4[1]) + (rr4[2] + rr4[3]);
                        reinterpret_cast<__half*>(page + L.k_rnorm)[row] = __float2half_rn(sqrtf(rr) / rs);
                    }
                }
            }
            // this warp's rows of the tile's tensor memory are read
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tfree);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// The driver's tensor-map encoder: from the runtime's entry-point query, else
// the driver library's own export; looked up under a lock until found.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder(char* why, size_t why_len) {
    static std::mutex mu;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (fn) return fn;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess) p = nullptr;
    if (!p) {
        if (void* h = dlopen("libcuda.so.1", RTLD_NOW | RTLD_LOCAL)) p = dlsym(h, "cuTensorMapEncodeTiled");
    }
    if (!p) {
        snprintf(why, why_len, "cuTensorMapEncodeTiled not found (entry-point query: %s, result %d; libcuda.so.1: %s)",
                 cudaGetErrorName(e), (int)q, dlerror() ? "no symbol" : "not loaded");
        return nullptr;
    }
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return fn;
}

// rows [n][128] bf16 at base as a 2-D map with 8 x 128 boxes (zero fill past n)
static tq_status rows_map(CUtensorMap* m, const void* base, int64_t n) {
    char why[200] = "";
    auto enc = tensor_map_encoder(why, sizeof why);
    if (!enc) return driver_failure("%s", why);
    // the encoder wants a current context: a host thread whose first call this
    // is has none until the runtime binds the device's primary context
    static thread_local bool bound = false;
    if (!bound) {
        int dev = 0;
        const tq_status st = cuda_status_detail(cudaGetDevice(&dev), "binding the device context");
        if (st == TQ_OK) bound = cuda_status_detail(cudaSetDevice(dev), "binding the device context") == TQ_OK;
        if (!bound) return TQ_ERR_CUDA;
    }
    const cuuint64_t dims[2] = {128, (cuuint64_t)n};
    const cuuint64_t strides[1] = {256};
    const cuuint32_t box[2] = {8, 128};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return driver_failure("cuTensorMapEncodeTiled failed (CUresult %d) for rows at %p, n = %lld", (int)r, base,
                              (long long)n);
    return TQ_OK;
}

template <int KB, bool VG, int VB>
static tq_status launch_tc(const StoreArgs& a, cudaStream_t s, int sms) {
    auto kern = store_tc_kernel<KB, VG, VB>;
    const tq_status fs = ensure_dynamic_smem((const void*)kern, (int)TcLayout::total, "store_tc_kernel");
    if (fs != TQ_OK) return fs;
    const int64_t nvec = a.num_tokens * a.heads;
    CUtensorMap mk, mv;
    tq_status ms = rows_map(&mk, a.k, nvec);
    if (ms == TQ_OK) ms = rows_map(&mv, a.v, nvec);
    if (ms != TQ_OK) return ms;
    const int64_t tiles = (nvec + 127) / 128;
    const int grid = (int)std::min<int64_t>((tiles + kTcWG - 1) / kTcWG, (int64_t)sms);
    kern<<<grid, kTcThreads, TcLayout::total, s>>>(a, mk, mv);
    return cuda_status(cudaGetLastError());
}

template <int KB>
static tq_status launch_tc_v(const StoreArgs& a, cudaStream_t s, int sms) {
    if (a.lay.v_mode == TQ_V_G32) return a.lay.v_bits == 4 ? launch_tc<KB, true, 4>(a, s, sms)
                                                            : launch_tc<KB, true, 2>(a, s, sms);
    switch (a.lay.v_bits) {
        case 2: return launch_tc<KB, false, 2>(a, s, sms);
        case 3: return launch_tc<KB, false, 3>(a, s, sms);
        default: return launch_tc<KB, false, 4>(a, s, sms);
    }
}

tq_status launch_store_tc(const StoreArgs& a, cudaStream_t s, int sms) {
    switch (a.lay.k_bits) {
        case 2: return launch_tc_v<2>(a, s, sms);
        case 3: return launch_tc_v<3>(a, s, sms);
        default: return launch_tc_v<4>(a, s, sms);
    }
}

}  // namespace tq
