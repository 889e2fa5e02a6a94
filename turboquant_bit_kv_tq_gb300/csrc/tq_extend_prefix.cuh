// Extend attention's compressed prefix as a tensor-core GEMM (head dim 128;
// included by the tq_extend_prefix_*.cu translation units).
//
// [Roadmap] §4.1: in an extend (prefill) call every new token attends to its
// sequence's whole compressed prefix, so the new tokens of a chunk share every
// prefix tile.  A work item is one query block (up to 8 consecutive new tokens
// of one sequence, one head group of four query heads: 32 query heads), one
// KV head and one prefix split.  The CTA streams the split as 128-token tiles
// and contracts each tile against all 32 query heads at once:
//   scores   the decode's fp8 bit-plane contraction (key code planes and the
//            QJL sign plane as exact e4m3 A operands in tensor memory), with
//            the block's 8 query operand images stacked along N: one tcgen05
//            MMA per 32-byte K step covers N = 8 x 16 = 128 columns
//   softmax  online exp2 per query head with one lazily moved reference per
//            head for the whole CTA (a tile maximum across the 4 consumer
//            warps); rescaling the output accumulator in tensor memory is rare
//   P V      a second tcgen05 contraction, D[128 coordinates x 64] in
//            tensor memory: A = the tile's dequantised values (bf16 high and
//            low parts, MN-major: token-major rows as the thread that owns a
//            token writes them), B = [P_hi | P_lo], the probabilities' bf16
//            high and low parts side by side (MN-major, N = 64); the two
//            column halves add up at the end; fp32 accumulation
// Every (new token, query head) of the item gets the split's partial
// (m, l, acc) in the decode's workspace format, which the combine merges with
// the exact causal part (chunk_attn_kernel).
//
// Roles (384 threads, one CTA per SM, all 512 tensor-memory columns):
//   warps 0-3  thread t = token t of the tile: key bit-plane operands of the
//              next tile into tensor memory, then the token's dequantised
//              value row of this tile into shared memory
//   warps 4-7  same token mapping: scores out of tensor memory, softmax,
//              probability operands; at an item's end the output accumulator
//              (lane = coordinate) becomes the partial
//   warp 8     bulk async copies of the pages (ring of stages) and of the
//              block's query operand images
//   warp 9     one thread issues the MMAs: the scores of tile i + 1, then
//              the P V of tile i
//   warps 10-11 idle (they complete the third warpgroup's register split)
#pragma once

#include "tq_decode_ws.cuh"

namespace tq {

constexpr int kXpImgs = 8;                 // query operand images per item (16 columns each)
constexpr int kXpHeads = 4 * kXpImgs;      // query heads per item
constexpr int kXpCols = 16 * kXpImgs;      // score accumulator columns (key | sign each)
constexpr int kXpThreads = 384;           // score/value, consumer and copy/MMA warpgroups
constexpr int kXpStages = 3;
// setmaxnreg split of the 3 x 168 registers per thread a CTA launches with:
// the copy/MMA warpgroup keeps 56, the two compute warpgroups take 224 each
constexpr int kXpRegsLaunch = 168, kXpRegsIssue = 56, kXpRegsWork = (3 * kXpRegsLaunch - kXpRegsIssue) / 2;
constexpr int kXpMaxItems = 64;            // items per CTA at most (the launch sizes the grid for it)
constexpr int kXpTmemCols = 512;
constexpr int kXpColA = 2 * kXpCols;       // A operand: npl planes x 32 columns
constexpr int kXpColO = 448;               // P V accumulator: 64 columns (probability high | low part)
constexpr int kXpTileTok = kTilePages * kBlock;  // 128 prefix tokens per tile
constexpr int kXpVBytes = kXpTileTok * 128 * 2;  // one bf16 piece of the value operand
constexpr int kXpPBytes = kXpTileTok * kXpHeads * 2;  // one bf16 piece of the probability operand

// Byte offset of the 16-byte row (token t, 8-element group c) in the MN-major
// no-swizzle layout of a [128 tokens x 8 ng elements] 16-bit operand: core
// matrices of 8 tokens x 8 elements (128 B, tokens 16 B apart), the ng
// element groups of 8 tokens side by side (128 B apart), blocks of 8 tokens
// ng * 128 B apart.  The tensor cores read a K step's groups as one
// contiguous run.
__host__ __device__ constexpr uint32_t xp_mn_off(int t, int c, int ng) {
    return (uint32_t)(t >> 3) * (uint32_t)(ng * 128) + (uint32_t)c * 128u + (uint32_t)(t & 7) * 16u;
}

// MN-major shared-memory descriptor of such an operand.  For MN-major
// operands without swizzling the leading-byte-offset field holds the step
// between K-adjacent core matrices (ng * 128 B here) and the stride-byte-offset
// field the step between MN-adjacent ones (128 B), the reverse of their
// K-major roles (measured: of the four assignments for A and B only this one
// reproduces an integer-valued product).
__device__ __forceinline__ uint64_t xp_mn_desc(uint32_t addr, int ng) {
    return smem_desc(addr, (uint32_t)(128 * ng), 128);
}
constexpr int kXpVGroups = 16;  // value operand: 128 coordinates
constexpr int kXpPGroups = 8;   // probability operand: 32 heads high | 32 heads low

// kind::f16 instruction descriptor: fp32 accumulation, bf16 A and B, both
// MN-major, M = 128, N = n
__host__ __device__ constexpr uint32_t xp_pv_idesc(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) | ((uint32_t)(n >> 3) << 17) |
           ((128u >> 4) << 24);
}

// D[128 x N] (+)= A[128 x 16] B[16 x N], both operands in shared memory
__device__ __forceinline__ void xp_mma_ss(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

// generic-proxy shared-memory writes become visible to the tensor cores
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

struct XpItem {
    int b, g, hgi, c;       // sequence, KV head, head group, prefix split
    int t0, n;              // the block's first new token (entry) and its entry count
    int p0, n_pages, n_tiles;
    int tok0, tok1;         // prefix tokens [tok0, tok1) of the split
    int load, lidx, release;  // image load of this item (and its index), release after it
};

struct XpLayout {
    size_t img, ring, vhi, vlo, phi, plo, tile, vcent, icst, red, items, smask, bars, tslot, total;
};

__host__ __device__ inline XpLayout xp_layout(int page_bytes, int bimg_bytes) {
    auto up = [](size_t x) { return (x + 127) & ~(size_t)127; };
    XpLayout l;
    size_t off = 0;
    l.tile = up((size_t)kTilePages * page_bytes);
    l.vhi = off;
    off = up(off + kXpVBytes);
    l.vlo = off;
    off = up(off + kXpVBytes);
    l.phi = off;
    off = up(off + kXpPBytes);
    l.plo = off;
    off = up(off + kXpPBytes);
    l.img = off;
    off = up(off + (size_t)kXpImgs * bimg_bytes);
    l.ring = off;
    off = up(off + (size_t)kXpStages * l.tile);
    l.vcent = off;
    off = up(off + 16 * 4);
    l.icst = off;
    off = up(off + (size_t)kXpHeads * 4 * 4);
    l.red = off;  // [2][4][32] tile maxima (double-buffered), [4][32] row sums
    off = up(off + (size_t)3 * 4 * kXpHeads * 4);
    l.items = off;
    off = up(off + (size_t)kXpMaxItems * sizeof(XpItem));
    l.smask = off;
    off = up(off + (size_t)kXpStages * 4);
    l.bars = off;
    off = up(off + (size_t)(2 * kXpStages + 11) * 8);
    l.tslot = off;
    off = up(off + 16);
    l.total = off;
    return l;
}

// A configuration runs on the prefix kernel when its head groups are full
// groups of 4 query heads (one 16-column image each) and all its score
// planes fit the A operand columns.
inline bool xp_supported(const DecodeGeom& gm, int d) {
    return d == 128 && gm.hc == 4 && gm.nth == 1 && gm.n_cols == 16 && gm.npl * (d / 4) <= kXpColO - kXpColA;
}

// new tokens per query block: one query image per token and head group, and
// an item takes one head group, so a block of kXpImgs tokens fills the
// item's kXpImgs images whatever the group size
__host__ __device__ inline int xp_block_tokens() { return kXpImgs; }

// the prefix kernels of one key configuration (all value modes), compiled in
// their own translation units: KB-bit keys, KU = uniform codebook with its KB
// single-bit planes only
template <int KB, bool KU>
tq_status dispatch_extend_prefix(const DecodeArgs& a, cudaStream_t s, int grid);

// (x, y) as bf16 high parts (the top 16 bits of each fp32 value) and bf16
// low parts (the top 16 bits of the exact remainders): ~16 significant bits
// together, from logic operations and byte permutes (no conversions)
__device__ __forceinline__ void xp_split2(float x, float y, uint32_t& hi, uint32_t& lo) {
    const uint32_t xb = __float_as_uint(x), yb = __float_as_uint(y);
    hi = __byte_perm(xb, yb, 0x7632u);
    const float lx = x - __uint_as_float(xb & 0xFFFF0000u);
    const float ly = y - __uint_as_float(yb & 0xFFFF0000u);
    lo = __byte_perm(__float_as_uint(lx), __float_as_uint(ly), 0x7632u);
}

// bf16 high and low parts of eight values, as the two 16-byte operand rows
__device__ __forceinline__ void xp_store8(uint8_t* vh, uint8_t* vl, uint32_t off, const float (&v)[8]) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) xp_split2(v[2 * u], v[2 * u + 1], h[u], l[u]);
    *reinterpret_cast<uint4*>(vh + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(vl + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

// Dequantised value row of page row r (token t of the tile), coordinates
// 64 ch .. 64 ch + 63, into the value operand: element group c holds
// coordinates 8c .. 8c + 7.  Group-32 values:
// v = zero + scale * code in fp32 (the product is exact; one rounding), with
// the code read as 2^23 + code * 2^(w*n) from the float bits (w-bit field n of
// a 16-bit window) and the 2^(-w*n) folded into the scale; the field of
// coordinate 32M + 4g + 2m' + e is slot 16g + 4M + 2m' + e of the row (the
// cache's group-32 order), so the 8 coordinates of group c sit in two
// neighbouring 16-bit (4-bit codes) or 8-bit (2-bit codes) windows.  MSE
// values: v = norm * centroid[code] in the rotated space, the code's bits
// from the bit planes.  A row that is not a valid token gets zeros.
template <bool G32, int VB>
__device__ __forceinline__ void xp_value_row(const uint8_t* pg, int r, bool valid, const Layout& L,
                                             const float* vcent, uint8_t* vh, uint8_t* vl, int t, int ch) {
    constexpr int D = 128;
    constexpr float kMagic = 8388608.f;  // 2^23
    // loops over groups are not unrolled: this code shares the instruction
    // cache with the consumers' and is short that way
    if constexpr (G32) {
        constexpr int NWD = D * VB / 32;  // 32-bit words of the code row
        uint32_t w[NWD];
        const uint8_t* row = pg + L.v_codes + r * L.v_code_row;
#pragma unroll
        for (int q = 0; q < NWD / 4; ++q) {
            const uint4 u = *reinterpret_cast<const uint4*>(row + 16 * q);
            w[4 * q] = u.x;
            w[4 * q + 1] = u.y;
            w[4 * q + 2] = u.z;
            w[4 * q + 3] = u.w;
        }
        const uint32_t* meta = reinterpret_cast<const uint32_t*>(pg + L.v_meta + r * L.v_meta_row);
#pragma unroll 1
        for (int M = 2 * ch; M < 2 * ch + 2; ++M) {
            const uint32_t mw = meta[M];
            const float2 sz = __half22float2(*reinterpret_cast<const __half2*>(&mw));
            const float s = valid ? sz.x : 0.f, z = valid ? sz.y : 0.f;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int c = 4 * M + jj;
                float v[8];
                if constexpr (VB == 4) {
                    const bool odd = (M & 1) != 0, up = M >= 2;
                    const uint32_t wa = up ? w[4 * jj + 1] : w[4 * jj];
                    const uint32_t wb = up ? w[4 * jj + 3] : w[4 * jj + 2];
                    const uint32_t x = __byte_perm(wa, wb, odd ? 0x7632u : 0x5410u);
                    const uint32_t xh = x >> 16;
#pragma unroll
                    for (int n = 0; n < 4; ++n) {
                        const float sn = s * (1.f / (float)(1 << (4 * n)));
                        const float f0 = __uint_as_float(0x4B000000u | (x & (0xFu << (4 * n)))) - kMagic;
                        const float f1 = __uint_as_float(0x4B000000u | (xh & (0xFu << (4 * n)))) - kMagic;
                        v[n] = fmaf(f0, sn, z);
                        v[4 + n] = fmaf(f1, sn, z);
                    }
                } else {
                    const uint32_t x = __byte_perm(w[2 * jj], w[2 * jj + 1], (uint32_t)(M | ((4 + M) << 4)));
#pragma unroll
                    for (int n = 0; n < 8; ++n) {
                        const float sn = s * (1.f / (float)(1 << (2 * n)));
                        const float f = __uint_as_float(0x4B000000u | (x & (0x3u << (2 * n)))) - kMagic;
                        v[n] = fmaf(f, sn, z);
                    }
                }
                xp_store8(vh, vl, xp_mn_off(t, c, kXpVGroups), v);
            }
        }
    } else {
        const float nv = valid ? __half2float(*reinterpret_cast<const __half*>(pg + L.v_meta + 2 * r)) : 0.f;
#pragma unroll 1
        for (int cw4 = 2 * ch; cw4 < 2 * ch + 2; ++cw4) {
            uint32_t pw[VB];
#pragma unroll
            for (int pp = 0; pp < VB; ++pp)
                pw[pp] = *reinterpret_cast<const uint32_t*>(pg + L.v_codes + (pp * kBlock + r) * (D / 8) + 4 * cw4);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                float v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    uint32_t code = 0;
#pragma unroll
                    for (int pp = 0; pp < VB; ++pp) code |= ((pw[pp] >> (8 * cc + q)) & 1u) << pp;
                    v[q] = nv * vcent[code];
                }
                xp_store8(vh, vl, xp_mn_off(t, 4 * cw4 + cc, kXpVGroups), v);
            }
        }
    }
}

// The CTA's items [first, first + nk) from the block plan: blocks[k] =
// {first entry, entries, sequence, index of the block's first item}, items of
// a block ordered split fastest, then head group, then KV head.  Run by one
// thread.  Returns the item count.
__device__ inline int xp_items(const DecodeArgs& a, XpItem* items, int cta, int grid) {
    const int n_blocks = a.xcounts[0], n_items = a.xcounts[1];
    const int per = (n_items + grid - 1) / grid;
    const int first = cta * per;
    int nk = max(0, min(per, n_items - first));
    if (nk > kXpMaxItems) {
        // more items than the plan's bound allows (only an overlapping,
        // already flagged cu_q gets here): the rest are left out
        set_error(a.dp.err, TQ_DEVERR_CHUNK);
        nk = kXpMaxItems;
    }
    if (nk == 0) return 0;
    // last block whose first item is <= first
    int lo = 0, hi = n_blocks - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.xblocks[mid].w <= first) lo = mid; else hi = mid - 1;
    }
    int k = lo;
    int4 blk = a.xblocks[k];
    const int hn = a.heads * a.gm.nhg, ST = a.split_blocks * kBlock, maxlen = a.max_blocks * kBlock;
    // prefix length of a block's sequence (the entries' compressed length)
    auto len_of = [&](const int4& bk) { return max(0, min(a.seq_lens[bk.x], maxlen)); };
    int ns = (len_of(blk) + ST - 1) / ST;
    int idx = first - blk.w;
    for (int i = 0; i < nk; ++i) {
        while (idx >= hn * ns && k + 1 < n_blocks) {
            idx -= hn * ns;
            blk = a.xblocks[++k];
            ns = (len_of(blk) + ST - 1) / ST;
        }
        XpItem it;
        it.b = blk.z;
        it.t0 = blk.x;
        it.n = blk.y;
        it.c = ns > 0 ? idx % ns : 0;
        const int gh = ns > 0 ? idx / ns : 0;
        it.hgi = gh % a.gm.nhg;
        it.g = gh / a.gm.nhg;
        const int len = len_of(blk);
        it.tok0 = it.c * ST;
        it.tok1 = min(len, it.tok0 + ST);
        it.p0 = it.c * a.split_blocks;
        it.n_pages = it.tok1 > it.tok0 ? (it.tok1 - it.tok0 + kBlock - 1) / kBlock : 0;
        it.n_tiles = (it.n_pages + kTilePages - 1) / kTilePages;
        it.load = it.lidx = it.release = 0;
        items[i] = it;
        ++idx;
    }
    // image loads: one per run of items of the same (block, KV head, head group)
    int nload = 0, last = -1;
    for (int i = 0; i < nk; ++i) {
        XpItem& it = items[i];
        if (it.n_tiles == 0) continue;
        const bool same = last >= 0 && items[last].t0 == it.t0 && items[last].g == it.g && items[last].hgi == it.hgi;
        if (!same) {
            if (last >= 0) items[last].release = 1;
            it.load = 1;
            it.lidx = nload++;
        }
        last = i;
    }
    return nk;
}

template <int KB, bool KU, bool G32, int VB>
__global__ void __launch_bounds__(kXpThreads, 1) extend_prefix_kernel(DecodeArgs a) {
    static_assert(kXpRegsWork <= 256 && kXpRegsWork % 8 == 0, "register split");
    constexpr int D = 128;
    constexpr int NPK = KU ? KB : 1 << (KB - 1);
    constexpr int NW = D / 32;
    constexpr int NCOL = D / 4;
    extern __shared__ __align__(16) uint8_t smem[];
    const Layout& L = a.lay;
    const DecodeGeom gm = a.gm;
    const int npl = NPK + (L.k_qjl ? 1 : 0);
    const XpLayout sl = xp_layout(L.page_bytes, gm.bimg_bytes);
    constexpr int S = kXpStages;
    uint8_t* ring = smem + sl.ring;
    uint8_t* img = smem + sl.img;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + sl.bars);
    uint64_t* full = bars;                // [S] pages landed (tx)
    uint64_t* empty = bars + S;           // [S] pages read (4 score + 4 consumer warps)
    uint64_t* ifull = bars + 2 * S;       // query images landed (tx)
    uint64_t* ifree = ifull + 1;          // query images released (MMA commit)
    uint64_t* aready = ifull + 2;         // key operands stored (4 score warps)
    uint64_t* mdone = ifull + 3;          // score MMAs done (commit)
    uint64_t* dfree = ifull + 4;          // scores read (4 consumer warps)
    // the value operand and its P V go in two token halves (tokens 0-63, 64-127)
    uint64_t* vready = ifull + 5;         // [half] value operands stored (4 score warps)
    uint64_t* pready = ifull + 7;         // probability operands stored (4 consumer warps)
    uint64_t* pvdone = ifull + 8;         // [half] P V MMAs of the half done (commit; half 1: all)
    uint64_t* oread = ifull + 10;         // output accumulator read (4 consumer warps)
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + sl.tslot);
    XpItem* items = reinterpret_cast<XpItem*>(smem + sl.items);
    uint32_t* smask = reinterpret_cast<uint32_t*>(smem + sl.smask);
    float* vcent = reinterpret_cast<float*>(smem + sl.vcent);
    float* icst = reinterpret_cast<float*>(smem + sl.icst);  // [32 heads][4]
    float* red = reinterpret_cast<float*>(smem + sl.red);
    int* nk_slot = reinterpret_cast<int*>(smem + sl.tslot) + 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint32_t* err = a.dp.err;
    auto B = [&](const uint64_t* p) { return smem_u32(p); };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(B(&full[s]), 1);
            mbar_init(B(&empty[s]), 8);
        }
        mbar_init(B(ifull), 1);
        mbar_init(B(ifree), 1);
        mbar_init(B(aready), 4);
        mbar_init(B(mdone), 1);
        mbar_init(B(dfree), 4);
        for (int h = 0; h < 2; ++h) {
            mbar_init(B(&vready[h]), 4);
            mbar_init(B(&pvdone[h]), 1);
        }
        mbar_init(B(pready), 4);
        mbar_init(B(oread), 4);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid == 32 * 8) *nk_slot = xp_items(a, items, blockIdx.x, gridDim.x);
    if (tid < 16) vcent[tid] = G32 ? 0.f : a.dp.v_cent[tid];
    if (warp == 0) tmem_alloc(tslot, kXpTmemCols);
    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const int nk = *nk_slot;
    const uint32_t tmem = *tslot;
    pdl_wait();  // the query prep's images and constants
    bool dead = false;
    const int hc = gm.hc;

    if (warp >= 8) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kXpRegsIssue));
        if (warp == 8) {
            // -------------------------------------------------- producer
            int tseq = 0, nimg = 0;
            auto wait_uniform = [&](uint64_t* bar, uint32_t par) {
                int ok = 1;
                if (lane == 0 && !dead) ok = mbar_wait(B(bar), par, err);
                dead = dead || __shfl_sync(0xffffffffu, ok, 0) == 0;
            };
            for (int k = 0; k < nk && !dead; ++k) {
                const XpItem it = items[k];
                if (it.n_tiles == 0) continue;
                if (it.load) {
                    if (it.lidx >= 1) wait_uniform(ifree, (it.lidx - 1) & 1);
                    if (dead) break;
                    if (lane == 0) mbar_expect_tx(B(ifull), (uint32_t)(it.n * gm.bimg_bytes));
                    __syncwarp();
                    if (lane < it.n)
                        bulk_copy(smem_u32(img + (size_t)lane * gm.bimg_bytes),
                                  a.ws_bimg +
                                      (((int64_t)(it.t0 + lane) * a.heads + it.g) * gm.nhg + it.hgi) * gm.bimg_bytes,
                                  gm.bimg_bytes, B(ifull));
                    ++nimg;
                }
                for (int t = 0; t < it.n_tiles && !dead; ++t, ++tseq) {
                    const int s = tseq % S;
                    if (tseq >= S) wait_uniform(&empty[s], ((tseq / S) - 1) & 1);
                    if (dead) break;
                    const int p0 = t * kTilePages, np = min(kTilePages, it.n_pages - p0);
                    int blk = -1;
                    if (lane < np) blk = a.block_table[(int64_t)it.b * a.max_blocks + it.p0 + p0 + lane];
                    const bool ok = lane < np && blk >= 0 && blk < a.num_blocks;
                    const uint32_t mask = __ballot_sync(0xffffffffu, ok);
                    if (lane < np && !ok) set_error(err, TQ_DEVERR_BLOCK);
                    if (lane == 0) {
                        smask[s] = mask;
                        mbar_expect_tx(B(&full[s]), (uint32_t)__popc(mask) * L.page_bytes);
                    }
                    __syncwarp();
                    if (ok)
                        bulk_copy(smem_u32(ring + s * sl.tile + (size_t)lane * L.page_bytes),
                                  a.cache + ((int64_t)blk * a.heads + it.g) * L.page_bytes, L.page_bytes, B(&full[s]));
                }
            }
            // copies still in flight must land before the block exits
            if (lane == 0) {
                bool d2 = false;
                for (int k = max(0, tseq - S); k < tseq; ++k) ws_wait(B(&full[k % S]), (k / S) & 1, d2, err);
                if (nimg > 0) ws_wait(B(ifull), (nimg - 1) & 1, d2, err);
            }
        } else if (warp == 9 && lane == 0) {
            // ----------------------------------------------- MMA issue
            const uint32_t idesc_s = fp8_idesc(kXpCols);
            const uint32_t idesc_pv = xp_pv_idesc(2 * kXpHeads);
            const uint32_t sbo = 8u * (uint32_t)(npl * D);
            const uint32_t vhi = smem_u32(smem + sl.vhi), vlo = smem_u32(smem + sl.vlo);
            const uint32_t pb = smem_u32(smem + sl.phi);  // [P_hi | P_lo]: 8 column groups
            const uint32_t dO = tmem + kXpColO;
            int tseq = 0, ki = 0;
            int pv_t = -1, pv_first = 0, pv_item = 0;  // the tile whose P V is still to issue
            auto issue_pv = [&]() {
                ws_wait(B(pready), pv_t & 1, dead, err);
                if (pv_first && pv_item >= 1) ws_wait(B(oread), (pv_item - 1) & 1, dead, err);
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    ws_wait(B(&vready[h]), pv_t & 1, dead, err);
                    tc_fence_after();
#pragma unroll 1
                    for (int kk = 4 * h; kk < 4 * h + 4; ++kk) {
                        // K step kk: tokens 16 kk .. 16 kk + 15, two blocks of 8
                        const uint64_t bd = xp_mn_desc(pb + 2 * 128 * kXpPGroups * kk, kXpPGroups);
                        const uint32_t ao = 2 * 128 * kXpVGroups * kk;
                        xp_mma_ss(dO, xp_mn_desc(vhi + ao, kXpVGroups), bd, idesc_pv, (pv_first && kk == 0) ? 0u : 1u);
                        xp_mma_ss(dO, xp_mn_desc(vlo + ao, kXpVGroups), bd, idesc_pv, 1u);
                    }
                    tc_commit(B(&pvdone[h]));
                }
            };
            for (int k = 0; k < nk; ++k) {
                const XpItem it = items[k];
                if (it.n_tiles == 0) continue;
                if (it.load) ws_wait(B(ifull), it.lidx & 1, dead, err);
                const uint64_t bd0 = smem_desc(smem_u32(img), 128, sbo);
                for (int t = 0; t < it.n_tiles; ++t, ++tseq) {
                    ws_wait(B(aready), tseq & 1, dead, err);
                    if (tseq >= 1) ws_wait(B(dfree), (tseq - 1) & 1, dead, err);
                    tc_fence_after();
                    ws_issue_planes<D, NPK, kXpCols, kXpColA>(0, npl, tmem, bd0, idesc_s);
                    tc_commit(B(mdone));
                    if (t == it.n_tiles - 1 && it.release) tc_commit(B(ifree));
                    if (pv_t >= 0) issue_pv();
                    pv_t = tseq;
                    pv_first = t == 0;
                    pv_item = ki;
                }
                ++ki;
            }
            if (pv_t >= 0) issue_pv();
        }
    } else if (warp < 4) {
        // ------------------------------------- key and value operands
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kXpRegsWork));
        const int pj = tid >> 4, r = tid & 15;
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        const bool qjl = L.k_qjl;
        uint8_t* vh = smem + sl.vhi;
        uint8_t* vl = smem + sl.vlo;
        // the key operands of tile u (item k, tile t of it): they go into the
        // single A buffer once the score MMAs of tile u - 1 are done
        auto key_operands = [&](int u, int t) {
            const int s = u % S;
            ws_wait(B(&full[s]), (u / S) & 1, dead, err);
            const uint8_t* pg = ring + s * sl.tile + pj * L.page_bytes;
            uint32_t kw[KB][NW], sw[NW];
#pragma unroll
            for (int p = 0; p < KB; ++p) {
                const uint4 v4 = *reinterpret_cast<const uint4*>(pg + L.k_codes + (p * kBlock + r) * (D / 8));
                kw[p][0] = v4.x;
                kw[p][1] = v4.y;
                kw[p][2] = v4.z;
                kw[p][3] = v4.w;
            }
            {
                uint4 v4 = make_uint4(0u, 0u, 0u, 0u);
                if (qjl) v4 = *reinterpret_cast<const uint4*>(pg + L.k_signs + r * (D / 8));
                sw[0] = v4.x;
                sw[1] = v4.y;
                sw[2] = v4.z;
                sw[3] = v4.w;
            }
            (void)t;
            if (u >= 1) ws_wait(B(mdone), (u - 1) & 1, dead, err);  // A operand free
            tc_fence_after();
            const uint32_t abase = tmem + lane_base + kXpColA;
#pragma unroll 1
            for (int P = 0; P < npl; ++P) {
                // plane P < NPK: XOR of the code bits in subset P; P = NPK: signs
                const uint32_t sub = P < NPK ? (uint32_t)plane_subset(KB, P) : 0u;
                uint32_t a32[32];
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    uint32_t x = P < NPK ? 0u : sw[w];
#pragma unroll
                    for (int p = 0; p < KB; ++p) x ^= ((sub >> p) & 1u) ? kw[p][w] : 0u;
                    a32[8 * w + 0] = bit_operand<0>(x);
                    a32[8 * w + 1] = bit_operand<1>(x);
                    a32[8 * w + 2] = bit_operand<2>(x);
                    a32[8 * w + 3] = bit_operand<3>(x);
                    a32[8 * w + 4] = bit_operand<4>(x);
                    a32[8 * w + 5] = bit_operand<5>(x);
                    a32[8 * w + 6] = bit_operand<6>(x);
                    a32[8 * w + 7] = bit_operand<7>(x);
                }
                tmem_st32(abase + P * NCOL, a32);
            }
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B(aready));
        };
        // tiles in order; the key operands of the next tile go before the
        // values of this one, so that the next score MMAs overlap the value
        // expansion and the P V of this tile
        int k = 0, t = 0, u = 0;
        while (k < nk && items[k].n_tiles == 0) ++k;
        if (k < nk) key_operands(0, 0);
        while (k < nk) {
            const XpItem it = items[k];
            int k2 = k, t2 = t + 1;
            if (t2 == it.n_tiles) {
                t2 = 0;
                ++k2;
                while (k2 < nk && items[k2].n_tiles == 0) ++k2;
            }
            if (k2 < nk) key_operands(u + 1, t2);
            // the tile's value rows, dequantised, as bf16 high and low parts:
            // tokens 0-63, then 64-127, two threads per token (coordinate
            // halves ch), so that the first half's P V overlaps the second's
            const int s = u % S;
            const int np = min(kTilePages, it.n_pages - t * kTilePages);
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                const int tok = 64 * h + (tid >> 1), ch = tid & 1;
                const int pj2 = tok >> 4, r2 = tok & 15;
                const int pos = it.tok0 + (t * kTilePages + pj2) * kBlock + r2;
                const bool valid = pj2 < np && pos < it.tok1 && ((smask[s] >> pj2) & 1);
                const uint8_t* pg = ring + s * sl.tile + pj2 * L.page_bytes;
                if (u >= 1) ws_wait(B(&pvdone[h]), (u - 1) & 1, dead, err);  // this half of the operand free
                xp_value_row<G32, VB>(pg, r2, valid, L, vcent, vh, vl, tok, ch);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(B(&vready[h]));
            }
            if (lane == 0) mbar_arrive(B(&empty[s]));
            k = k2;
            t = t2;
            ++u;
        }
    } else {
        // ------------------------------------------------------ consumers
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kXpRegsWork));
        const int ctid = tid - 128, cw = warp - 4;
        const int pj = ctid >> 4, r = ctid & 15;
        const uint32_t lane_base = (uint32_t)(32 * cw) << 16;
        const bool qjl = L.k_qjl;
        uint8_t* pbuf = smem + sl.phi;              // [P_hi | P_lo]
        float* tmax = red;                          // [2][32 heads][4 warps]
        float* lsum_s = red + 2 * 4 * kXpHeads;     // [4 warps][32 heads]
        int tseq = 0;
        for (int k = 0; k < nk; ++k) {
            const XpItem it = items[k];
            if (it.n_tiles == 0) continue;
            // the block's per-head constants (from the prep): head j = 4 e + hl
            {
                const int j = ctid >> 2, e = j >> 2, hl = j & 3;
                float v = 0.f;
                if (e < it.n)
                    v = a.ws_cst[((int64_t)(it.t0 + e) * a.q_heads + it.g * a.group + it.hgi * hc + hl) * 4 + (ctid & 3)];
                icst[ctid] = v;
            }
            named_sync(1, 128);
            float mref[kXpHeads], lp[kXpHeads];
#pragma unroll
            for (int j = 0; j < kXpHeads; ++j) {
                mref[j] = -INFINITY;
                lp[j] = 0.f;
            }
            for (int t = 0; t < it.n_tiles; ++t, ++tseq) {
                const int s = tseq % S;
                ws_wait(B(&full[s]), (tseq / S) & 1, dead, err);
                const int np = min(kTilePages, it.n_pages - t * kTilePages);
                const int pos = it.tok0 + (t * kTilePages + pj) * kBlock + r;
                const bool valid = pj < np && pos < it.tok1 && ((smask[s] >> pj) & 1);
                const uint8_t* pg = ring + s * sl.tile + pj * L.page_bytes;
                const float n16 = __half2float(*reinterpret_cast<const __half*>(pg + L.k_norm + 2 * r));
                const float rho = qjl ? __half2float(*reinterpret_cast<const __half*>(pg + L.k_rnorm + 2 * r)) : 0.f;
                __syncwarp();
                if (lane == 0) mbar_arrive(B(&empty[s]));

                // ---------------- scores of this token (log2 units), 32 heads
                float sc[kXpHeads];
                ws_wait(B(mdone), tseq & 1, dead, err);
                tc_fence_after();
#pragma unroll
                for (int q = 0; q < kXpHeads / 8; ++q) {
                    // 8 heads (two images): 32 key and 32 sign columns
                    uint32_t kc[32], sg[32];
                    tmem_ld32(tmem + lane_base + 32 * q, kc);
                    if (qjl) tmem_ld32(tmem + lane_base + kXpCols + 32 * q, sg);
                    tc_wait_ld();
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        const int j = 8 * q + h;
                        const float4 cst = *reinterpret_cast<const float4*>(icst + 4 * j);
                        float v = n16 * (cst.x + piece_sum(&kc[kPieces * h]) * cst.z);
                        if (qjl) v += rho * (cst.y + piece_sum(&sg[kPieces * h]) * cst.w);
                        sc[j] = (valid && (j >> 2) < it.n) ? v : -INFINITY;  // head j of entry j / 4
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(B(dfree));

                // ---------------- tile maxima: a transposed butterfly leaves the
                // warp's maximum of head `lane` in lane `lane`
                float* tm = tmax + (tseq & 1) * 4 * kXpHeads;
                {
                    float v[kXpHeads];
#pragma unroll
                    for (int j = 0; j < kXpHeads; ++j) v[j] = sc[j];
#pragma unroll
                    for (int w = kXpHeads / 2; w >= 1; w >>= 1) {
                        const bool up = (lane & w) != 0;
#pragma unroll
                        for (int j = 0; j < w; ++j) {
                            const float send = up ? v[j] : v[j + w];
                            const float keep = up ? v[j + w] : v[j];
                            v[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, w));
                        }
                    }
                    tm[lane * 4 + cw] = v[0];
                }
                named_sync(1, 128);
                // every consumer thread takes the same decisions (the maxima and
                // references are the same everywhere)
                bool any = false;
#pragma unroll
                for (int j = 0; j < kXpHeads; ++j) {
                    const float4 m4 = *reinterpret_cast<const float4*>(tm + 4 * j);
                    const float mt = fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w));
                    if (t == 0) mref[j] = mt;
                    else any |= mt > mref[j] + kRescaleSlack;
                }
                // the previous tile's P V must be done before the output
                // accumulator is rescaled or the probability operand rewritten
                if (tseq >= 1) ws_wait(B(&pvdone[1]), (tseq - 1) & 1, dead, err);
                if (any) {
                    tc_fence_after();
                    uint32_t o0[32], o1[32];
                    tmem_ld32(tmem + lane_base + kXpColO, o0);
                    tmem_ld32(tmem + lane_base + kXpColO + kXpHeads, o1);
                    tc_wait_ld();
#pragma unroll
                    for (int j = 0; j < kXpHeads; ++j) {
                        const float4 m4 = *reinterpret_cast<const float4*>(tm + 4 * j);
                        const float mt = fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w));
                        if (mt > mref[j] + kRescaleSlack) {
                            const float alpha = mref[j] == -INFINITY ? 0.f : fast_exp2(mref[j] - mt);
                            mref[j] = mt;
                            lp[j] *= alpha;
                            o0[j] = __float_as_uint(__uint_as_float(o0[j]) * alpha);
                            o1[j] = __float_as_uint(__uint_as_float(o1[j]) * alpha);
                        }
                    }
                    tmem_st32(tmem + lane_base + kXpColO, o0);
                    tmem_st32(tmem + lane_base + kXpColO + kXpHeads, o1);
                    tc_wait_st();
                    tc_fence_before();
                }

                // ---------------- probability operands (bf16 high | low parts)
#pragma unroll
                for (int c = 0; c < kXpHeads / 8; ++c) {
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int j = 8 * c + 2 * u;
                        const float p0 = sc[j] == -INFINITY ? 0.f : fast_exp2(sc[j] - mref[j]);
                        const float p1 = sc[j + 1] == -INFINITY ? 0.f : fast_exp2(sc[j + 1] - mref[j + 1]);
                        lp[j] += p0;
                        lp[j + 1] += p1;
                        xp_split2(p0, p1, hi[u], lo[u]);
                    }
                    *reinterpret_cast<uint4*>(pbuf + xp_mn_off(ctid, c, kXpPGroups)) =
                        make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4*>(pbuf + xp_mn_off(ctid, c + kXpHeads / 8, kXpPGroups)) =
                        make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(B(pready));
            }

            // ---------------- item end: the split partial of every (entry, head)
#pragma unroll
            for (int j = 0; j < kXpHeads; ++j) {
                const float l = warp_sum(lp[j]);
                if (lane == 0) lsum_s[cw * kXpHeads + j] = l;
            }
            ws_wait(B(&pvdone[1]), (tseq - 1) & 1, dead, err);
            tc_fence_after();
            uint32_t o0[32], o1[32];
            tmem_ld32(tmem + lane_base + kXpColO, o0);
            tmem_ld32(tmem + lane_base + kXpColO + kXpHeads, o1);
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B(oread));
            const int i = ctid;  // coordinate (tensor-memory lane)
            const int S_ = a.sp.n_splits;
#pragma unroll
            for (int j = 0; j < kXpHeads; ++j) {
                const int e = j >> 2;
                if (e < it.n) {
                    const int64_t row =
                        ((int64_t)(it.t0 + e) * a.q_heads + it.g * a.group + it.hgi * hc + (j & 3)) * S_ + it.c;
                    a.ws_acc[row * D + i] = __uint_as_float(o0[j]) + __uint_as_float(o1[j]);
                }
            }
            named_sync(1, 128);  // row sums published
            if (cw == 0) {
                float m = -INFINITY;
#pragma unroll
                for (int j = 0; j < kXpHeads; ++j)
                    if (lane == j) m = mref[j];
                const int j = lane, e = j >> 2;
                if (e < it.n) {
                    const float l =
                        (lsum_s[j] + lsum_s[kXpHeads + j]) + (lsum_s[2 * kXpHeads + j] + lsum_s[3 * kXpHeads + j]);
                    const int64_t row =
                        ((int64_t)(it.t0 + e) * a.q_heads + it.g * a.group + it.hgi * hc + (j & 3)) * S_ + it.c;
                    a.ws_ml[row * 2] = m;
                    a.ws_ml[row * 2 + 1] = l;
                }
            }
            named_sync(1, 128);  // icst and the row sums are free for the next item
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kXpTmemCols);
}

template <int KB, bool KU, bool G32, int VB>
tq_status launch_extend_prefix(const DecodeArgs& a, cudaStream_t s, int grid) {
    const size_t smem = xp_layout(a.lay.page_bytes, a.gm.bimg_bytes).total;
    const void* fn = (const void*)extend_prefix_kernel<KB, KU, G32, VB>;
    tq_status st = ensure_dynamic_smem(fn, (int)smem, "extend_prefix_kernel");
    if (st != TQ_OK) return st;
    return cuda_status(launch_pdl(a.pdl, extend_prefix_kernel<KB, KU, G32, VB>, dim3(grid), dim3(kXpThreads), smem, s, a));
}

template <int KB, bool KU>
inline tq_status xp_dispatch_v(const DecodeArgs& a, cudaStream_t s, int grid) {
    if (a.gm.npk != (KU ? KB : 1 << (KB - 1))) return TQ_ERR_UNSUPPORTED;
    if (a.lay.v_mode == TQ_V_G32)
        return a.lay.v_bits == 4 ? launch_extend_prefix<KB, KU, true, 4>(a, s, grid)
                                 : launch_extend_prefix<KB, KU, true, 2>(a, s, grid);
    switch (a.lay.v_bits) {
        case 2: return launch_extend_prefix<KB, KU, false, 2>(a, s, grid);
        case 3: return launch_extend_prefix<KB, KU, false, 3>(a, s, grid);
        default: return launch_extend_prefix<KB, KU, false, 4>(a, s, grid);
    }
}

}  // namespace tq
