// Warp-specialized, persistent split kernel of the decode path (included by
// the split translation units after tq_decode_kernels.cuh).
//
// Two CTAs per SM (bulk-copy throughput is per CTA) each walk a list of work
// items (one split of one KV head's head group of one sequence) as a stream of
// 128-token tiles, with three warpgroups running concurrently and handing
// tiles over through mbarriers:
//   producer   (warp 8, one thread): bulk async copies of the tiles' pages into
//              a ring of `stages` tiles and of each item's query operand image,
//              each issued as soon as its buffer is released
//   scores     (warps 0-3, thread t = token t of the tile): expand the key
//              bit-planes into fp8 operands in tensor memory, in two halves
//   MMA        (warp 9, one thread): the tcgen05 MMAs of each half into the
//              accumulator columns as soon as the half is stored
//   consumers  (warps 4-7, same token mapping): read the scores, online exp2
//              softmax, probability operands, value contraction of the warp's
//              two pages on fp16 tensor cores, per-item merge of the partials
// so that the expansion and MMAs of tile i+1 overlap the value contraction of
// tile i.  The score and value arithmetic is the
// same as in split_kernel (tq_decode_kernels.cuh).
#pragma once

#include "tq_decode_kernels.cuh"

namespace tq {

constexpr int kWsWarps = 12;  // 4 score + 4 consumer + 4 producer (one thread)
constexpr int kWsThreads = 32 * kWsWarps;
constexpr int kWsMaxStages = 8;
constexpr int kWsCtasPerSm = 2;   // bulk-copy throughput is per CTA: two CTAs per SM stream ~1.7x one
constexpr int kWsTmemCols = 256;  // 512 / kWsCtasPerSm
// setmaxnreg split of the 3 x 80 registers per thread (three warpgroups) a
// CTA launches with: the producer keeps 40, the score warpgroup 64, the
// consumers take the rest
constexpr int kWsRegsLaunch = 80, kWsRegsProducer = 40, kWsRegsScore = 64;
constexpr int kWsRegsCons = 3 * kWsRegsLaunch - kWsRegsProducer - kWsRegsScore;

// tensor-memory plan: one accumulator buffer of 2*score_cols (key | sign),
// then one A operand buffer
__host__ __device__ constexpr int ws_dcols(int nth) { return 2 * score_cols(nth); }
__host__ __device__ constexpr int ws_acap(int nth) { return kWsTmemCols - ws_dcols(nth); }

struct WsLayout {
    size_t tile, ring, bimg, pbuf, zsm, red, items, icst, ids, smask, bars, tslot, total;
    int pls, pbuf_words;
};

struct WsItem {
    int b, g, hgi, chunk, t0, t1, n_pages, n_tiles;
    // query operand image: buffer slot, whether this item loads it (and the
    // load's index among the slot's loads) and whether the slot is released
    // after the item's last MMA
    int slot, load, lidx, release;
};

// items per CTA (the largest share of the round-robin distribution)
__host__ __device__ inline int ws_items_per_cta(int n_items, int grid) { return (n_items + grid - 1) / grid; }

// kitems: items per CTA; split_blocks: pages per item at most
// image buffers: one per head group of a KV head (at most two)
__host__ __device__ inline int ws_nimg(const DecodeGeom& gm) { return gm.nhg < 2 ? 1 : 2; }

template <int D>
__host__ __device__ inline WsLayout ws_layout(int page_bytes, const DecodeGeom& gm, int nsets, int stages,
                                              int kitems, int split_blocks) {
    auto up = [](size_t x) { return (x + 127) & ~(size_t)127; };
    const int h4 = 4 * gm.nth;
    WsLayout l;
    l.tile = up((size_t)kTilePages * page_bytes);
    l.pls = nsets * h4 * 24 + 16;
    l.pbuf_words = 2 * l.pls;
    size_t off = 0;
    l.ring = off;
    off = up(off + (size_t)stages * l.tile);
    l.bimg = off;
    off = up(off + (size_t)ws_nimg(gm) * gm.bimg_bytes);
    // the per-item merge buffer reuses the probability buffers
    l.pbuf = l.red = off;
    const size_t pb = (size_t)4 * l.pbuf_words * 4, rb = (size_t)4 * h4 * (D + 2) * 4;
    off = up(off + (pb > rb ? pb : rb));
    l.zsm = off;
    off = up(off + (size_t)4 * h4 * (D / 32) * 4);
    l.items = off;
    off = up(off + (size_t)kitems * sizeof(WsItem));
    l.icst = off;
    off = up(off + (size_t)kitems * h4 * 4 * 4);
    l.ids = off;
    off = up(off + (size_t)kitems * split_blocks * 4);
    l.smask = off;
    off = up(off + (size_t)stages * 4);
    l.bars = off;
    off = up(off + (size_t)(2 * stages + 10) * 8);
    l.tslot = off;  // the tensor-memory address, then 4 ints of the located first item
    off = up(off + 20);
    l.total = off;
    return l;
}

// a configuration runs here when all its score planes fit one A buffer
__host__ __device__ inline bool ws_fits(const DecodeGeom& gm, int d) { return gm.npl * (d / 4) <= ws_acap(gm.nth); }

// compressed length of sequence b, clamped to the block table (bad: out of range)
__device__ __forceinline__ int ws_seq_len(const DecodeArgs& a, int b, bool* bad) {
    const int len = a.seq_lens[b];
    *bad = len < 0 || len > a.max_blocks * kBlock;
    return max(0, min(len, a.max_blocks * kBlock));
}
// splits of sequence b that hold tokens
__device__ __forceinline__ int ws_seq_chunks(const DecodeArgs& a, int len) {
    const int st = a.split_blocks * kBlock;
    return (len + st - 1) / st;
}
// work items: the non-empty splits of every (sequence, KV head, head group),
// split fastest, then head group, KV head, sequence (empty splits are left to
// the combine, which reads none beyond a sequence's length); every CTA takes
// a contiguous run of items, so consecutive items of a CTA are mostly
// consecutive splits of one head group, which its consumers merge as one (the
// other head group's CTAs, a few positions on, read the same pages at about
// the same time and find them in L2)
// items of sequence b: its non-empty splits x KV heads x head groups
__device__ __forceinline__ int ws_seq_items(const DecodeArgs& a, int b) {
    bool bad;
    return a.heads * a.gm.nhg * ws_seq_chunks(a, ws_seq_len(a, b, &bad));
}
// item idx_in_seq (in the order above) of sequence b
__device__ inline WsItem ws_item_at(const DecodeArgs& a, int b, int idx) {
    WsItem it;
    bool bad;
    const int nhg = a.gm.nhg;
    const int len = ws_seq_len(a, b, &bad), nch = ws_seq_chunks(a, len);
    it.b = b;
    it.chunk = idx % nch;
    idx /= nch;
    it.hgi = idx % nhg;
    it.g = idx / nhg;
    it.t0 = it.chunk * a.split_blocks * kBlock;
    it.t1 = min(len, it.t0 + a.split_blocks * kBlock);
    it.n_pages = it.t1 > it.t0 ? (it.t1 - it.t0 + kBlock - 1) / kBlock : 0;
    it.n_tiles = (it.n_pages + kTilePages - 1) / kTilePages;
    it.slot = it.load = it.lidx = it.release = 0;
    return it;
}
// Warp-cooperative, every lane returning the same values: the launch's item
// count, the items per CTA for `grid` CTAs, and for item `first` of CTA cta
// the sequence that holds it and that sequence's first item index (lanes
// read 32 sequences' lengths at a time; two passes over the batch).
struct WsLocate {
    int n_items, per_cta, b0, base0;
};
__device__ inline WsLocate ws_warp_locate(const DecodeArgs& a, int cta, int grid, int lane) {
    WsLocate r;
    int total = 0;
    for (int c = 0; c < a.batch; c += 32) {
        int n = c + lane < a.batch ? ws_seq_items(a, c + lane) : 0;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
        total += n;
    }
    r.n_items = total;
    r.per_cta = ws_items_per_cta(total, grid);
    const int first = cta * r.per_cta;
    r.b0 = a.batch;
    r.base0 = total;
    int base = 0;
    for (int c = 0; c < a.batch && first < total; c += 32) {
        const int n = c + lane < a.batch ? ws_seq_items(a, c + lane) : 0;
        int incl = n;  // inclusive prefix over the lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        const bool hit = n > 0 && first >= base + incl - n && first < base + incl;
        const uint32_t m = __ballot_sync(0xffffffffu, hit);
        if (m) {
            const int l = __ffs(m) - 1;
            r.b0 = c + l;
            r.base0 = base + __shfl_sync(0xffffffffu, incl - n, l);
            break;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    return r;
}
// item idx of the launch, found by walking forward from sequence b (whose
// first item index is base, with base <= idx)
__device__ inline WsItem ws_item_from(const DecodeArgs& a, int b, int base, int idx) {
    for (;;) {
        const int n = ws_seq_items(a, b);
        if (idx < base + n || b == a.batch - 1) break;
        base += n;
        ++b;
    }
    return ws_item_at(a, b, idx - base);
}

// non-blocking: has the phase of the given parity completed?
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
// bounded wait that is skipped once the caller has given up (dead)
__device__ __forceinline__ void ws_wait(uint32_t bar, uint32_t parity, bool& dead, uint32_t* err) {
    if (!dead) dead = !mbar_wait(bar, parity, err);
}

// Copy issue cursor of a split CTA, run by one whole warp: walks the tiles of
// the CTA's non-empty items in order, loading an item's query operand image
// before its first tile when it needs one; lane j issues the copy of a tile's
// page j, so a tile costs a handful of warp instructions.  issue_upto runs up
// to limit_seq, blocking only for tiles up to need_seq (whose stage releases
// depend on MMAs already issued) and otherwise stopping at the first stage or
// image not yet free.
struct WsIssuer {
    const WsItem* items;
    const int32_t* ids;
    uint32_t* smask;
    uint8_t* ring;
    uint8_t* bimg;
    uint64_t *full, *empty, *bfull, *bempty;
    const uint8_t* cache;
    const uint8_t* ws_bimg;
    uint32_t* err;
    size_t tile;
    int nk, SB, S, page_bytes, bimg_bytes, heads, nhg;
    int64_t num_blocks;
    int c_k = 0, c_t = 0, c_seq = 0;
    bool c_img = false, dead = false;

    __device__ void next_item() {
        while (c_k < nk && items[c_k].n_tiles == 0) ++c_k;
    }

    // warp-uniform wait: lane 0 waits (bounded), the others take its outcome
    __device__ bool wait_uniform(uint64_t* bar, uint32_t par, bool block, int lane) {
        int ok = 1;
        if (lane == 0) {
            if (block) {
                if (!mbar_wait(smem_u32(bar), par, err)) {
                    dead = true;
                    ok = 0;
                }
            } else {
                ok = mbar_test(smem_u32(bar), par);
            }
        }
        dead = __shfl_sync(0xffffffffu, (int)dead, 0) != 0;
        return __shfl_sync(0xffffffffu, ok, 0) != 0;
    }

    __device__ __noinline__ void issue_upto(int limit_seq, int need_seq, int max_tiles) {
        const int lane = threadIdx.x & 31;
#pragma unroll 1
        for (int n = 0; c_k < nk && c_seq <= limit_seq && !dead && (n < max_tiles || c_seq <= need_seq); ++n) {
            const WsItem& it = items[c_k];
            if (!c_img) {
                if (it.load) {
                    if (it.lidx >= 1) {
                        if (!wait_uniform(&bempty[it.slot], (it.lidx - 1) & 1, c_seq <= need_seq, lane) || dead)
                            break;
                    }
                    if (lane == 0) {
                        mbar_expect_tx(smem_u32(&bfull[it.slot]), bimg_bytes);
                        bulk_copy(smem_u32(bimg + (size_t)it.slot * bimg_bytes),
                                  ws_bimg + (((int64_t)it.b * heads + it.g) * nhg + it.hgi) * bimg_bytes, bimg_bytes,
                                  smem_u32(&bfull[it.slot]));
                    }
                }
                c_img = true;
            }
            const int s = c_seq % S;
            if (c_seq >= S) {
                if (!wait_uniform(&empty[s], ((c_seq / S) - 1) & 1, c_seq <= need_seq, lane) || dead) break;
            }
            // the consumers' reads of this stage happen-before the copies
            // through the empty barrier (release/acquire)
            const int p0 = c_t * kTilePages, np = min(kTilePages, it.n_pages - p0);
            int blk = -1;
            if (lane < np) blk = ids[c_k * SB + p0 + lane];
            const bool ok = lane < np && blk >= 0 && blk < num_blocks;
            const uint32_t mask = __ballot_sync(0xffffffffu, ok);
            if (lane < np && !ok) set_error(err, TQ_DEVERR_BLOCK);
            if (lane == 0) {
                smask[s] = mask;  // published by the arrive below
                mbar_expect_tx(smem_u32(&full[s]), (uint32_t)__popc(mask) * page_bytes);
            }
            __syncwarp();
            if (ok)
                bulk_copy(smem_u32(ring + s * tile + (size_t)lane * page_bytes),
                          cache + ((int64_t)blk * heads + it.g) * page_bytes, page_bytes, smem_u32(&full[s]));
            ++c_seq;
            if (++c_t == it.n_tiles) {
                c_t = 0;
                c_img = false;
                ++c_k;
                next_item();
            }
        }
    }
};

// The MMAs of score planes [P0, P1) of a tile, with addresses stepped
// incrementally: the issuing thread shares its SM sub-partition with busy
// warps, so each MMA gets a few instructions at most.  bd0 is the descriptor
// of the operand image at plane 0, k-block 0.
template <int D, int NPK, int NCOLS, int TA>
__device__ __forceinline__ void ws_issue_planes(int P0, int P1, uint32_t tmem, uint64_t bd0, uint32_t idesc) {
    constexpr int NW = D / 32, NCOL = D / 4;
    uint32_t a_addr = tmem + TA + P0 * NCOL;
    uint64_t bd = bd0 + (uint64_t)(P0 * (D / 16) * 8);
#pragma unroll 1
    for (int P = P0; P < P1; ++P) {
        const uint32_t d = P < NPK ? tmem : tmem + NCOLS;
        const uint32_t first = (P == 0 || P == NPK) ? 0u : 1u;  // a fresh accumulator starts at plane 0 / NPK
#pragma unroll
        for (int kb = 0; kb < NW; ++kb) mma_fp8_ts(d, a_addr + 8 * kb, bd + (uint64_t)(16 * kb), idesc, kb ? 1u : first);
        a_addr += NCOL;
        bd += (uint64_t)((D / 16) * 8);
    }
}

// KU: the key codebook is a uniform grid, whose expansion over XOR bit-planes
// has only the KB single-bit terms (plane_subset lists those first)
template <int D, int KB, bool KU, bool G32, int VB, int NTH>
__global__ void __launch_bounds__(kWsThreads, kWsCtasPerSm) split_ws_kernel(DecodeArgs a) {
    static_assert(kWsRegsCons <= 256 && kWsRegsCons % 8 == 0, "register split");
    constexpr int NPK = KU ? KB : 1 << (KB - 1);
    constexpr int NW = D / 32;
    constexpr int NCOL = D / 4;
    constexpr int NMT = D / 16;
    constexpr int NPV = G32 ? 1 : (1 << (VB - 1));
    constexpr int NSET = G32 ? D / 32 : NPV;
    constexpr int NZ = G32 ? D / 32 : 1;
    constexpr int H4 = 4 * NTH;
    constexpr int NCOLS = score_cols(NTH);
    constexpr int DC = ws_dcols(NTH);  // accumulator columns (key | sign)
    constexpr int TA = DC;             // first A operand column
    extern __shared__ __align__(16) uint8_t smem[];
    const DecodeGeom gm = a.gm;
    const Layout& L = a.lay;
    const int S = a.stages;
    // shared-memory arrays hold KI items (every split of every head group);
    // the non-empty ones are dealt out KR per CTA
    const int KI = ws_items_per_cta(a.batch * a.heads * gm.nhg * a.sp.n_chunks, gridDim.x);
    const WsLayout sl = ws_layout<D>(L.page_bytes, gm, NSET, S, KI, a.split_blocks);
    uint8_t* ring = smem + sl.ring;
    uint8_t* bimg = smem + sl.bimg;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + sl.bars);
    uint64_t* full = bars;               // [S]  tile landed (tx)
    uint64_t* empty = bars + S;          // [S]  tile released (4 consumer warps + score group)
    uint64_t* bfull = bars + 2 * S;      // [slot] operand image landed (tx)
    uint64_t* bempty = bfull + 2;        // [slot] operand image released (MMA commit)
    // the score planes of a tile go in two halves (planes [0, PX) and [PX, npl))
    // so that the MMAs of one half overlap the expansion of the other
    uint64_t* mdone = bempty + 2;        // [half] MMAs of a half done (commit); half 1: scores ready
    uint64_t* dfree = mdone + 2;         // scores read (4 consumer warps)
    uint64_t* aready = dfree + 1;        // [half] A operand half stored (4 score warps)
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + sl.tslot);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint32_t* err = a.dp.err;
    WsItem* items = reinterpret_cast<WsItem*>(smem + sl.items);
    float* icst = reinterpret_cast<float*>(smem + sl.icst);      // [item][head][4]
    int32_t* ids = reinterpret_cast<int32_t*>(smem + sl.ids);     // [item][split_blocks] block ids
    uint32_t* smask = reinterpret_cast<uint32_t*>(smem + sl.smask);  // [stage] pages copied
    auto B = [&](const uint64_t* p) { return smem_u32(p); };

    // Thread 0 initialises the barriers; warp 8 locates the CTA's first item
    // (a warp-cooperative scan of the lengths instead of a walk over every
    // sequence per item).  loc: [items, items per CTA, first item's sequence,
    // that sequence's first item].
    int* loc = reinterpret_cast<int*>(smem + sl.tslot) + 1;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(B(&full[s]), 1);
            mbar_init(B(&empty[s]), 5);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(B(&bfull[i]), 1);
            mbar_init(B(&bempty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(B(&mdone[i]), 1);
            mbar_init(B(&aready[i]), 4);
        }
        mbar_init(B(dfree), 4);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 8) {
        const WsLocate w = ws_warp_locate(a, blockIdx.x, gridDim.x, lane);
        if (lane == 0) {
            loc[0] = w.n_items;
            loc[1] = w.per_cta;
            loc[2] = w.b0;
            loc[3] = w.base0;
        }
    }
    if (warp == 0) tmem_alloc(tslot, kWsTmemCols);
    pdl_launch_dependents();
    __syncthreads();  // the barriers and the located first item
    const int n_items = loc[0], KR = loc[1];
    const int k0 = blockIdx.x * KR;                 // this CTA's first item
    const int nk = max(0, min(KR, n_items - k0));  // and its item count

    // prologue: this CTA's items, their per-head constants and block ids into
    // shared memory (batches of independent loads), so that the tile loop
    // below makes no global loads
    const int hc = gm.hc, SB = a.split_blocks;
    {
        const int b0 = loc[2], base0 = loc[3];
        for (int k = tid; k < nk; k += blockDim.x) items[k] = ws_item_from(a, b0, base0, k0 + k);
    }
    if (blockIdx.x == 0)
        for (int b = tid; b < a.batch; b += blockDim.x) {
            bool bad = false;
            ws_seq_len(a, b, &bad);
            if (bad) set_error(err, TQ_DEVERR_SEQLEN);
        }
    __syncthreads();
    if (tid == 0) {
        const int nimg = ws_nimg(gm);
        int key[2] = {-1, -1}, nload[2] = {0, 0}, last[2] = {-1, -1};
        for (int k = 0; k < nk; ++k) {
            WsItem& it = items[k];
            it.slot = it.load = it.lidx = it.release = 0;
            if (it.n_tiles == 0) continue;
            const int sl_ = it.hgi % nimg, kk = (it.b * a.heads + it.g) * gm.nhg + it.hgi;
            it.slot = sl_;
            if (key[sl_] != kk) {
                if (last[sl_] >= 0) items[last[sl_]].release = 1;
                it.load = 1;
                it.lidx = nload[sl_]++;
                key[sl_] = kk;
            }
            last[sl_] = k;
        }
    }
    pdl_wait();  // the query prep's results
    {
        // the items' per-head constants (from the prep) and block ids, their
        // loads issued together
        const int n_cst = nk * H4 * 4, n_ids = nk * SB, n_all = max(n_cst, n_ids);
        for (int base = tid; base < n_all; base += blockDim.x * 4) {
            float cv[4];
            int32_t iv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = base + u * blockDim.x;
                cv[u] = 0.f;
                iv[u] = -1;
                if (e < n_cst) {
                    const WsItem& it = items[e / (H4 * 4)];
                    const int h = (e >> 2) % H4;
                    if (h < hc)
                        cv[u] = a.ws_cst[((int64_t)it.b * a.q_heads + it.g * a.group + it.hgi * hc + h) * 4 + (e & 3)];
                }
                if (e < n_ids) {
                    const WsItem& it = items[e / SB];
                    const int pg = e % SB;
                    if (pg < it.n_pages) {
                        const int row = a.row_of ? a.row_of[it.b] : it.b;
                        iv[u] = a.block_table[(int64_t)row * a.max_blocks + it.t0 / kBlock + pg];
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = base + u * blockDim.x;
                if (e < n_cst) icst[e] = cv[u];
                if (e < n_ids) ids[e] = iv[u];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool dead = false;

    const int PX = (gm.npl + 1) / 2;  // planes in the first half
    if (warp >= 8) {
        // ------------------------------------------------------ producer
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kWsRegsProducer));
        if (tid == 288) {
            // MMA issue (one thread; tcgen05.mma blocks while the tensor pipe is busy)
            const uint32_t idesc = fp8_idesc(NCOLS);
            const uint32_t sbo = 8u * (uint32_t)(gm.npl * D);
            int tseq = 0;
            for (int k = 0; k < nk; ++k) {
                const WsItem it = items[k];
                if (it.n_tiles == 0) continue;
                const uint32_t img = smem_u32(bimg + (size_t)it.slot * gm.bimg_bytes);
                for (int t = 0; t < it.n_tiles; ++t, ++tseq) {
                    const int s = tseq % S;
                    if (t == 0 && it.load) ws_wait(B(&bfull[it.slot]), it.lidx & 1, dead, err);
                    if (tseq >= 1) ws_wait(B(dfree), (tseq - 1) & 1, dead, err);  // accumulators read
                    const uint64_t bd0 = smem_desc(img, 128, sbo);
                    ws_wait(B(&aready[0]), tseq & 1, dead, err);
                    tc_fence_after();
                    ws_issue_planes<D, NPK, NCOLS, TA>(0, PX, tmem, bd0, idesc);
                    tc_commit(B(&mdone[0]));
                    ws_wait(B(&aready[1]), tseq & 1, dead, err);
                    tc_fence_after();
                    mbar_arrive(B(&empty[s]));  // the keys of this stage are read
                    ws_issue_planes<D, NPK, NCOLS, TA>(PX, gm.npl, tmem, bd0, idesc);
                    tc_commit(B(&mdone[1]));
                    if (t == it.n_tiles - 1 && it.release) tc_commit(B(&bempty[it.slot]));
                }
            }
        }
        if (warp == 8) {
            WsIssuer iss{items, ids, smask, ring, bimg, full, empty, bfull, bempty, a.cache, a.ws_bimg, err,
                         sl.tile, nk, SB, S, L.page_bytes, gm.bimg_bytes, a.heads, gm.nhg, a.num_blocks};
            iss.next_item();
            iss.issue_upto(0x7fffffff, 0x7fffffff, 0x7fffffff);  // every wait blocks: nothing else to do
            // copies still in flight must land before the block exits
            bool d2 = lane != 0;  // lane 0 drains
            for (int k = max(0, iss.c_seq - S); k < iss.c_seq; ++k) ws_wait(B(&full[k % S]), (k / S) & 1, d2, err);
            int nl[2] = {0, 0};
            for (int k = 0; k < nk; ++k)
                if (items[k].n_tiles > 0 && items[k].load && (k < iss.c_k || (k == iss.c_k && iss.c_img)))
                    nl[items[k].slot] = items[k].lidx + 1;
            for (int i = 0; i < 2; ++i)
                if (nl[i] > 0) ws_wait(B(&bfull[i]), (nl[i] - 1) & 1, d2, err);
        }
    } else if (warp < 4) {
        // ------------------------------------------------- score operands
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kWsRegsScore));
        const int pj = tid >> 4, r = tid & 15;
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        const bool qjl = L.k_qjl;
        int tseq = 0;
        for (int k = 0; k < nk; ++k) {
            const WsItem it = items[k];
            if (it.n_tiles == 0) continue;
            for (int t = 0; t < it.n_tiles; ++t, ++tseq) {
                const int s = tseq % S;
                ws_wait(B(&full[s]), (tseq / S) & 1, dead, err);
                const uint8_t* pg = ring + s * sl.tile + pj * L.page_bytes;
                uint32_t kw[KB][NW], sw[NW];
#pragma unroll
                for (int p = 0; p < KB; ++p)
#pragma unroll
                    for (int w4 = 0; w4 < NW; w4 += 4) {
                        const uint4 u =
                            *reinterpret_cast<const uint4*>(pg + L.k_codes + (p * kBlock + r) * (D / 8) + 4 * w4);
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
                const uint32_t abase = tmem + lane_base + TA;
#pragma unroll
                for (int P = 0; P <= NPK; ++P) {
                    if (P == NPK && !qjl) break;
                    if (P == 0 || P == PX) {
                        // half h of the A operand: wait until the previous tile's MMAs
                        // of that half are done (after storing and publishing half 0)
                        if (P == PX) {
                            tc_wait_st();
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(B(&aready[0]));
                        }
                        if (tseq >= 1) ws_wait(B(&mdone[P == 0 ? 0 : 1]), (tseq - 1) & 1, dead, err);
                        tc_fence_after();
                    }
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
                        tmem_st32(abase + P * NCOL + 32 * q, a32);
                    }
                }
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(B(&aready[1]));
            }
        }
    } else {
        // ------------------------------------------------------ consumers
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kWsRegsCons));
        const int cw = warp - 4, ctid = tid - 128;
        const int gq = lane >> 2, tq = lane & 3;
        const int pj = ctid >> 4, r = ctid & 15;
        const int pl = pj & 1, pair = r & 7, hf = r >> 3;
        const uint32_t lane_base = (uint32_t)(32 * cw) << 16;
        const bool qjl = L.k_qjl;
        uint32_t* pbw = reinterpret_cast<uint32_t*>(smem + sl.pbuf) + cw * sl.pbuf_words;
        float* zsm = reinterpret_cast<float*>(smem + sl.zsm) + cw * H4 * (D / 32);
        float* red = reinterpret_cast<float*>(smem + sl.red);
        for (int e = lane; e < sl.pbuf_words; e += 32) pbw[e] = 0u;
        float v_dc = 0.f, v_beta[NPV];
        if constexpr (!G32) {
            v_dc = a.dp.v_walsh[0];
#pragma unroll
            for (int P = 0; P < NPV; ++P) {
                v_beta[P] = -0.5f * a.dp.v_walsh[1 + P];
                v_dc += 0.5f * a.dp.v_walsh[1 + P];
            }
        }
        int tseq = 0, st = 0;
        uint32_t sph = 0;  // stage of tile tseq and the parity of its fill
        // a run: consecutive items of one (sequence, KV head, head group), i.e.
        // consecutive splits, accumulated as one and written as split run0
        float m_ref[H4], l_part[H4], zacc[H4][NZ];
        float pv[NTH][NMT][4];
        int run0 = -1;
        bool fresh = true;  // nothing accumulated in this run yet
        for (int k = 0; k < nk; ++k) {
            const WsItem it = items[k];
            const float* cst = icst + k * H4 * 4;
            if (run0 < 0) {
                run0 = it.chunk;
                fresh = true;
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
            }
            for (int t = 0; t < it.n_tiles; ++t, ++tseq) {
                const int s = st;
                ws_wait(B(&full[s]), sph, dead, err);
                ws_wait(B(&mdone[1]), tseq & 1, dead, err);
                tc_fence_after();
                const int p0 = t * kTilePages, np = min(kTilePages, it.n_pages - p0);
                const uint8_t* tile = ring + s * sl.tile;
                const int pos = it.t0 + (p0 + pj) * kBlock + r;
                const bool valid = pj < np && pos < it.t1 && ((smask[s] >> pj) & 1);
                const uint8_t* pg = tile + pj * L.page_bytes;

                // ---------------- scores of this token (log2 units)
                const float n16 = __half2float(*reinterpret_cast<const __half*>(pg + L.k_norm + 2 * r));
                const float rho = qjl ? __half2float(*reinterpret_cast<const __half*>(pg + L.k_rnorm + 2 * r)) : 0.f;
                float sc[H4];
                {
                    uint32_t acc[NCOLS];
                    float sk[H4];
                    const uint32_t dk = tmem + lane_base;
#pragma unroll
                    for (int q = 0; q < NCOLS / 16; ++q)
                        tmem_ld16(dk + 16 * q, *reinterpret_cast<uint32_t(*)[16]>(&acc[16 * q]));
                    tc_wait_ld();
#pragma unroll
                    for (int h = 0; h < H4; ++h) sk[h] = piece_sum(&acc[kPieces * h]);
                    if (qjl) {
#pragma unroll
                        for (int q = 0; q < NCOLS / 16; ++q)
                            tmem_ld16(dk + NCOLS + 16 * q, *reinterpret_cast<uint32_t(*)[16]>(&acc[16 * q]));
                        tc_wait_ld();
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(B(dfree));
#pragma unroll
                    for (int h = 0; h < H4; ++h) {
                        float v = n16 * (cst[4 * h] + sk[h] * cst[4 * h + 2]);
                        if (qjl) v += rho * (cst[4 * h + 1] + piece_sum(&acc[kPieces * h]) * cst[4 * h + 3]);
                        sc[h] = (valid && h < hc) ? v : -INFINITY;
                    }
                }

                // ---------------- online softmax per warp (lazy reference maximum)
                if (fresh) {
                    // the run's first tile: nothing accumulated yet to rescale
#pragma unroll
                    for (int h = 0; h < H4; ++h) m_ref[h] = warp_max(sc[h]);
                    fresh = false;
                } else {
                    // a reference moves only when a score passes it by kRescaleSlack
                    bool mv = false;
#pragma unroll
                    for (int h = 0; h < H4; ++h) mv |= sc[h] > m_ref[h] + kRescaleSlack;
                    if (__any_sync(0xffffffffu, mv)) {
#pragma unroll
                        for (int h = 0; h < H4; ++h) {
                            if (!__any_sync(0xffffffffu, sc[h] > m_ref[h] + kRescaleSlack)) continue;
                            const float mx = warp_max(sc[h]);
                            const float alpha = m_ref[h] == -INFINITY ? 0.f : fast_exp2(m_ref[h] - mx);
                            m_ref[h] = mx;
                            l_part[h] *= alpha;
#pragma unroll
                            for (int z = 0; z < NZ; ++z) zacc[h][z] *= alpha;
                            if (tq == (h & 3)) {
#pragma unroll
                                for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
                                    for (int e = 0; e < 4; ++e) pv[h >> 2][mt][e] *= alpha;
                            }
                        }
                    }
                }
                float p[H4];
#pragma unroll
                for (int h = 0; h < H4; ++h) {
                    p[h] = sc[h] == -INFINITY ? 0.f : fast_exp2(sc[h] - m_ref[h]);
                    l_part[h] += p[h];
                }

                // ---------------- probability operands (masked heads write zeros)
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
                        constexpr int MW = D / 32;
                        uint32_t mw[MW];
#pragma unroll
                        for (int w4 = 0; w4 < MW; w4 += 4) {
                            const uint4 u =
                                *reinterpret_cast<const uint4*>(pg + L.v_meta + r * L.v_meta_row + 4 * w4);
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
                                put(gr, h, p[h] * sv);
                                zacc[h][gr] = fmaf(p[h], zv, zacc[h][gr]);
                            }
                        }
                    } else {
                        const float nv =
                            valid ? __half2float(*reinterpret_cast<const __half*>(pg + L.v_meta + 2 * r)) : 0.f;
#pragma unroll
                        for (int h = 0; h < H4; ++h) {
                            const float pn = p[h] * nv;
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
                    const int pjw = 2 * cw + pl2;
                    if (pjw >= np) break;
                    const uint8_t* pgw = tile + pjw * L.page_bytes;
                    const uint32_t* pbr = pbw + pl2 * sl.pls + (gq >> 1) * 24 + (gq & 1) + 2 * tq;
                    if constexpr (G32) {
                        constexpr int TB = D * VB / 64;
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
                        constexpr int CB = D / 64;
                        uint32_t wlo[VB][2], whi[VB][2];
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
                if (lane == 0) mbar_arrive(B(&empty[s]));
                if (++st == S) {
                    st = 0;
                    sph ^= 1u;
                }
            }

            // ---------------- run end: per-warp partials -> merged split partial
            if (k + 1 < nk && items[k + 1].b == it.b && items[k + 1].g == it.g && items[k + 1].hgi == it.hgi)
                continue;  // the next item continues this run
            named_sync(2, 128);  // every warp is done with its probability buffer
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
                    red[(cw * H4 + h) * (D + 2) + D] = m_ref[h];
                    red[(cw * H4 + h) * (D + 2) + D + 1] = l_part[h];
                }
            __syncwarp();
#pragma unroll
            for (int nt = 0; nt < NTH; ++nt) {
                const int head = 4 * nt + tq;
                float* my = red + (cw * H4 + head) * (D + 2);
#pragma unroll
                for (int mt = 0; mt < NMT; ++mt) {
                    float v0v = pv[nt][mt][0] + pv[nt][mt][1], v1v = pv[nt][mt][2] + pv[nt][mt][3];
                    int c0;
                    if constexpr (G32) {
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
            named_sync(2, 128);
            // merge weights once per (warp, head): 2^(m_w - M) against the
            // largest reference M; they go where the zero-point sums were
            const int64_t o0 = ((int64_t)it.b * a.q_heads + it.g * a.group + it.hgi * hc) * a.sp.n_splits + run0;
            // the run's other splits are empty (m = -inf, l = 0)
            for (int e = ctid; e < hc * (it.chunk - run0); e += 128) {
                const int h = e / (it.chunk - run0), c = 1 + e % (it.chunk - run0);
                reinterpret_cast<float2*>(a.ws_ml)[o0 + (int64_t)h * a.sp.n_splits + c] = make_float2(-INFINITY, 0.f);
            }
            float* wts = reinterpret_cast<float*>(smem + sl.zsm);  // [warp][head]
            if (ctid < hc) {
                const int h = ctid;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < 4; ++w) M = fmaxf(M, red[(w * H4 + h) * (D + 2) + D]);
                float l = 0.f;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float mw = red[(w * H4 + h) * (D + 2) + D];
                    const float wt = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
                    wts[w * H4 + h] = wt;
                    l = fmaf(wt, red[(w * H4 + h) * (D + 2) + D + 1], l);
                }
                const int64_t o = o0 + (int64_t)h * a.sp.n_splits;
                a.ws_ml[o * 2] = M;
                a.ws_ml[o * 2 + 1] = l;
            }
            named_sync(2, 128);
            for (int e = ctid; e < hc * D; e += 128) {
                const int h = e / D, i = e % D;
                float acc = 0.f;
#pragma unroll
                for (int w = 0; w < 4; ++w) acc = fmaf(wts[w * H4 + h], red[(w * H4 + h) * (D + 2) + i], acc);
                a.ws_acc[(o0 + (int64_t)h * a.sp.n_splits) * D + i] = acc;
            }
            named_sync(2, 128);
            run0 = -1;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kWsTmemCols);
}

// Exact hybrid-tail tokens of every (KV head, sequence, query head) as split
// n_chunks: one query head per CTA, so that the short tail spreads over the
// SMs (the key and value rows are read once per query head, from L2)
template <int D>
__global__ void __launch_bounds__(128) tail_kernel(DecodeArgs a) {
    pdl_launch_dependents();
    extern __shared__ __align__(16) uint8_t smem[];
    const int g = blockIdx.x, b = blockIdx.y, h = blockIdx.z;
    // it reads only the caller's inputs, final once the query prep (its
    // predecessor) has started, and writes only its own partials, so it runs
    // beside the prep; it waits for the prep at its end because the split
    // kernel after it waits only on it
    if (b < a.batch && h < a.group) tail_split<D>(a, g, b, smem, h, 1);
    pdl_wait();
}

template <int D, int KB, bool KU, bool G32, int VB, int NTH>
inline tq_status launch_split_ws(const DecodeArgs& a, cudaStream_t s, size_t smem, int grid) {
    auto kern = split_ws_kernel<D, KB, KU, G32, VB, NTH>;
    {
        const tq_status fs = ensure_dynamic_smem((const void*)kern, 227 * 1024, "split_ws_kernel");
        if (fs != TQ_OK) return fs;
    }
    const cudaError_t e = launch_pdl(a.pdl, kern, dim3(grid), dim3(kWsThreads), smem, s, a);
    if (e != cudaSuccess) {
        cudaFuncAttributes fa{};
        cudaFuncGetAttributes(&fa, kern);
        return cuda_status_detail(e, "split_ws_kernel regs %d, max threads %d, static smem %zu, dynamic %zu, "
                                     "block %d, grid %d", fa.numRegs, fa.maxThreadsPerBlock, fa.sharedSizeBytes,
                                  smem, kWsThreads, grid);
    }
    return TQ_OK;
}

template <int D, int KB, bool KU, int NTH>
inline tq_status dispatch_ws_v(const DecodeArgs& a, cudaStream_t s, size_t smem, int grid) {
    if (a.gm.nth != NTH || a.gm.npk != (KU ? KB : 1 << (KB - 1))) return TQ_ERR_UNSUPPORTED;
    if (a.lay.v_mode == TQ_V_G32)
        return a.lay.v_bits == 4 ? launch_split_ws<D, KB, KU, true, 4, NTH>(a, s, smem, grid)
                                 : launch_split_ws<D, KB, KU, true, 2, NTH>(a, s, smem, grid);
    switch (a.lay.v_bits) {
        case 2: return launch_split_ws<D, KB, KU, false, 2, NTH>(a, s, smem, grid);
        case 3: return launch_split_ws<D, KB, KU, false, 3, NTH>(a, s, smem, grid);
        default: return launch_split_ws<D, KB, KU, false, 4, NTH>(a, s, smem, grid);
    }
}

// the uniform-key (KU) instances of the warp-specialized kernel, compiled in
// their own translation units
template <int D, int KB>
tq_status dispatch_ws_uniform(const DecodeArgs& a, cudaStream_t s, size_t smem, int grid);

}  // namespace tq
