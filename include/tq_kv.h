/*
 * tq_kv.h -- C ABI of a GB300 (sm_103a) library for TurboQuant's compressed
 * KV cache: the fused cache store and decode attention over the paged,
 * bit-packed cache.
 *
 * Sources (cited by short key below):
 *   [Roadmap]   "From paper to practice: the TurboQuant integration roadmap
 *               for vLLM, SGLang and TRT-LLM" (miraclefarms.github.io notes,
 *               2026-04-21), §1 core design, §3.1-3.2 vLLM store/decode
 *               kernels, §4.1-4.4 SGLang fused kernels.
 *   [Hub]       "TurboQuant: extreme KV-cache compression for LLM inference"
 *               (pomoai.com hub, 0xSero/turboquant), "Technical principle"
 *               steps 1-5, "vLLM integration" (hybrid mode).
 *   [Paged]     "PagedAttention + TurboQuant" (ithelp.ithome.com.tw article
 *               10406003), "TurboQuant's core idea", "Which path vLLM takes".
 *   [Explainer] "TurboQuant: 3-bit KV cache" (yage.ai, 2026-03-25), the
 *               three-component pipeline.
 *
 * Conventions
 *   - Every call returns a tq_status; TQ_OK is 0, errors are negative.  No
 *     C++ exception crosses this boundary.
 *   - All device memory is owned by the caller and passed as raw pointers; the
 *     library never allocates or frees device memory.  A tq_cache handle is a
 *     small host object that records the caller's params/workspace pointers.
 *   - tq_store and tq_decode_attention are asynchronous on the caller's
 *     stream, launch a fixed grid that depends only on the cache
 *     configuration (CUDA-graph capturable), and do not synchronise the host.
 *     Calls on distinct streams may run concurrently only if they use distinct
 *     workspaces (one cache handle = one workspace).
 *   - Any host thread may call any entry point, on any device (the one current
 *     on the calling thread).  The first tq_store / tq_decode_attention /
 *     tq_extend_attention call on a device does that device's launch set-up
 *     (its SM count, the kernels' shared-memory limits) under a lock, once per
 *     device; make it before capturing a stream on that device.
 *   - Bad arguments found on the host return TQ_ERR_INVALID_ARG and launch
 *     nothing.  Bad indices found on the device (a slot or block id outside
 *     the cache, a sequence longer than its block-table row) skip the item and
 *     set a bit in a device error word read by tq_get_device_error; kernels
 *     never trap.
 *
 * Page layout (a reading: the pages fix only the packing density, 2-bit codes
 * a quarter byte and 4-bit codes half a byte, [Hub] step 5).  cache = uint8
 * [num_blocks][num_kv_heads][page_bytes]; a page holds the 16 token rows of one
 * block for one KV head.  Bit c of a d-bit row is bit c%8 of byte c/8.  Planes,
 * each of 16 rows, in this order:
 *   K code planes  k_bits x 16 x (d/8)  bit-sliced: plane p, bit c of row r =
 *                                       bit p of the code of coordinate c
 *   K signs        16 x (d/8)           (k_qjl) bit c = [(S r)_c >= 0]
 *   K norm         16 x fp16            ||k|| rounded to fp16
 *   K rnorm        16 x fp16            (k_qjl) ||residual|| rounded to fp16
 *   V codes   MSE: v_bits x 16 x (d/8)  bit-sliced like the keys
 *             G32: 16 x (d*v_bits/8)    v_bits-bit fields, LSB-first; field
 *                                       slot k = (d/8)*g + 2*m + e (g < 8,
 *                                       m < d/16, e < 2) holds coordinate
 *                                       32*(m/2) + 4*g + 2*(m%2) + e
 *   V meta    MSE: 16 x fp16 norm
 *             G32: 16 x (d/32) x {fp16 scale, fp16 zero}  (natural group order)
 * Every plane size is a multiple of 16 bytes.  Token t of sequence b is
 * stored in block block_table[b][t/16] at row t%16 (slot = block*16 + row).
 * The bit order lets the decode build tensor-core operands from stored words
 * with one logic operation per register.
 */
#ifndef TQ_KV_H
#define TQ_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int tq_status;
enum {
    TQ_OK = 0,
    TQ_ERR_INVALID_ARG = -1,      /* null pointer, size out of range, inconsistent config */
    TQ_ERR_UNSUPPORTED = -2,      /* d not in {128,256}, bits not in {2,3,4} (group-32: {2,4}),
                                     block != 16, H_q/H_kv > 4 and not a multiple of 4 (or > 16) */
    TQ_ERR_BUFFER_TOO_SMALL = -3, /* a caller buffer is smaller than tq_cache_sizes says */
    TQ_ERR_CUDA = -4,             /* a CUDA runtime call failed (launch, copy) */
    TQ_ERR_MISALIGNED = -5        /* a device pointer is not 16-byte aligned */
};

enum { TQ_DTYPE_F32 = 0, TQ_DTYPE_BF16 = 1 };
/*
 * Decode output flag, OR-ed into out_dtype: with MSE-quantised values, return
 * the attention output in the rotated space, R out = sum_t p_t n16_t c_v[idx_t],
 * leaving the inverse rotation R^T = D H / sqrt(d) to be folded into the
 * caller's output projection ([Roadmap] §3.2: the rotation can be absorbed
 * into the neighbouring weights).  TQ_ERR_INVALID_ARG with group-32 values
 * (their output is not rotated).
 */
enum { TQ_OUT_ROTATED = 0x100 };
enum { TQ_V_MSE = 0, TQ_V_G32 = 1 };
/*
 * Codebook of the rotated-coordinate quantiser (keys, and MSE values).
 * TQ_CODEBOOK_LLOYD: Lloyd-Max for the Beta-distributed coordinate ([Hub]
 * "Technical principle" step 2).  TQ_CODEBOOK_UNIFORM: equally spaced
 * centroids, a code dequantising as idx * step + c0 ([Roadmap] §4.3, SGLang's
 * "tq4u" mode), with the step that minimises the same distortion
 * (tq_make_uniform_codebook).  The cache layout is the same for both.
 */
enum { TQ_CODEBOOK_LLOYD = 0, TQ_CODEBOOK_UNIFORM = 1 };

/* Device error bits (tq_get_device_error). */
enum {
    TQ_DEVERR_SLOT = 1u << 0,      /* store: slot >= num_blocks*16 or < -1; token skipped */
    TQ_DEVERR_BLOCK = 1u << 1,     /* decode: block id outside [0, num_blocks); block skipped */
    TQ_DEVERR_SEQLEN = 1u << 2,    /* decode: seq_len < 0 or > 16*max_blocks_per_seq; clamped */
    TQ_DEVERR_TAIL = 1u << 3,      /* decode: tail_len < 0 or > tail_cap; clamped */
    TQ_DEVERR_TIMEOUT = 1u << 4,   /* a bounded wait (2^24 polls) on a staged tile or an MMA gave up; work abandoned */
    TQ_DEVERR_CHUNK = 1u << 5      /* extend: a token row outside every sequence's chunk (cu_q); its output is 0 */
};

typedef struct tq_cache_config {
    int32_t head_dim;           /* d, 128 or 256 ([Hub] step 2: codebooks for 128 and 256) */
    int32_t num_kv_heads;       /* H_kv >= 1 */
    int32_t num_q_heads;        /* H_q = G * H_kv with G <= 4 or G in {8, 12, 16}; q head h reads
                                   KV head h / G */
    int32_t block_size;         /* tokens per cache block; must be 16 */
    int64_t num_blocks;         /* blocks in the cache pool */
    int32_t k_bits;             /* key code bits, 2..4 */
    int32_t k_qjl;              /* 1: keys also keep ||r|| and sign(S r) ([Roadmap] §1); 0: MSE only */
    int32_t v_mode;             /* TQ_V_MSE (rotate + codebook) or TQ_V_G32 (uniform group-32) */
    int32_t v_bits;             /* value code bits: 2..4 (MSE), 2 or 4 (group-32) */
    uint64_t seed_rot;          /* seed of the rotation's +-1 diagonal */
    uint64_t seed_qjl;          /* seed of the d x d Gaussian QJL matrix S */
    int32_t max_batch;          /* sequences per decode call (grid size) */
    int32_t max_blocks_per_seq; /* columns of the block table */
    int32_t split_blocks;       /* cache blocks per decode split (fixed split-KV grid); >= 1 */
    int32_t tail_cap;           /* max exact bf16 "newest tokens" per sequence (0 = none) */
    int32_t k_codebook;         /* TQ_CODEBOOK_LLOYD (0) or TQ_CODEBOOK_UNIFORM */
    int32_t v_codebook;         /* the same for TQ_V_MSE values; must be 0 with TQ_V_G32 */
} tq_cache_config;

typedef struct tq_cache tq_cache;

/* Message for a status code (static storage; never NULL). */
const char* tq_status_string(tq_status s);

/*
 * The CUDA runtime's name and message for the most recent failing CUDA call
 * made by this library on the calling host thread (the cause behind a
 * TQ_ERR_CUDA status); "" if there was none.  The pointer stays valid until
 * the next library call on the same thread.  Diagnostic only: the pages have
 * no counterpart.
 */
const char* tq_last_cuda_error(void);

/*
 * Lloyd-Max codebook for one coordinate of a randomly rotated unit vector in
 * R^d ([Hub] step 2: the rotated coordinate is Beta distributed; density
 * f(t) ~ (1-t^2)^((d-3)/2) on [-1,1]).  Host only, deterministic.
 *   centroids  [2^bits]   ascending, symmetric (c[L-1-i] = -c[i])
 *   boundaries [2^bits-1] midpoints of neighbouring centroids
 *   mse        per-unit-vector distortion 1 - d*sum_i P_i c_i^2 (nullable)
 * d >= 3, 1 <= bits <= 8.  Buffers are caller-owned host memory.
 */
tq_status tq_make_codebook(int d, int bits, double* centroids, double* boundaries, double* mse);

/*
 * Uniform codebook for the same coordinate ([Roadmap] §4.3 "uniform" mode):
 * centroids c_i = step * (i - (2^bits - 1)/2), boundaries at the midpoints,
 * and the step that minimises the per-vector distortion.  For a fixed step
 * the nearest-neighbour cells are optimal; for fixed cells the distortion is
 * a quadratic in the step; the two alternate to the fixed point.
 *   centroids  [2^bits]   ascending, symmetric
 *   boundaries [2^bits-1]
 *   mse        per-unit-vector distortion d * E[(t - Q(t))^2] (nullable)
 * d >= 3, 1 <= bits <= 8.  Buffers are caller-owned host memory.
 */
tq_status tq_make_uniform_codebook(int d, int bits, double* centroids, double* boundaries, double* mse);

/*
 * The seeded parameters of a cache, host only (the library's own generator:
 * SplitMix64 counter stream, Steele-Lea-Flood 2014; the pages fix none).
 *   tq_make_rotation_signs: signs[i] = -1 if the top bit of draw i is set,
 *     else +1, i < d -- the diagonal D of R = H D / sqrt(d) ([Roadmap] §1
 *     randomised Walsh-Hadamard rotation).
 *   tq_make_qjl_matrix: S row-major (s_bf16[j*d + i]), N(0,1) entries by
 *     Box-Muller on consecutive draw pairs (cos branch, then sin), each rounded
 *     to the nearest bfloat16 ([Hub] step 3: the d x d random projection).
 * d >= 2 (even for the QJL matrix); buffers are caller-owned host memory.
 */
tq_status tq_make_rotation_signs(int d, uint64_t seed, float* signs);
tq_status tq_make_qjl_matrix(int d, uint64_t seed, uint16_t* s_bf16);

/*
 * Sizes, in bytes, of the caller-owned device buffers a configuration needs:
 *   page_bytes       one (block, KV head) page (layout above)
 *   cache_bytes      num_blocks * num_kv_heads * page_bytes
 *   params_bytes     rotation signs, QJL matrix, codebooks, device error word
 *   workspace_bytes  decode split partials and per-query projections
 * Any output pointer may be NULL.  Returns TQ_ERR_UNSUPPORTED/INVALID_ARG for a
 * bad configuration.
 */
tq_status tq_cache_sizes(const tq_cache_config* cfg, size_t* page_bytes, size_t* cache_bytes,
                         size_t* params_bytes, size_t* workspace_bytes);

/*
 * Build the parameter tables on the host (D from seed_rot, S from seed_qjl,
 * key/value codebooks) and upload them into params_dev (>= params_bytes, 256-
 * byte aligned); zero the device error word.  workspace_dev (>= workspace_bytes,
 * 16-byte aligned) is recorded for decode.  Synchronises `stream` once (setup
 * only).  The handle is freed with tq_cache_destroy; the device buffers stay
 * the caller's and must outlive the handle's use.
 */
tq_status tq_cache_create(const tq_cache_config* cfg, void* params_dev, void* workspace_dev, void* stream,
                          tq_cache** out);
tq_status tq_cache_destroy(tq_cache* cache);

/*
 * Copy the host-side parameter tables out (any pointer may be NULL):
 *   signs      [d]        +-1 diagonal of the rotation R = H D / sqrt(d)
 *   qjl_bf16   [d*d]      S row-major (S[j*d + i]), bfloat16 bit patterns
 *   k_centroids[2^k_bits], k_boundaries[2^k_bits - 1]
 *   v_centroids[2^v_bits], v_boundaries[2^v_bits - 1]   (TQ_V_MSE only)
 */
tq_status tq_cache_export_params(const tq_cache* cache, float* signs, uint16_t* qjl_bf16, double* k_centroids,
                                 double* k_boundaries, double* v_centroids, double* v_boundaries);

/*
 * Fused KV-cache store ([Roadmap] §3.1: rotation and quantisation fused into the
 * store; [Paged] "Which path vLLM takes": quantise, pack, write the paged cache).
 * For every token t with slot_mapping[t] >= 0 and every KV head g:
 *   keys:   n16 = fp16(||k||); y = R k/||k||; idx_i = #{boundaries < y_i};
 *           if k_qjl: r = k - n16 R^T c[idx], rnorm16 = fp16(||r||),
 *                     sign bit j = [(S r)_j >= 0]
 *   values: TQ_V_MSE as the key codes (own codebook), or TQ_V_G32 per 32
 *           coordinates: zero = fp16(min), scale = fp16((max-min)/(2^b-1)),
 *           q = clamp(floor((v - zero)/scale + 1/2), 0, 2^b-1) (0 if scale = 0)
 * and write the rows at block = slot/16, row = slot%16.
 *   k, v          device [num_tokens][num_kv_heads][d], in_dtype (TQ_DTYPE_*)
 *   slot_mapping  device int64 [num_tokens]; -1 skips the token; a slot outside
 *                 [0, num_blocks*16) also skips it and sets TQ_DEVERR_SLOT
 *   cache         device, cache_bytes
 * num_tokens == 0 is a no-op.
 */
tq_status tq_store(const tq_cache* cache, const void* k, const void* v, int in_dtype, int64_t num_tokens,
                   const int64_t* slot_mapping, void* cache_buf, void* stream);

/*
 * Decode attention over the compressed paged cache ([Paged]: decode reads the
 * compressed K/V through the block table; [Roadmap] §3.2 grouped query heads,
 * exp2 softmax, fixed split-KV grid; [Hub] "Technical principle": unbiased
 * score estimator; hybrid mode keeps the newest tokens exact).
 * For sequence b < batch and query head h (KV head g = h / (H_q/H_kv)):
 *   compressed token t < seq_lens[b]:
 *     s_t = scale*(n16_t <R q, c[idx_t]> + rnorm16_t sqrt(pi/2)/d <S q, 2 sign_t - 1>)
 *     v_t = n16_t R^T c_v[idx_t] (MSE) | q_t*scale16 + zero16 (G32)
 *   tail token u < tail_lens[b] (if tail_k != NULL): s_u = scale*<q, k_u>, v_u
 *   out[b][h] = sum_t softmax(s)_t v_t ; 0 when the sequence has no token.
 *   q           device [batch][H_q][d], q_dtype
 *   cache_buf   device, as written by tq_store
 *   block_table device int32 [batch][max_blocks_per_seq]
 *   seq_lens    device int32 [batch], compressed tokens, 0..16*max_blocks_per_seq
 *   tail_k/v    device bf16 [batch][H_kv][tail_cap][d] or NULL (no tail);
 *               16-byte aligned (else TQ_ERR_MISALIGNED)
 *   tail_lens   device int32 [batch] or NULL (no tail)
 *   scale       softmax scale; <= 0 means 1/sqrt(d)
 *   out         device [batch][H_q][d], out_dtype (TQ_DTYPE_F32 or TQ_DTYPE_BF16,
 *               optionally | TQ_OUT_ROTATED)
 * 1 <= batch <= max_batch.  The grid is fixed by (max_batch, H_kv, split count).
 */
tq_status tq_decode_attention(const tq_cache* cache, const void* q, int q_dtype, const void* cache_buf,
                              const int32_t* block_table, const int32_t* seq_lens, const void* tail_k,
                              const void* tail_v, const int32_t* tail_lens, float scale, int batch, void* out,
                              int out_dtype, void* stream);

/*
 * One decode step of the fused path ([Paged]: the new token's K/V are
 * compressed into the paged cache and the decode then reads the cache): the
 * same results, bit for bit, as tq_store(k, v, in_dtype, num_tokens,
 * slot_mapping) followed by tq_decode_attention(q, ...) on the same stream.
 * Arguments, layouts and errors are those of the two calls; every argument
 * of both is checked before anything launches, so an error status means
 * nothing was enqueued.  num_tokens == 0 stores nothing.
 * Ordering: q (like k and v) must be final when the call's first kernel
 * starts, i.e. written by work that precedes the call in the stream and that
 * finishes in plain stream order.  With num_tokens > 0 the decode's query
 * pass then reads q while the store kernel runs; it writes nothing before the
 * store completes.
 */
tq_status tq_store_decode_attention(const tq_cache* cache, const void* k, const void* v, int in_dtype,
                                    int64_t num_tokens, const int64_t* slot_mapping, const void* q, int q_dtype,
                                    void* cache_buf, const int32_t* block_table, const int32_t* seq_lens,
                                    const void* tail_k, const void* tail_v, const int32_t* tail_lens, float scale,
                                    int batch, void* out, int out_dtype, void* stream);

/*
 * Extend (prefill) attention over the compressed paged cache ([Roadmap] §4.1:
 * the extend kernel, like the decode kernel, reads the compressed pool
 * directly).  Sequence b < batch brings n_b = cu_q[b+1] - cu_q[b] new tokens:
 * rows cu_q[b] .. cu_q[b+1]-1 of q, new_k and new_v.  Its first
 * prefix_lens[b] tokens are in the cache (block-table row b).  New token j of
 * the chunk attends to every prefix token as tq_decode_attention scores it and
 * to new tokens 0..j with their exact bf16 keys and values (causal), in one
 * softmax:
 *   out[cu_q[b] + j][h] = tq_decode_attention of that query over the prefix
 *                         with new tokens 0..j as its tail.
 * (The new tokens are stored into the cache separately, by tq_store.)
 *   q            device [n_tokens][H_q][d], q_dtype
 *   block_table  device int32 [batch][max_blocks_per_seq]
 *   prefix_lens  device int32 [batch], 0..16*max_blocks_per_seq
 *   cu_q         device int32 [batch+1], non-decreasing, cu_q[0] = 0,
 *                cu_q[batch] = n_tokens.  A row of q that no chunk holds gets
 *                out = 0 and sets TQ_DEVERR_CHUNK; every row a chunk names
 *                lies in [0, n_tokens).  A cu_q that decreases or leaves
 *                [0, n_tokens] also sets TQ_DEVERR_CHUNK; the rows it names
 *                are clamped into [0, n_tokens) and their outputs are then
 *                unspecified.
 *   new_k/new_v  device bf16 [n_tokens][H_kv][d], 16-byte aligned
 *   scale, out_dtype as for tq_decode_attention; out device [n_tokens][H_q][d]
 * Each token is one entry of the workspace (its split partials, as in the
 * decode): n_tokens <= max_batch, and a chunk may hold at most tail_cap
 * tokens (tail_cap >= 1; a longer chunk is clamped and sets TQ_DEVERR_TAIL).
 * At d = 128 with head groups of four query heads and at most six score
 * planes, blocks of 8 new tokens of a chunk (and one head group of four query
 * heads) share one tensor-core pass over every prefix tile; other configurations
 * run the decode kernels over one entry per new token.  The results agree to
 * the decode's error bar either way.  A prefix block id outside
 * [0, num_blocks) is skipped and sets TQ_DEVERR_BLOCK.  Uses the cache's
 * workspace, like tq_decode_attention.  n_tokens == 0 is a no-op.
 */
tq_status tq_extend_attention(const tq_cache* cache, const void* q, int q_dtype, const void* cache_buf,
                              const int32_t* block_table, const int32_t* prefix_lens, const int32_t* cu_q,
                              const void* new_k, const void* new_v, float scale, int batch, int n_tokens, void* out,
                              int out_dtype, void* stream);

/*
 * Profiling hook: record the caller's CUDA events (cudaEvent_t, passed as
 * void*) on the call's stream immediately before and after the named kernel
 * in every later tq_store (TQ_PROF_STORE) or tq_decode_attention
 * (TQ_PROF_DECODE_SPLIT: the split-KV kernel, the decode's dominant launch).
 * NULL events switch the hook off.  The events stay the caller's.
 */
enum { TQ_PROF_STORE = 0, TQ_PROF_DECODE_SPLIT = 1 };
tq_status tq_set_profile_events(tq_cache* cache, int kernel, void* start_event, void* stop_event);

/*
 * Tuning: tq_store encodes at most `max_vectors` (token, KV head) vectors with
 * one CTA per vector, without staging S in shared memory (the latency-bound
 * shape of a decode step's new tokens), and larger calls with a bulk kernel
 * (tiles of 128 vectors on the tensor cores for d = 128 bf16 inputs, else
 * eight vectors per CTA).  Every path computes the same definition; their
 * fp32 sums round in different orders, so their bytes can differ only in the
 * boundary cases where such a rounding decides a code, an fp16 field or a sign.
 * A negative value restores the default, 16 x the device's SM count.
 * Process-wide; takes effect for later calls.  Returns TQ_OK.
 */
tq_status tq_set_store_small_max(int64_t max_vectors);

/*
 * Read and clear the device error word (TQ_DEVERR_* bits).  Synchronises
 * `stream`; the only synchronising call besides tq_cache_create.
 */
tq_status tq_get_device_error(const tq_cache* cache, uint32_t* flags, void* stream);

/*
 * Diagnostic; the pages have no counterpart.  Every wait of the store and
 * decode kernels on an mbarrier (a staged page, a tensor-core result) is
 * bounded: after 2^24 unsuccessful polls it gives up, sets TQ_DEVERR_TIMEOUT,
 * drains its copies in flight and returns, so a stalled copy becomes an error
 * status instead of a hung GPU.  This call launches one thread that makes that
 * wait (the same polling loop, with a time limit of limit_us microseconds,
 * 1 .. 4 * 10^6, added) on an mbarrier nothing ever completes, and OR-s
 * TQ_DEVERR_TIMEOUT into *err_word (caller-owned device uint32, 4-byte
 * aligned) when it gives up.  Asynchronous on `stream`; lets a test check that
 * a wait that runs out ends its kernel with the error bit set and leaves the
 * context usable.
 */
tq_status tq_check_wait_timeout(uint32_t* err_word, uint32_t limit_us, void* stream);

/*
 * Decode attention that allocates nothing and takes no workspace buffer.
 * The paper has no counterpart: this is an interface for callers that cannot
 * allocate device memory themselves -- an engine whose block manager
 * pre-budgets every byte of the GPU (a library cudaMalloc would bypass its
 * accounting or fail once the pool has taken the memory), or code that must
 * not risk the device-wide synchronisation a cudaMalloc can cause.
 *
 * Same arguments, results and errors as tq_decode_attention, except that the
 * split-KV scratch lives in one file-scope device array of
 * TQ_NOALLOC_SCRATCH_BYTES per GPU (reserved on every GPU that loads the
 * library's module, held until the process exits) instead of the handle's
 * workspace, which this call never touches.
 *   - Returns TQ_ERR_BUFFER_TOO_SMALL, launching nothing, when the
 *     configuration's workspace (tq_cache_sizes) exceeds the array.
 *   - The first call on a device looks the array up (cudaGetSymbolAddress)
 *     with that device current; make that first call before any stream
 *     capture.
 *   - All calls share the array and it keeps the last call's contents; every
 *     byte a call reads was written earlier by the same call.  Calls whose
 *     kernels overlap on the GPU (other streams, other threads) race on it:
 *     order them on one stream.
 * Calls no cudaMalloc, cudaFree or allocating library routine.
 */
#define TQ_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
tq_status tq_decode_attention_noalloc(const tq_cache* cache, const void* q, int q_dtype, const void* cache_buf,
                                      const int32_t* block_table, const int32_t* seq_lens, const void* tail_k,
                                      const void* tail_v, const int32_t* tail_lens, float scale, int batch,
                                      void* out, int out_dtype, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TQ_KV_H */
