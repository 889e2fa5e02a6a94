// Decode attention without any allocation and without the handle's
// workspace: the split-KV scratch is a file-scope device array.  For callers
// that cannot allocate device memory themselves (an engine that pre-budgets
// the whole GPU, code that must not trigger the synchronisation of a
// cudaMalloc).  The kernels are the ordinary decode kernels; only where their
// scratch lives differs.

#include <mutex>

#include "tq_decode_kernels.cuh"

namespace tq {

constexpr size_t kNoAllocScratch = TQ_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Reserved on every GPU that loads this module; lives until process exit.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratch];

// Device address of the array on the current device, looked up once per
// device.  In host code g_noalloc_scratch is only a host-side stand-in, never
// a device pointer.
static tq_status scratch_address(uint8_t** out) {
    static std::mutex mu;
    static uint8_t* addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return TQ_ERR_CUDA;
        addr[dev] = static_cast<uint8_t*>(p);
    }
    *out = addr[dev];
    return TQ_OK;
}

}  // namespace tq

using namespace tq;

extern "C" tq_status tq_decode_attention_noalloc(const tq_cache* c, const void* q, int q_dtype,
                                                 const void* cache_buf, const int32_t* block_table,
                                                 const int32_t* seq_lens, const void* tail_k, const void* tail_v,
                                                 const int32_t* tail_lens, float scale, int batch, void* out,
                                                 int out_dtype, void* stream) {
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
    const WorkspaceLayout wl = workspace_layout(c->cfg);
    if (wl.total > kNoAllocScratch) return TQ_ERR_BUFFER_TOO_SMALL;
    uint8_t* ws = nullptr;
    const tq_status st = scratch_address(&ws);
    if (st != TQ_OK) return st;
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
    a.out_rotated = out_rot;
    a.k_uniform = c->cfg.k_codebook == TQ_CODEBOOK_UNIFORM;
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
    a.gm = c->geom;
    // every scratch byte read below is written earlier by the same call
    a.ws_q = reinterpret_cast<float*>(ws + wl.q);
    a.ws_bimg = ws + wl.bimg;
    a.ws_cst = reinterpret_cast<float*>(ws + wl.cst);
    a.ws_acc = reinterpret_cast<float*>(ws + wl.acc);
    a.ws_ml = reinterpret_cast<float*>(ws + wl.ml);
    cudaStream_t s = (cudaStream_t)stream;
    return launch_decode(a, s, nullptr, nullptr);
}
