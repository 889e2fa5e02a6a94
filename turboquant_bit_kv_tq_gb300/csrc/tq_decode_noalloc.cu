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
    DecodeArgs a;
    const tq_status st = decode_args(c, q, q_dtype, cache_buf, block_table, seq_lens, tail_k, tail_v, tail_lens,
                                     scale, batch, out, out_dtype, &a);
    if (st != TQ_OK) return st;
    const WorkspaceLayout wl = workspace_layout(c->cfg);
    if (wl.total > kNoAllocScratch) return TQ_ERR_BUFFER_TOO_SMALL;
    uint8_t* ws = nullptr;
    const tq_status sa = scratch_address(&ws);
    if (sa != TQ_OK) return sa;
    // every scratch byte read below is written earlier by the same call
    a.ws_bimg = ws + wl.bimg;
    a.ws_cst = reinterpret_cast<float*>(ws + wl.cst);
    a.ws_acc = reinterpret_cast<float*>(ws + wl.acc);
    a.ws_ml = reinterpret_cast<float*>(ws + wl.ml);
    return launch_decode(a, (cudaStream_t)stream, nullptr, nullptr);
}
