// Split-KV decode kernels for head dim 128, 4-bit keys.
#include "tq_decode_ws.cuh"

namespace tq {

template <>
tq_status dispatch_split<128, 4>(const DecodeArgs& a, cudaStream_t s, size_t smem, int grid) {
    // a Lloyd-Max codebook's eight score planes exceed one tensor-memory A
    // buffer; a uniform one's four fit, so those keys run warp-specialized
    if (grid > 0) return a.gm.npk == 4 ? dispatch_ws_v<128, 4, true, 1>(a, s, smem, grid) : TQ_ERR_UNSUPPORTED;
    return dispatch_nth<128, 4>(a, s, smem);
}

}  // namespace tq
