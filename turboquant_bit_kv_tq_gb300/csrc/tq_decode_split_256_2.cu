// Split-KV decode kernels for head dim 256, 2-bit keys.
#include "tq_decode_ws.cuh"

namespace tq {

template <>
tq_status dispatch_split<256, 2>(const DecodeArgs& a, cudaStream_t s, size_t smem, int grid) {
    if (grid > 0) return dispatch_ws_v<256, 2, false, 1>(a, s, smem, grid);
    return dispatch_nth<256, 2>(a, s, smem);
}

}  // namespace tq
