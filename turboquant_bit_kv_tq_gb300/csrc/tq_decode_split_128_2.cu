// Split-KV decode kernels for head dim 128, 2-bit keys.
#include "tq_decode_ws.cuh"

namespace tq {

template <>
tq_status dispatch_split<128, 2>(const DecodeArgs& a, cudaStream_t s, size_t smem, int grid) {
    // two planes whatever the codebook: every 2-bit symmetric codebook has
    // only single-bit terms
    if (grid > 0) return dispatch_ws_v<128, 2, false, 1>(a, s, smem, grid);
    return dispatch_nth<128, 2>(a, s, smem);
}

}  // namespace tq
