// Warp-specialized split-KV kernels for head dim 128, 3-bit keys on a uniform
// codebook (three key planes instead of four).
#include "tq_decode_ws.cuh"

namespace tq {

template <>
tq_status dispatch_ws_uniform<128, 3>(const DecodeArgs& a, cudaStream_t s, size_t smem, int grid) {
    return dispatch_ws_v<128, 3, true, 1>(a, s, smem, grid);
}

}  // namespace tq
