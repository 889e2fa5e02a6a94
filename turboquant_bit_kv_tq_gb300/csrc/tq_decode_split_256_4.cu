// Split-KV decode kernels for head dim 256, 4-bit keys.
#include "tq_decode_kernels.cuh"

namespace tq {

template <>
tq_status dispatch_split<256, 4>(const DecodeArgs& a, cudaStream_t s, size_t smem, int grid) {
    if (grid > 0) return TQ_ERR_UNSUPPORTED;  // score planes exceed one tensor-memory A buffer
    return dispatch_nth<256, 4>(a, s, smem);
}

}  // namespace tq
