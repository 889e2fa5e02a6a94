// Split-KV decode kernels for head dim 128, 3-bit keys.
#include "tq_decode_kernels.cuh"

namespace tq {

template <>
tq_status dispatch_split<128, 3>(const DecodeArgs& a, cudaStream_t s, size_t smem) {
    return dispatch_nth<128, 3>(a, s, smem);
}

}  // namespace tq
