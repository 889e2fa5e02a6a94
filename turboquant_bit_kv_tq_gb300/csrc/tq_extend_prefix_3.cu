// Extend prefix kernels (head dim 128) for 3-bit keys, every value mode.
#include "tq_extend_prefix.cuh"

namespace tq {

template <>
tq_status dispatch_extend_prefix<3, false>(const DecodeArgs& a, cudaStream_t s, int grid) {
    return xp_dispatch_v<3, false>(a, s, grid);
}

}  // namespace tq
