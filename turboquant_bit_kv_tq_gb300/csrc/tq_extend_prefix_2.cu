// Extend prefix kernels (head dim 128) for 2-bit keys, every value mode.
#include "tq_extend_prefix.cuh"

namespace tq {

template <>
tq_status dispatch_extend_prefix<2, false>(const DecodeArgs& a, cudaStream_t s, int grid) {
    return xp_dispatch_v<2, false>(a, s, grid);
}

}  // namespace tq
