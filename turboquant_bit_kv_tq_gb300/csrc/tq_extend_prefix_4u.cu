// Extend prefix kernels (head dim 128) for 4-bit keys on a uniform codebook (4 key planes), every value mode.
#include "tq_extend_prefix.cuh"

namespace tq {

template <>
tq_status dispatch_extend_prefix<4, true>(const DecodeArgs& a, cudaStream_t s, int grid) {
    return xp_dispatch_v<4, true>(a, s, grid);
}

}  // namespace tq
