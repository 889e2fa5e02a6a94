// Split-KV decode kernels for head dim 128, 3-bit keys.
#include "tq_decode_ws.cuh"

namespace tq {

template <>
tq_status dispatch_split<128, 3>(const DecodeArgs& a, cudaStream_t s, size_t smem, int grid) {
    if (grid > 0)
        return a.gm.npk == 3 ? dispatch_ws_uniform<128, 3>(a, s, smem, grid)
                             : dispatch_ws_v<128, 3, false, 1>(a, s, smem, grid);
    return dispatch_nth<128, 3>(a, s, smem);
}

}  // namespace tq
