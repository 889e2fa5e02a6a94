// Store path: arguments shared by the store kernels, and the tensor-core bulk
// store's launcher (tq_store_tc.cu).
#pragma once

#include "tq_device.cuh"

namespace tq {

struct StoreArgs {
    const void* k;
    const void* v;
    const int64_t* slots;
    uint8_t* cache;
    int64_t num_tokens;
    int64_t num_slots;  // num_blocks * 16
    int heads;
    Layout lay;
    DeviceParams dp;
};

// Whether the tensor-core bulk store serves a call: d = 128, bf16 inputs,
// symmetric codebooks (every codebook the library makes is), K and V rows
// 16-byte aligned (bulk-tensor copies) and fewer than 2^31 vectors.
inline bool store_tc_supported(const StoreArgs& a, int in_dtype) {
    const auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    return a.lay.d == 128 && in_dtype == TQ_DTYPE_BF16 && al(a.k) && al(a.v) &&
           a.num_tokens * a.heads < ((int64_t)1 << 31);
}

// Launch the tensor-core bulk store on at most `sms` CTAs (one per SM).
tq_status launch_store_tc(const StoreArgs& a, cudaStream_t s, int sms);

}  // namespace tq
