// Device helpers shared by the store and decode kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "tq_internal.h"

namespace tq {

// Programmatic dependent launch.  A kernel launched with launch_pdl may start
// while the previous kernel in the stream is still running: it must pdl_wait()
// before it reads that kernel's results (the wait returns once the previous
// grid has completed and its writes are visible; without a programmatic
// launch it returns at once).  pdl_launch_dependents() lets the next kernel
// start early.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// (pdl false: an ordinary launch, e.g. next to a profiling event record)
template <typename... P, typename... A>
inline cudaError_t launch_pdl(bool pdl, void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<A&&>(args)...);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

template <typename T>
__device__ __forceinline__ float load_as_float(const T* p);
template <>
__device__ __forceinline__ float load_as_float<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float load_as_float<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}

// In-warp unnormalised Walsh-Hadamard transform (Sylvester order, y = H x) of
// a length-32*PER vector whose element i = lane + 32*k sits in x[k] of lane
// `lane`.  Butterfly span h pairs (i, i^h): for h < 32 the partner is lane^h
// (shuffle), for h >= 32 it is slot k^(h/32) of the same lane.
template <int PER>
__device__ __forceinline__ void fwht_warp(float (&x)[PER], int lane) {
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
        // lower lane: x + other; upper lane: other - x (one exact fma by +-1)
        const float sgn = (lane & h) ? -1.f : 1.f;
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const float other = __shfl_xor_sync(0xffffffffu, x[k], h);
            x[k] = fmaf(sgn, x[k], other);
        }
    }
#pragma unroll
    for (int s = 1; s < PER; s <<= 1) {
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            if (!(k & s)) {
                const float a = x[k], b = x[k | s];
                x[k] = a + b;
                x[k | s] = a - b;
            }
        }
    }
}

__device__ __forceinline__ void set_error(uint32_t* err, uint32_t bit) { atomicOr(err, bit); }

}  // namespace tq
