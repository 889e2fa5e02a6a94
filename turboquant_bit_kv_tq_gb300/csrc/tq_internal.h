// Private to the library: the cache handle, page layout and the kernel
// launchers shared between tq_host.cpp, tq_store.cu and tq_decode.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "tq_kv.h"

namespace tq {

constexpr int kBlock = 16;  // tokens per cache block
constexpr int kMaxLevels = 16;

// Byte offsets of the planes of one (block, KV head) page; see tq_kv.h.
struct Layout {
    int d, k_bits, v_bits, k_qjl, v_mode;
    int k_code_row, k_sign_row, v_code_row, v_meta_row;  // bytes per token row
    int k_codes, k_signs, k_norm, k_rnorm, v_codes, v_meta;  // plane offsets
    int page_bytes;
};

// Device pointers into the caller's params buffer.
struct DeviceParams {
    const float* signs;      // [d] +-1
    const float* s_f32;      // S row-major [d][d]
    const float* st_f32;     // S^T [d][d] (st[i*d + j] = S[j][i])
    const uint16_t* s_bf16;  // S row-major, bf16 bits
    const uint16_t* st_bf16; // S^T, bf16 bits
    const float* k_cent;     // [16] key centroids (padded)
    const float* k_bound;    // [16] key boundaries
    const float* v_cent;     // [16] value centroids (MSE)
    const float* v_bound;    // [16]
    // code value = alpha + sum_P beta[P] * u_P(code bits), u_P = XOR of the
    // code bits in the P-th odd subset (plane_subset); [0] = alpha
    const float* k_walsh;    // [1 + 8]
    const float* v_walsh;    // [1 + 8] (MSE values)
    // T = S R^T = S D H / sqrt(d) as fp16 high and low parts (T ~ t_hi + t_lo
    // to ~22 significant bits), row-major [d][d]: the tensor-core store projects
    // the rotated residual with it (S r = T R r)
    const uint16_t* t_hi;
    const uint16_t* t_lo;
    uint32_t* err;           // device error word
};

// Odd-size subsets of the code bits: the planes of a b-bit symmetric codebook
// (2^(b-1) of them), the b single bits first (all a uniform codebook has), then
// the rest in increasing mask order.
__host__ __device__ constexpr int plane_subset(int bits, int i) {
    return bits == 2 ? (i == 0 ? 1 : 2)
         : bits == 3 ? (i == 0 ? 1 : i == 1 ? 2 : i == 2 ? 4 : 7)
                     : (i == 0 ? 1 : i == 1 ? 2 : i == 2 ? 4 : i == 3 ? 8 : i == 4 ? 7 : i == 5 ? 11 : i == 6 ? 13 : 14);
}

// Split-KV geometry of a configuration.
struct Splits {
    int n_chunks;  // ceil(max_blocks_per_seq / split_blocks)
    int n_splits;  // n_chunks + (tail_cap > 0)
};

struct ParamsLayout {
    size_t signs, s_f32, st_f32, s_bf16, st_bf16, k_cent, k_bound, v_cent, v_bound, k_walsh, v_walsh, t_hi, t_lo, err,
        total;
};

// Query-side fp8 pieces of the score contraction: piece k carries the
// residual of pieces 0..k-1 times 16^k, ~4 significant bits each (~16 in all,
// a relative error of ~2^-17 per operand element).
constexpr int kPieces = 4;

// Decode geometry.  One split CTA serves a head group of hc query heads
// (nhg groups per KV head); its value contraction runs in nth n-tiles of 4
// heads; the score contraction has npl planes (npk key code planes + the QJL
// sign plane) and n_cols columns, kPieces per head (4 nth heads, rounded up to
// a multiple of 16).  bimg_bytes is the score operand image of one head group:
// n_cols rows of npl*d fp8 bytes in the tensor-core shared-memory layout.
struct DecodeGeom {
    int hc, nhg, nth, npk, npl, n_cols, bimg_bytes;
};
DecodeGeom decode_geom(const tq_cache_config& c);

struct WorkspaceLayout {
    // bimg: [B][Hkv][nhg][bimg_bytes] (score operands); cst: [B][Hq][4] fp32; acc: [B][Hq][S][d]; ml: [B][Hq][S][2];
    // ext: 4 x [B] int32 (extend attention's per-token lengths and rows), then
    // 4 int32 and [B] int4 (the extend prefix kernel's query blocks)
    size_t bimg, cst, acc, ml, ext, total;
};

// TQ_OK for cudaSuccess; otherwise records the runtime's message for
// tq_last_cuda_error (per host thread) and returns TQ_ERR_CUDA
tq_status cuda_status(cudaError_t e);
// the same, with printf-style context appended to the message
tq_status cuda_status_detail(cudaError_t e, const char* fmt, ...);
// TQ_ERR_CUDA with a printf-style message for a failed driver-level step
tq_status driver_failure(const char* fmt, ...);

// Per-device launch set-up, safe to call from any host thread, any number of
// times: the current device's SM count (looked up once per device), and
// raising `func`'s dynamic shared-memory limit to at least `bytes` on the
// current device (done once per device and kernel).  Both run on the first
// call of an entry point on a device, so that call should precede any stream
// capture on it.
tq_status device_sms(int* sms);
tq_status ensure_dynamic_smem(const void* func, int bytes, const char* name);

tq_status compute_layout(const tq_cache_config& c, Layout* lay);
Splits compute_splits(const tq_cache_config& c);
ParamsLayout params_layout(const tq_cache_config& c);
WorkspaceLayout workspace_layout(const tq_cache_config& c);

}  // namespace tq

struct tq_cache {
    tq_cache_config cfg;
    tq::Layout lay;
    tq::Splits splits;
    tq::DeviceParams dp;
    tq::DecodeGeom geom;
    uint8_t* ws_bimg;
    float* ws_cst;
    float* ws_acc;
    float* ws_ml;
    int32_t* ws_ext;
    // profiling events (cudaEvent_t) around the store / decode-split kernels
    void* prof_start[2] = {nullptr, nullptr};
    void* prof_stop[2] = {nullptr, nullptr};
    // host copies of the tables
    std::vector<float> signs;
    std::vector<uint16_t> s_bf16;
    std::vector<double> k_cent, k_bound, v_cent, v_bound;
};
