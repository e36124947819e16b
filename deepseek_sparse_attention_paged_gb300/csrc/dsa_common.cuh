// dsa_common.cuh -- small device/host helpers shared by the DSA kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa.h"

namespace dsa {

constexpr int kPage = 64;                 // tokens per page (both caches)
constexpr int kIndexHeads = 64;           // lightning-indexer heads
constexpr int kIndexDim = 128;            // lightning-indexer head dim
constexpr int kIndexPageBytes = 64 * 132; // 64 x (128 FP8 codes + fp32 scale), page-blocked
constexpr int kIndexScaleOffset = 64 * 128;
constexpr int kLatentDim = 576;           // 512 latent + 64 rope
constexpr int kValueDim = 512;

// OR a bit into the caller's device error word (nullable).
__device__ __forceinline__ void raise_error(int32_t* err, int32_t bit) {
    if (err != nullptr) atomicOr(err, bit);
}

__device__ __forceinline__ float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t packed) { return __uint_as_float(packed & 0xffff0000u); }

// Request of global query row r: the b with cu_q[b] <= r < cu_q[b+1] (binary search).
__device__ __forceinline__ int row_request(const int32_t* __restrict__ cu_q, int B, int r) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu_q + mid) <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Keys visible to row j of a request with L cached tokens and q_len query tokens: the row sits
// at absolute position L - q_len + j and sees positions [0, L - q_len + j].
__device__ __forceinline__ int visible_len(int L, int q_len, int j) {
    int v = L - q_len + j + 1;
    return v < 0 ? 0 : v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Multiprocessor count of the current device (the launch heuristics size grids by it); `fallback`
// when no device can be queried (a size query made without a GPU).
inline int device_sm_count(int fallback = 152) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
        cudaGetLastError();   // leave no sticky error behind
        return fallback;
    }
    return sms;
}

inline dsa_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

// Internal launchers shared by the one-call indexer: the logits call and the top-k call, each with
// an optional per-row 4096-bin histogram of the top 12 bits of the logits' order keys (written by
// the logits kernel into zeroed memory, read by the top-k kernels instead of a first pass).
constexpr int kHistBins = 4096;
dsa_status indexer_logits_launch(const void* q_bf16, const float* weights, const uint8_t* index_k_pool,
                                 int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                 const int32_t* seq_lens, const int32_t* cu_q, int32_t B, int32_t max_seq_len,
                                 int32_t max_q_len, int32_t row_begin, int32_t row_end, float* logits, int64_t ld,
                                 uint32_t flags, void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream,
                                 uint32_t* hist_g);
dsa_status topk_launch(const float* logits, int64_t ld, const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                       int32_t max_seq_len, int32_t row_begin, int32_t row_end, int32_t k, int32_t n_init,
                       int32_t n_local, int32_t* idx, void* stream, const uint32_t* hist_g);

}  // namespace dsa
