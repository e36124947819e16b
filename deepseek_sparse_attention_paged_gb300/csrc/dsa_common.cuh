// dsa_common.cuh -- small device/host helpers shared by the DSA kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa.h"

namespace dsa {

constexpr int kPage = 64;                 // tokens per page (both caches)
constexpr int kIndexHeads = 64;           // lightning-indexer heads
constexpr int kIndexDim = 128;            // lightning-indexer head dim
constexpr int kIndexPageBytes = 64 * 132; // 64 x (128 FP8 codes + fp32 scale), page-blocked
constexpr int kIndexScaleOffset = 64 * 128;
constexpr int kC8PageBytes = 64 * 130;    // int8 ("c8") index cache: 64 x 128 codes, then 64 fp16 scales
constexpr int kC8ScaleOffset = 64 * 128;
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

// Error of the fp32 sum s = a + b (Knuth's TwoSum: s + err == a + b exactly).
__device__ __forceinline__ float two_sum_err(float a, float b, float s) {
    const float bb = __fsub_rn(s, a);
    return __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// The int8 ("c8") indexer transform of one 128-vector held by a warp (lane l: elements 4l .. 4l+3,
// exact fp32 values of bf16 numbers).  Follows vllm-ascend sfa_v1.py with use_sparse_c8_indexer:
// x @ qk_hadamard, where qk_hadamard = bf16(scipy.linalg.hadamard(128)) / 128**0.5 has entries +-c,
// c = bf16(128^-0.5) = 181 * 2^-11; then npu_dynamic_quant to int8 with one scale per vector.
//   * y_j = bf16(c * sum_i (-1)^popcount(i & j) x_i), the exact value rounded once: the Sylvester
//     butterflies (h = 1, 2 inside the lane, 4 .. 64 across lanes l ^ h / 4) run in fp32 with every
//     add checked exact by TwoSum; c * S is the fp32 product p plus its exact FMA error e, and the
//     one rounding of p + e to bf16 equals that of p except when p sits on a bf16 midpoint, where p
//     is first moved one fp32 ulp towards p + e.  If any add of the warp's vector was inexact (an
//     exponent spread beyond fp32's 24 bits) or a product is too small for the FMA error to be
//     exact, the warp redoes the vector in fp64, where sums of 128 bf16 values are exact;
//   * scale = amax / 127 (fp32, IEEE division); code = round-to-nearest-even(y / scale) (fp32 IEEE
//     division), within [-127, 127]; all codes 0 when amax = 0.
// Returns the lane's 4 codes packed little-endian; *scale_out = the fp32 scale.
__device__ __forceinline__ uint32_t c8_rotate_quant(const float (&xin)[4], int lane, float* scale_out) {
    constexpr float kCf = 181.0f / 2048.0f;
    constexpr double kC = 181.0 / 2048.0;
    float y[4];
    {
        float x[4] = {xin[0], xin[1], xin[2], xin[3]};
        bool inexact = false;
        auto bfly = [&](float& lo, float& hi) {
            const float a = lo, b = hi;
            lo = __fadd_rn(a, b);
            hi = __fsub_rn(a, b);
            inexact |= two_sum_err(a, b, lo) != 0.0f || two_sum_err(a, -b, hi) != 0.0f;
        };
        bfly(x[0], x[1]);
        bfly(x[2], x[3]);
        bfly(x[0], x[2]);
        bfly(x[1], x[3]);
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float other = __shfl_xor_sync(0xffffffffu, x[e], m);
                const float a = upper ? other : x[e];
                const float b = upper ? -x[e] : other;
                x[e] = __fadd_rn(a, b);
                inexact |= two_sum_err(a, b, x[e]) != 0.0f;
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float p = __fmul_rn(x[e], kCf);
            const float err = __fmaf_rn(x[e], kCf, -p);
            if (x[e] != 0.0f && !(fabsf(p) >= 0x1p-100f)) inexact = true;   // also catches inf / NaN
            const uint32_t pb = __float_as_uint(p);
            if ((pb & 0xffffu) == 0x8000u && err != 0.0f)                      // on a bf16 midpoint
                p = __uint_as_float(((err > 0.0f) == (p > 0.0f)) ? pb + 1u : pb - 1u);
            y[e] = __bfloat162float(__float2bfloat16_rn(p));
        }
        if (__any_sync(0xffffffffu, inexact)) {
            double d[4] = {xin[0], xin[1], xin[2], xin[3]};
            {
                double a = d[0], b = d[1];
                d[0] = a + b; d[1] = a - b;
                a = d[2]; b = d[3];
                d[2] = a + b; d[3] = a - b;
            }
            {
                double a = d[0], b = d[2];
                d[0] = a + b; d[2] = a - b;
                a = d[1]; b = d[3];
                d[1] = a + b; d[3] = a - b;
            }
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
                const bool upper = (lane & m) != 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const double other = __shfl_xor_sync(0xffffffffu, d[e], m);
                    d[e] = upper ? other - d[e] : d[e] + other;
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) y[e] = __bfloat162float(__double2bfloat16(d[e] * kC));
        }
    }
    const float amax = warp_max(fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3]))));
    const float scale = __fdiv_rn(amax, 127.0f);
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        int c = 0;
        if (amax > 0.0f) c = max(-127, min(127, __float2int_rn(__fdiv_rn(y[e], scale))));
        packed |= static_cast<uint32_t>(c & 0xff) << (8 * e);
    }
    *scale_out = scale;
    return packed;
}

// Four int8 values (packed little-endian) -> four f16 (exact), as two f16x2 words: with u = b ^ 0x80
// (the value + 128), the f16 bits 0x6400 | u encode 1024 + u, and subtracting 1152 leaves the value.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
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
dsa_status indexer_logits_c8_launch(const void* q_bf16, const float* weights, const uint8_t* index_k_pool_c8,
                                    int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                    const int32_t* seq_lens, const int32_t* cu_q, int32_t B, int32_t max_seq_len,
                                    int32_t max_q_len, int32_t row_begin, int32_t row_end, float* logits, int64_t ld,
                                    void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream);
dsa_status topk_launch(const float* logits, int64_t ld, const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                       int32_t max_seq_len, int32_t row_begin, int32_t row_end, int32_t k, int32_t n_init,
                       int32_t n_local, int32_t* idx, void* stream, const uint32_t* hist_g, int32_t cmp_shift = 0);

}  // namespace dsa
