// store_index_k.cu -- Hadamard-rotate, FP8-quantise and scatter new indexer keys into the paged
// index-K cache.
//
// Follows sglang dsa_indexer.py, Indexer._store_index_k_cache (quantise per 128 values with an
// fp32 scale, write codes and scale at the token's slot) and rotate_activation (Walsh-Hadamard
// transform with scale 128^-0.5, applied to the bf16 key before quantisation).
//
// One warp per token; lane l holds key elements 4l .. 4l+3.  The butterfly network is the
// Sylvester-order one (h = 1, 2, ..., 64; (a, b) -> (a + b, a - b)) evaluated in fp32: levels
// h = 1, 2 stay inside a lane, levels 4 .. 64 pair lane l with lane l ^ (h / 4).  Every output of
// every level is the same fp32 add or subtract of the same two inputs as in the sequential
// definition, so the rotated key is bit-identical to it.  The work is HBM-bound: 256 bytes read
// and 132 bytes written per token.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "dsa_common.cuh"

namespace dsa {
namespace {

// fp32 value nearest to 1/sqrt(128) = 2^-3.5.
constexpr float kInvSqrt128 = 0x1.6a09e6p-4f;

__global__ void __launch_bounds__(256)
store_index_k_kernel(const uint16_t* __restrict__ keys, const int64_t* __restrict__ slots, int64_t n,
                     uint8_t* __restrict__ pool, int64_t num_pages, int32_t* err) {
    const int64_t token = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (token >= n) return;                      // warp-uniform
    const int64_t slot = __ldg(slots + token);
    if (slot < 0) return;                        // padding token
    const int64_t page = slot >> 6;
    const int row = static_cast<int>(slot & 63);
    if (page >= num_pages) {
        if (lane == 0) raise_error(err, DSA_DEVERR_SLOT_RANGE);
        return;
    }

    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(keys + token * kIndexDim) + lane);
    float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};

    // h = 1: pairs (0,1), (2,3) of this lane's elements
    {
        float a = x[0], b = x[1];
        x[0] = a + b; x[1] = a - b;
        a = x[2]; b = x[3];
        x[2] = a + b; x[3] = a - b;
    }
    // h = 2: pairs (0,2), (1,3)
    {
        float a = x[0], b = x[2];
        x[0] = a + b; x[2] = a - b;
        a = x[1]; b = x[3];
        x[1] = a + b; x[3] = a - b;
    }
    // h = 4 .. 64: element j pairs with j ^ h, which lives in lane l ^ (h / 4), same slot
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float other = __shfl_xor_sync(0xffffffffu, x[e], m);
            // lower element: a + b (own + partner); upper element: a - b (partner - own)
            x[e] = upper ? __fsub_rn(other, x[e]) : __fadd_rn(x[e], other);
        }
    }

    // y = bf16(x / sqrt(128)), kept as fp32 for the quantisation
    float y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(x[e], kInvSqrt128)));

    float amax = fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3])));
    amax = warp_max(amax);
    const float scale = __fdiv_rn(fmaxf(amax, 1e-4f), 448.0f);

    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(__fdiv_rn(y[e], scale), __NV_SATFINITE, __NV_E4M3);
        packed |= static_cast<uint32_t>(c) << (8 * e);
    }
    uint8_t* pg = pool + page * kIndexPageBytes;
    reinterpret_cast<uint32_t*>(pg + row * kIndexDim)[lane] = packed;
    if (lane == 0) reinterpret_cast<float*>(pg + kIndexScaleOffset)[row] = scale;
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_store_index_k(const void* k_bf16, const int64_t* slot_mapping, int64_t n,
                                        uint8_t* index_k_pool, int64_t num_pages, int32_t page_size,
                                        int32_t* dev_err, void* stream) {
    if (n < 0 || num_pages < 0) return DSA_ERR_INVALID_ARG;
    if (page_size != dsa::kPage) return DSA_ERR_UNSUPPORTED;
    if (n == 0) return DSA_OK;
    if (!k_bf16 || !slot_mapping || !index_k_pool) return DSA_ERR_INVALID_ARG;
    if (!dsa::aligned16(k_bf16) || !dsa::aligned16(index_k_pool)) return DSA_ERR_INVALID_ARG;
    const int64_t blocks = (n + 7) / 8;
    if (blocks > 0x7fffffffLL) return DSA_ERR_INVALID_ARG;
    dsa::store_index_k_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(k_bf16), slot_mapping, n, index_k_pool, num_pages, dev_err);
    return dsa::launch_status();
}
