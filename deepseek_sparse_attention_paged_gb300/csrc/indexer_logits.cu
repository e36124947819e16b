// indexer_logits.cu -- lightning-indexer logits over the paged FP8 index-K cache.
//
// Follows sglang dsa_indexer.py, Indexer._get_topk_paged (paged MQA logits over block_tables and
// seqlens, kv cache viewed as [pages, 64, 1, 132]) with the head gate of _get_logits_head_gate
// (weights * q_scale) and the per-128 FP8 quantisation of the query in Indexer.forward_cuda:
//     I[r,s] = sum_h w[r,h] * q_scale[r,h] * ReLU(k_scale[s] * sum_d q_code[r,h,d] * k_code[s,d])
// for s < v_r.
//
// This translation unit holds the query prologue (shared by every logits kernel) and the launch
// logic.  One CTA scores one 64-token page of one request against a group of up to 4 query rows.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr float kInvSqrt128 = 0x1.6a09e6p-4f;
constexpr int kRowsPerGroup = 4;
constexpr int kThreads = 256;

// Quantise one 128-wide query head held as 4 values per lane (lane l: dims 4l .. 4l+3), with the
// optional Hadamard rotation first (same butterflies and rounding as the key store).  Returns the
// 4 codes packed little-endian and the fp32 scale.
__device__ __forceinline__ uint32_t quantise_head(float x[4], bool rotate, int lane, float* scale_out) {
    if (rotate) {
        {
            float a = x[0], b = x[1];
            x[0] = a + b; x[1] = a - b;
            a = x[2]; b = x[3];
            x[2] = a + b; x[3] = a - b;
        }
        {
            float a = x[0], b = x[2];
            x[0] = a + b; x[2] = a - b;
            a = x[1]; b = x[3];
            x[1] = a + b; x[3] = a - b;
        }
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float other = __shfl_xor_sync(0xffffffffu, x[e], m);
                x[e] = upper ? __fsub_rn(other, x[e]) : __fadd_rn(x[e], other);
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(x[e], kInvSqrt128)));
    }
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
    amax = warp_max(amax);
    const float scale = __fdiv_rn(fmaxf(amax, 1e-4f), 448.0f);
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(__fdiv_rn(x[e], scale), __NV_SATFINITE, __NV_E4M3);
        packed |= static_cast<uint32_t>(c) << (8 * e);
    }
    *scale_out = scale;
    return packed;
}

__device__ __forceinline__ float e4m3_to_float(uint32_t c) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E4M3);
    return __half2float(__half(h));
}

struct SimtSmem {
    uint32_t qcode[kRowsPerGroup][kIndexHeads][kIndexDim / 4];  // packed FP8 query codes
    float wq[kRowsPerGroup][kIndexHeads];                        // w * q_scale
    float key[kPage][kIndexDim + 1];                             // decoded key codes (padded)
    float kscale[kPage];
};

__global__ void __launch_bounds__(kThreads)
indexer_logits_simt_kernel(const uint16_t* __restrict__ q, const float* __restrict__ w,
                           const uint8_t* __restrict__ pool, int64_t num_pages,
                           const int32_t* __restrict__ block_table, int max_pages,
                           const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu_q,
                           int row_begin, int row_end, float* __restrict__ logits, int64_t ld,
                           bool rotate, int32_t* err) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SimtSmem& sm = *reinterpret_cast<SimtSmem*>(smem_raw);
    const int b = blockIdx.z;
    const int lp = blockIdx.x;
    const int L = __ldg(seq_lens + b);
    const int q0 = __ldg(cu_q + b);
    const int q_len = __ldg(cu_q + b + 1) - q0;
    const int j0 = blockIdx.y * kRowsPerGroup;
    if (j0 >= q_len) return;
    const int nrows = min(kRowsPerGroup, q_len - j0);
    if (q0 + j0 >= row_end || q0 + j0 + nrows <= row_begin) return;
    const int vmax = visible_len(L, q_len, j0 + nrows - 1);
    if (lp * kPage >= vmax) return;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // query prologue: one warp per (row, head)
    for (int p = warp; p < nrows * kIndexHeads; p += kThreads / 32) {
        const int row = p / kIndexHeads, h = p % kIndexHeads;
        const int64_t r = q0 + j0 + row;
        const uint2 raw = __ldg(reinterpret_cast<const uint2*>(q + (r * kIndexHeads + h) * kIndexDim) + lane);
        float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
        float s;
        sm.qcode[row][h][lane] = quantise_head(x, rotate, lane, &s);
        if (lane == 0) sm.wq[row][h] = __ldg(w + r * kIndexHeads + h) * s;
    }
    // key page
    const int32_t page = __ldg(block_table + static_cast<int64_t>(b) * max_pages + lp);
    const bool page_ok = page >= 0 && page < num_pages;
    if (page_ok) {
        const uint8_t* pg = pool + static_cast<int64_t>(page) * kIndexPageBytes;
        for (int i = threadIdx.x; i < kPage * kIndexDim / 4; i += kThreads) {
            const uint32_t c4 = __ldg(reinterpret_cast<const uint32_t*>(pg) + i);
            const int key = i / (kIndexDim / 4), d = (i % (kIndexDim / 4)) * 4;
#pragma unroll
            for (int e = 0; e < 4; ++e) sm.key[key][d + e] = e4m3_to_float((c4 >> (8 * e)) & 0xffu);
        }
        if (threadIdx.x < kPage) sm.kscale[threadIdx.x] = __ldg(reinterpret_cast<const float*>(pg + kIndexScaleOffset) + threadIdx.x);
    } else if (threadIdx.x == 0) {
        raise_error(err, DSA_DEVERR_PAGE_RANGE);
    }
    __syncthreads();
    if (!page_ok) return;

    const int key = threadIdx.x & (kPage - 1);
    const int row = threadIdx.x / kPage;
    if (row >= nrows) return;
    const int64_t r = q0 + j0 + row;
    const int s = lp * kPage + key;
    const int v = visible_len(L, q_len, j0 + row);
    if (s >= v || s >= ld || r < row_begin || r >= row_end) return;
    float acc = 0.0f;
    for (int h = 0; h < kIndexHeads; ++h) {
        float dot = 0.0f;
#pragma unroll 8
        for (int d4 = 0; d4 < kIndexDim / 4; ++d4) {
            const uint32_t c4 = sm.qcode[row][h][d4];
#pragma unroll
            for (int e = 0; e < 4; ++e) dot = fmaf(e4m3_to_float((c4 >> (8 * e)) & 0xffu), sm.key[key][d4 * 4 + e], dot);
        }
        acc = fmaf(sm.wq[row][h], fmaxf(dot * sm.kscale[key], 0.0f), acc);
    }
    logits[(r - row_begin) * ld + s] = acc;
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_indexer_logits(const void* q_bf16, const float* weights, const uint8_t* index_k_pool,
                                         int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                         const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                                         int32_t max_seq_len, int32_t max_q_len, int32_t row_begin,
                                         int32_t row_end, float* logits, int64_t ld, uint32_t flags,
                                         int32_t* dev_err, void* stream) {
    using namespace dsa;
    if (B < 0 || max_seq_len < 0 || max_q_len < 0 || row_begin < 0 || row_end < row_begin || max_pages < 0 ||
        num_pages < 0)
        return DSA_ERR_INVALID_ARG;
    if ((flags & ~DSA_Q_ROTATE) != 0u) return DSA_ERR_INVALID_ARG;
    if (B == 0 || row_end == row_begin || max_seq_len == 0 || max_q_len == 0) return DSA_OK;
    if (!q_bf16 || !weights || !index_k_pool || !block_table || !seq_lens || !cu_q || !logits)
        return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_bf16) || !aligned16(index_k_pool)) return DSA_ERR_INVALID_ARG;
    if (ld < max_seq_len) return DSA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(max_pages) * kPage < max_seq_len) return DSA_ERR_INVALID_ARG;
    const int pages = (max_seq_len + kPage - 1) / kPage;
    const int groups = (max_q_len + kRowsPerGroup - 1) / kRowsPerGroup;
    if (groups > 65535 || B > 65535) return DSA_ERR_UNSUPPORTED;
    const size_t smem = sizeof(SimtSmem);
    if (cudaFuncSetAttribute(indexer_logits_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return DSA_ERR_CUDA;
    dim3 grid(pages, groups, B);
    indexer_logits_simt_kernel<<<grid, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(q_bf16), weights, index_k_pool, num_pages, block_table, max_pages, seq_lens,
        cu_q, row_begin, row_end, logits, ld, (flags & DSA_Q_ROTATE) != 0u, dev_err);
    return launch_status();
}
