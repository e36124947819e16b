// sparse_mla.cu -- absorbed sparse MLA decode over the top-k selected latent rows.
//
// Follows vllm_ascend sfa_v1.py, _execute_sparse_flash_attention_process
// (npu_sparse_flash_attention with query = ql_nope, key = value = latent cache, query_rope /
// key_rope, sparse_indices = top-k, sparse_block_size = 1, block_table) and vllm mla/common.py,
// MLACommonImpl.forward decode branch (absorbed 576-wide query, one shared KV head; _forward_decode
// returns (out, lse); merge_attn_states merges partial results by their log-sum-exp).
//
// Work split: CTA = (row, 16-head group, split of the k selected entries).  Each CTA streams its
// entries' 1152-byte latent rows through shared memory in tiles of 32, keeps an online softmax
// per head, and writes a normalised partial output and its log-sum-exp.  A second kernel merges
// the splits: lse = log sum_j e^{lse_j}, o = sum_j e^{lse_j - lse} o_j.
#include <cuda_bf16.h>

#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr int kHeadGroup = 16;
constexpr int kTile = 32;
constexpr int kSplitEntries = 256;
constexpr int kMlaThreads = 256;
constexpr int kRowStride = kLatentDim + 8;   // padded bf16 row in shared memory
constexpr float kLog2e = 1.4426950408889634f;

struct MlaSmem {
    float q[kHeadGroup][kLatentDim];            // query, pre-multiplied by scale * log2(e)
    uint16_t kv[kTile][kRowStride];             // bf16 latent rows of the tile
    float s[kHeadGroup][kTile];                 // scores (log2 domain), then probabilities
    float alpha[kHeadGroup];
    int64_t grow[kTile];                        // physical latent row, -1 = skip
};

__global__ void __launch_bounds__(kMlaThreads)
sparse_mla_split_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ kv, int64_t num_pages,
                        const int32_t* __restrict__ block_table, int max_pages,
                        const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu_q, int B,
                        const int32_t* __restrict__ idx, int k, int H, float scale, int splits,
                        float* __restrict__ part_o, float* __restrict__ part_lse, int32_t* err) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    MlaSmem& sm = *reinterpret_cast<MlaSmem*>(smem_raw);
    const int split = blockIdx.x;
    const int hg = blockIdx.y;
    const int r = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = row_request(cu_q, B, r);
    const int q0 = __ldg(cu_q + b);
    const int v = visible_len(__ldg(seq_lens + b), __ldg(cu_q + b + 1) - q0, r - q0);
    const float qscale = scale * kLog2e;

    for (int i = threadIdx.x; i < kHeadGroup * kLatentDim; i += kMlaThreads) {
        const int h = i / kLatentDim, d = i % kLatentDim;
        const uint16_t bits = __ldg(q + (static_cast<int64_t>(r) * H + hg * kHeadGroup + h) * kLatentDim + d);
        sm.q[h][d] = __uint_as_float(static_cast<uint32_t>(bits) << 16) * qscale;
    }
    // output accumulators: thread owns dims 2t, 2t+1 for the 16 heads
    float o[kHeadGroup][2];
#pragma unroll
    for (int h = 0; h < kHeadGroup; ++h) o[h][0] = o[h][1] = 0.0f;
    float m_run = -INFINITY, l_run = 0.0f;   // per head, owned by lane h of warp (h / 2)... see below

    const int e_begin = split * kSplitEntries;
    const int e_end = min(k, e_begin + kSplitEntries);
    for (int t0 = e_begin; t0 < e_end; t0 += kTile) {
        __syncthreads();
        if (threadIdx.x < kTile) {
            const int e = t0 + threadIdx.x;
            int64_t g = -1;
            if (e < e_end) {
                const int pos = __ldg(idx + static_cast<int64_t>(r) * k + e);
                if (pos >= 0) {
                    if (pos >= v || (pos >> 6) >= max_pages) {
                        raise_error(err, DSA_DEVERR_INDEX_RANGE);
                    } else {
                        const int32_t page = __ldg(block_table + static_cast<int64_t>(b) * max_pages + (pos >> 6));
                        if (page < 0 || page >= num_pages) raise_error(err, DSA_DEVERR_PAGE_RANGE);
                        else g = static_cast<int64_t>(page) * kPage + (pos & 63);
                    }
                }
            }
            sm.grow[threadIdx.x] = g;
        }
        __syncthreads();
        // gather the tile: 72 x 16-byte chunks per row
        for (int i = threadIdx.x; i < kTile * (kLatentDim / 8); i += kMlaThreads) {
            const int row = i / (kLatentDim / 8), c = i % (kLatentDim / 8);
            const int64_t g = sm.grow[row];
            uint4 val = make_uint4(0, 0, 0, 0);
            if (g >= 0) val = __ldg(reinterpret_cast<const uint4*>(kv + g * kLatentDim) + c);
            *reinterpret_cast<uint4*>(&sm.kv[row][c * 8]) = val;
        }
        __syncthreads();
        // scores: thread -> (key = t & 31, heads (t >> 5) and (t >> 5) + 8)
        {
            const int key = threadIdx.x & (kTile - 1);
            const int h0 = threadIdx.x >> 5;
            float a0 = 0.0f, a1 = 0.0f;
            const uint32_t* krow = reinterpret_cast<const uint32_t*>(sm.kv[key]);
#pragma unroll 4
            for (int d2 = 0; d2 < kLatentDim / 2; ++d2) {
                const uint32_t p = krow[d2];
                const float k0 = bf16_lo(p), k1 = bf16_hi(p);
                a0 = fmaf(sm.q[h0][2 * d2], k0, a0);
                a0 = fmaf(sm.q[h0][2 * d2 + 1], k1, a0);
                a1 = fmaf(sm.q[h0 + 8][2 * d2], k0, a1);
                a1 = fmaf(sm.q[h0 + 8][2 * d2 + 1], k1, a1);
            }
            const bool ok = sm.grow[key] >= 0;
            sm.s[h0][key] = ok ? a0 : -INFINITY;
            sm.s[h0 + 8][key] = ok ? a1 : -INFINITY;
        }
        __syncthreads();
        // online softmax: warp w handles heads w and w + 8, lane = key
        for (int hh = 0; hh < 2; ++hh) {
            const int h = warp + 8 * hh;
            const float sv = sm.s[h][lane];
            const float tmax = warp_max(sv);
            // every lane of the warp tracks the running stats of head h redundantly
            float m_old = __shfl_sync(0xffffffffu, m_run, hh);
            float l_old = __shfl_sync(0xffffffffu, l_run, hh);
            const float m_new = fmaxf(m_old, tmax);
            const float p = (m_new == -INFINITY) ? 0.0f : exp2f(sv - m_new);
            const float alpha = (m_old == -INFINITY) ? 0.0f : exp2f(m_old - m_new);
            const float psum = warp_sum(p);
            sm.s[h][lane] = p;
            if (lane == 0) sm.alpha[h] = (m_new == -INFINITY) ? 1.0f : alpha;
            const float l_new = l_old * alpha + psum;
            if (lane == hh) { m_run = m_new; l_run = l_new; }
        }
        __syncthreads();
        // O update: thread owns dims 2t, 2t+1
        {
#pragma unroll
            for (int h = 0; h < kHeadGroup; ++h) {
                const float a = sm.alpha[h];
                o[h][0] *= a;
                o[h][1] *= a;
            }
            for (int key = 0; key < kTile; ++key) {
                const uint32_t p2 = reinterpret_cast<const uint32_t*>(sm.kv[key])[threadIdx.x];
                const float v0 = bf16_lo(p2), v1 = bf16_hi(p2);
#pragma unroll
                for (int h = 0; h < kHeadGroup; ++h) {
                    const float p = sm.s[h][key];
                    o[h][0] = fmaf(p, v0, o[h][0]);
                    o[h][1] = fmaf(p, v1, o[h][1]);
                }
            }
        }
    }
    // publish per-head stats: lane hh of warp w holds head w + 8*hh
    __syncthreads();
    if (lane < 2) {
        const int h = warp + 8 * lane;
        sm.alpha[h] = l_run;            // reuse: l
        sm.s[h][0] = m_run;             // reuse: m (log2 domain)
    }
    __syncthreads();
    const int64_t base = (static_cast<int64_t>(r) * H + hg * kHeadGroup) * splits + split;
#pragma unroll
    for (int h = 0; h < kHeadGroup; ++h) {
        const float l = sm.alpha[h];
        const float inv = l > 0.0f ? 1.0f / l : 0.0f;
        float2 w2 = make_float2(o[h][0] * inv, o[h][1] * inv);
        reinterpret_cast<float2*>(part_o + (base + static_cast<int64_t>(h) * splits) * kValueDim)[threadIdx.x] = w2;
    }
    if (threadIdx.x < kHeadGroup) {
        const int h = threadIdx.x;
        const float l = sm.alpha[h], m = sm.s[h][0];
        // natural-log lse of the scaled scores: (m + log2 l) / log2(e)
        part_lse[base + static_cast<int64_t>(h) * splits] = (l > 0.0f) ? (m + log2f(l)) / kLog2e : -INFINITY;
    }
}

__global__ void __launch_bounds__(128)
sparse_mla_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse, int splits,
                          uint16_t* __restrict__ out, float* __restrict__ lse) {
    const int64_t rh = blockIdx.x;   // row * H + head
    const float* pl = part_lse + rh * splits;
    float m = -INFINITY;
    for (int j = 0; j < splits; ++j) m = fmaxf(m, __ldg(pl + j));
    float wsum = 0.0f;
    for (int j = 0; j < splits; ++j) {
        const float lj = __ldg(pl + j);
        wsum += (lj == -INFINITY) ? 0.0f : expf(lj - m);
    }
    for (int d = threadIdx.x * 4; d < kValueDim; d += 128 * 4) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m != -INFINITY) {
            for (int j = 0; j < splits; ++j) {
                const float lj = __ldg(pl + j);
                if (lj == -INFINITY) continue;
                const float wj = expf(lj - m) / wsum;
                const float4 oj = __ldg(reinterpret_cast<const float4*>(part_o + (rh * splits + j) * kValueDim + d));
                acc.x = fmaf(wj, oj.x, acc.x);
                acc.y = fmaf(wj, oj.y, acc.y);
                acc.z = fmaf(wj, oj.z, acc.z);
                acc.w = fmaf(wj, oj.w, acc.w);
            }
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 packed;
        packed.x = *reinterpret_cast<const uint32_t*>(&lo);
        packed.y = *reinterpret_cast<const uint32_t*>(&hi);
        reinterpret_cast<uint2*>(out + rh * kValueDim + d)[0] = packed;
    }
    if (lse != nullptr && threadIdx.x == 0) lse[rh] = (m == -INFINITY) ? -INFINITY : m + logf(wsum);
}

int mla_splits(int k) { return (k + kSplitEntries - 1) / kSplitEntries; }

}  // namespace
}  // namespace dsa

extern "C" size_t dsa_sparse_mla_workspace_size(int32_t T, int32_t H, int32_t k) {
    if (T <= 0 || H <= 0 || k <= 0) return 0;
    const size_t splits = static_cast<size_t>(dsa::mla_splits(k));
    return static_cast<size_t>(T) * H * splits * (dsa::kValueDim + 1) * sizeof(float);
}

extern "C" dsa_status dsa_sparse_mla_decode(const void* q_bf16, const void* kv_pool, int64_t num_pages,
                                            const int32_t* block_table, int32_t max_pages,
                                            const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                                            const int32_t* idx, int32_t k, int32_t T, int32_t H, float scale,
                                            void* out_bf16, float* lse, void* workspace,
                                            size_t workspace_bytes, int32_t* dev_err, void* stream) {
    using namespace dsa;
    if (k < 1 || k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
    if (H != 16 && H != 32 && H != 64 && H != 128) return DSA_ERR_UNSUPPORTED;
    if (T < 0 || B < 0 || max_pages < 0 || num_pages < 0) return DSA_ERR_INVALID_ARG;
    if (T == 0) return DSA_OK;
    if (B == 0 || !q_bf16 || !kv_pool || !block_table || !seq_lens || !cu_q || !idx || !out_bf16 || !workspace)
        return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_bf16) || !aligned16(kv_pool) || !aligned16(out_bf16) || !aligned16(workspace))
        return DSA_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || T > 65535) return DSA_ERR_INVALID_ARG;
    if (workspace_bytes < dsa_sparse_mla_workspace_size(T, H, k)) return DSA_ERR_INVALID_ARG;
    const int splits = mla_splits(k);
    float* part_o = static_cast<float*>(workspace);
    float* part_lse = part_o + static_cast<size_t>(T) * H * splits * kValueDim;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t smem = sizeof(MlaSmem);
    if (cudaFuncSetAttribute(sparse_mla_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return DSA_ERR_CUDA;
    dim3 grid(splits, H / kHeadGroup, T);
    sparse_mla_split_kernel<<<grid, kMlaThreads, smem, s>>>(
        static_cast<const uint16_t*>(q_bf16), static_cast<const uint16_t*>(kv_pool), num_pages, block_table,
        max_pages, seq_lens, cu_q, B, idx, k, H, scale, splits, part_o, part_lse, dev_err);
    if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
    sparse_mla_combine_kernel<<<static_cast<unsigned>(static_cast<int64_t>(T) * H), 128, 0, s>>>(
        part_o, part_lse, splits, static_cast<uint16_t*>(out_bf16), lse);
    return launch_status();
}
