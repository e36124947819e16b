// indexer_logits.cu -- lightning-indexer logits over the paged FP8 index-K cache.
//
// Follows sglang dsa_indexer.py, Indexer._get_topk_paged (paged MQA logits over block_tables and
// seqlens, kv cache viewed as [pages, 64, 1, 132]) with the head gate of _get_logits_head_gate
// (weights * q_scale) and the per-128 FP8 quantisation of the query in Indexer.forward_cuda:
//     I[r,s] = sum_h w[r,h] * q_scale[r,h] * ReLU(k_scale[s] * sum_d q_code[r,h,d] * k_code[s,d])
// for s < v_r.
//
// The contraction over the 128 dims is an FP8 tensor-core product (tcgen05, fp32 accumulation in
// tensor memory); the ReLU, head gates and head sum are fused into the epilogue that reads the
// accumulator, so only the final fp32 logit of each (row, key) reaches global memory.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "dsa_common.cuh"
#include "sm100_ptx.cuh"

namespace dsa {
namespace {

constexpr float kInvSqrt128 = 0x1.6a09e6p-4f;

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

// ---------------------------------------------------------------------------------------------
// tcgen05 kernel.  CTA = (request b, group of R query rows, chunk of `chunk_tiles` 128-key tiles).
//
//   D[key, n] = sum_d k_code[key, d] * q_code[n, d]      n = row_in_group * 64 + head
//
// is one M = 128 (keys) x N = 64 R x K = 128 FP8 UMMA per tile (4 instructions of K = 32), the
// key tile (two 64-token pages, 8 KB of codes each) arriving by TMA with the 128-byte swizzle and
// the quantised query tile resident in shared memory in the same layout.  The accumulator sits in
// tensor memory, double-buffered so the epilogue of tile i overlaps the MMA of tile i + 1.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM owner + MMA issuer, warps 2-5 =
// epilogue (warp w reads TMEM lanes 32 (w % 4) .. +31, i.e. one key per thread), which applies
// ReLU, the per-head gate w' = w * q_scale, the sum over heads and the key scale, and writes the
// logit.  All six warps quantise the query tile first.
// ---------------------------------------------------------------------------------------------

constexpr int kTileKeys = 128;
constexpr int kTileCodeBytes = kTileKeys * kIndexDim;  // 16 KB: two pages of codes
constexpr int kUmmaThreads = 192;

template <int R>
struct IdxCfg {
    static constexpr int N = 64 * R;
    static constexpr int kStages = (R == 2) ? 5 : 6;
    static constexpr int kQBytes = N * kIndexDim;
    // accumulator buffers in tensor memory: the MMA runs this many tiles ahead of the epilogue
    // (4 x 64 columns for one row; 2 x N columns for row groups, so that 2 CTAs fit one SM)
    static constexpr int kAcc = (R == 1) ? 4 : 2;
    static constexpr uint32_t kTmemCols = kAcc * N;
    static constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + size_t(kStages) * kTileCodeBytes + kQBytes +
                                         size_t(kStages) * kTileKeys * 4 /*scales*/ + R * 64 * 4 /*w'*/ +
                                         (2 * kStages + 2 * kAcc + 1) * 8 /*barriers*/ + 16 + 2 * kStages;
};

template <int R>
__global__ void __launch_bounds__(kUmmaThreads, (R == 4) ? 1 : 2)
indexer_logits_umma_kernel(const __grid_constant__ CUtensorMap kmap, const uint16_t* __restrict__ q,
                           const float* __restrict__ w, const uint8_t* __restrict__ pool, int64_t num_pages,
                           const int32_t* __restrict__ block_table, int max_pages,
                           const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu_q, int row_begin,
                           int row_end, float* __restrict__ logits, int64_t ld, int rotate, int chunk_tiles,
                           int32_t* err) {
    using C = IdxCfg<R>;
    constexpr int S = C::kStages;
    constexpr int N = C::N;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    unsigned char* base = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    unsigned char* codes = base;                                         // [S][16 KB], 1024-aligned
    unsigned char* qtile = codes + S * kTileCodeBytes;                   // [N][128] swizzled
    float* scales = reinterpret_cast<float*>(qtile + C::kQBytes);        // [S][128]
    float* wq = scales + S * kTileKeys;                                  // [R][64]
    uint64_t* full = reinterpret_cast<uint64_t*>(wq + R * 64);
    uint64_t* empty = full + S;
    constexpr int NA = C::kAcc;
    uint64_t* tfull = empty + S;
    uint64_t* tempty = tfull + NA;
    uint64_t* q_ready = tempty + NA;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_ready + 1);
    uint8_t* page_ok = reinterpret_cast<uint8_t*>(tmem_slot + 4);        // [S][2]

    const int b = blockIdx.z;
    const int L = __ldg(seq_lens + b);
    const int q0 = __ldg(cu_q + b);
    const int q_len = __ldg(cu_q + b + 1) - q0;
    const int j0 = blockIdx.y * R;
    if (j0 >= q_len) return;
    const int nrows = min(R, q_len - j0);
    if (q0 + j0 >= row_end || q0 + j0 + nrows <= row_begin) return;
    const int vmax = visible_len(L, q_len, j0 + nrows - 1);
    const int tiles_total = (vmax + kTileKeys - 1) / kTileKeys;
    const int t_begin = blockIdx.x * chunk_tiles;
    if (t_begin >= tiles_total) return;
    const int ntiles = min(tiles_total, t_begin + chunk_tiles) - t_begin;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1 + 4);   // MMA commit + one arrive per epilogue warp
        }
        for (int a = 0; a < NA; ++a) {
            ptx::mbar_init(&tfull[a], 1);
            ptx::mbar_init(&tempty[a], 4);
        }
        ptx::mbar_init(q_ready, 4);             // one arrive per query-prologue warp
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint64_t deadline = ptx::wait_deadline();
    bool timed_out = false;

    if (warp == 0) {       // ---------------- TMA producer (key tiles start streaming at once)
        // the chunk's block-table entries, one per lane (2 pages per tile, <= 32 entries)
        int32_t my_page = -1;
        if (lane < 2 * ntiles && 2 * t_begin + lane < max_pages)
            my_page = __ldg(block_table + static_cast<int64_t>(b) * max_pages + 2 * t_begin + lane);
        for (int i = 0; i < ntiles; ++i) {
            const int s = i % S;
            const uint32_t ph = (i / S) & 1;
            const int32_t pg0 = __shfl_sync(0xffffffffu, my_page, 2 * i);
            const int32_t pg1 = __shfl_sync(0xffffffffu, my_page, 2 * i + 1);
            if (lane == 0) {
                if (!ptx::mbar_wait(&empty[s], ph ^ 1u, deadline)) { timed_out = true; break; }
                const int t = t_begin + i;
                const bool need1 = t * kTileKeys + kPage < vmax;
                const bool ok0 = pg0 >= 0 && pg0 < num_pages;
                const bool ok1 = need1 && pg1 >= 0 && pg1 < num_pages;
                if (!ok0 || (need1 && !ok1)) raise_error(err, DSA_DEVERR_PAGE_RANGE);
                page_ok[2 * s] = ok0;
                page_ok[2 * s + 1] = ok1;
                const uint32_t bytes = (ok0 ? (kPage * kIndexDim + kPage * 4) : 0) + (ok1 ? (kPage * kIndexDim + kPage * 4) : 0);
                ptx::mbar_arrive_expect_tx(&full[s], bytes);
                unsigned char* dst = codes + s * kTileCodeBytes;
                if (ok0) {
                    ptx::tma_load_3d(dst, &kmap, &full[s], 0, 0, pg0);
                    ptx::bulk_load(scales + s * kTileKeys, pool + static_cast<int64_t>(pg0) * kIndexPageBytes + kIndexScaleOffset,
                                   kPage * 4, &full[s]);
                }
                if (ok1) {
                    ptx::tma_load_3d(dst + kPage * kIndexDim, &kmap, &full[s], 0, 0, pg1);
                    ptx::bulk_load(scales + s * kTileKeys + kPage,
                                   pool + static_cast<int64_t>(pg1) * kIndexPageBytes + kIndexScaleOffset, kPage * 4, &full[s]);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {   // ---------------- MMA issuer
            constexpr uint32_t idesc = ptx::instr_desc(0, 0, kTileKeys, N);
            const uint32_t q_addr = ptx::smem_addr(qtile);
            if (!ptx::mbar_wait(q_ready, 0, deadline)) timed_out = true;
            for (int i = 0; i < ntiles && !timed_out; ++i) {
                const int s = i % S;
                const uint32_t ph = (i / S) & 1;
                const int a = i % NA;
                const uint32_t aph = (i / NA) & 1;
                if (!ptx::mbar_wait(&full[s], ph, deadline)) { timed_out = true; break; }
                if (!ptx::mbar_wait(&tempty[a], aph ^ 1u, deadline)) { timed_out = true; break; }
                ptx::tc_fence_after_sync();
                const uint32_t a_addr = ptx::smem_addr(codes + s * kTileCodeBytes);
                const uint32_t d = tmem + static_cast<uint32_t>(a * N);
#pragma unroll
                for (int k = 0; k < kIndexDim / 32; ++k)
                    ptx::umma_f8f6f4(d, ptx::sw128_kmajor_desc(a_addr + k * 32), ptx::sw128_kmajor_desc(q_addr + k * 32),
                                     idesc, k > 0 ? 1u : 0u);
                ptx::umma_commit(&empty[s]);
                ptx::umma_commit(&tfull[a]);
            }
        }
    } else {               // ---------------- warps 2..5: query prologue, then epilogue
        {
            // quantise the group's (row, head) vectors: warp pw takes vectors p = pw, pw + 4, ...;
            // all loads of a batch are issued before any is used
            const int pw = warp - 2;
            constexpr int kPerWarp = R * kIndexHeads / 4;
            constexpr int kBatch = 16;
            for (int v0 = 0; v0 < kPerWarp; v0 += kBatch) {
                uint2 raw[kBatch];
                float wv[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int p = pw + 4 * (v0 + u);
                    const int jj = p / kIndexHeads, h = p % kIndexHeads;
                    raw[u] = make_uint2(0u, 0u);
                    wv[u] = 0.0f;
                    if (jj < nrows) {
                        const int64_t r = q0 + j0 + jj;
                        raw[u] = __ldg(reinterpret_cast<const uint2*>(q + (r * kIndexHeads + h) * kIndexDim) + lane);
                        wv[u] = __ldg(w + r * kIndexHeads + h);
                    }
                }
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int p = pw + 4 * (v0 + u);   // = row_in_group * 64 + head = B-operand row
                    const int jj = p / kIndexHeads;
                    uint32_t packed = 0;
                    float sq = 0.0f;
                    if (jj < nrows) {
                        float x[4] = {bf16_lo(raw[u].x), bf16_hi(raw[u].x), bf16_lo(raw[u].y), bf16_hi(raw[u].y)};
                        packed = quantise_head(x, rotate != 0, lane, &sq);
                    }
                    const uint32_t off = p * 128 + ((((lane >> 2) ^ (p & 7))) << 4) + ((lane & 3) << 2);
                    *reinterpret_cast<uint32_t*>(qtile + off) = packed;
                    if (lane == 0) wq[p] = wv[u] * sq;
                }
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(q_ready);
        }
        if (!ptx::mbar_wait(q_ready, 0, deadline)) timed_out = true;   // every warp's w' is visible
        const int quad = warp & 3;
        const int key_in_tile = quad * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        for (int i = 0; i < ntiles && !timed_out; ++i) {
            const int s = i % S;
            const uint32_t ph = (i / S) & 1;
            const int a = i % NA;
            const uint32_t aph = (i / NA) & 1;
            if (!ptx::mbar_wait(&full[s], ph, deadline)) { timed_out = true; break; }
            if (!ptx::mbar_wait(&tfull[a], aph, deadline)) { timed_out = true; break; }
            ptx::tc_fence_after_sync();
            const bool ok = page_ok[2 * s + (key_in_tile >> 6)] != 0;
            const float ks = scales[s * kTileKeys + key_in_tile];
            const int key = (t_begin + i) * kTileKeys + key_in_tile;
#pragma unroll 1
            for (int jj = 0; jj < nrows; ++jj) {   // one query row at a time: 64 accumulator columns
                uint32_t r0[32], r1[32];
                const uint32_t col = tmem + lane_base + static_cast<uint32_t>(a * N + jj * kIndexHeads);
                ptx::tmem_ld_32x32b_x32(col, r0);
                ptx::tmem_ld_32x32b_x32(col + 32, r1);
                ptx::tmem_wait_ld();
                const float* g = wq + jj * kIndexHeads;
                float acc = 0.0f;
#pragma unroll
                for (int h = 0; h < 32; ++h) acc = fmaf(g[h], fmaxf(__uint_as_float(r0[h]), 0.0f), acc);
#pragma unroll
                for (int h = 0; h < 32; ++h) acc = fmaf(g[32 + h], fmaxf(__uint_as_float(r1[h]), 0.0f), acc);
                const int r = q0 + j0 + jj;
                const int v = visible_len(L, q_len, j0 + jj);
                if (ok && key < v && key < ld && r >= row_begin && r < row_end)
                    logits[static_cast<int64_t>(r - row_begin) * ld + key] = acc * ks;
            }
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(&tempty[a]);
                ptx::mbar_arrive(&empty[s]);
            }
        }
    }
    if (timed_out) raise_error(err, DSA_DEVERR_TIMEOUT);
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up through the runtime (no link against libcuda).
EncodeTiledFn tensor_map_encoder() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<EncodeTiledFn>(fn);
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
    const int R = max_q_len >= 4 ? 4 : (max_q_len >= 2 ? 2 : 1);
    const int groups = (max_q_len + R - 1) / R;
    if (groups > 65535 || B > 65535) return DSA_ERR_UNSUPPORTED;
    if (num_pages > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
    const int tiles = (max_seq_len + kTileKeys - 1) / kTileKeys;
    const int chunk_tiles = (R == 1) ? 8 : 16;
    const int chunks = (tiles + chunk_tiles - 1) / chunk_tiles;

    // tensor map over the code bytes of the page-blocked pool: (byte in row, row in page, page)
    static_assert(sizeof(CUtensorMap) == 128, "CUtensorMap size");
    CUtensorMap kmap;
    {
        auto encode = tensor_map_encoder();
        if (encode == nullptr) return DSA_ERR_CUDA;
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kIndexDim), static_cast<cuuint64_t>(kPage),
                                    static_cast<cuuint64_t>(num_pages)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kIndexDim), static_cast<cuuint64_t>(kIndexPageBytes)};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(kIndexDim), static_cast<cuuint32_t>(kPage), 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(index_k_pool), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DSA_ERR_CUDA;
    }
    dim3 grid(chunks, groups, B);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int rotate = (flags & DSA_Q_ROTATE) != 0u ? 1 : 0;
    const uint16_t* qp = static_cast<const uint16_t*>(q_bf16);
#define DSA_LAUNCH_IDX(RR)                                                                                      \
    do {                                                                                                        \
        const size_t smem = IdxCfg<RR>::kSmemBytes;                                                             \
        if (cudaFuncSetAttribute(indexer_logits_umma_kernel<RR>, cudaFuncAttributeMaxDynamicSharedMemorySize,    \
                                 static_cast<int>(smem)) != cudaSuccess)                                        \
            return DSA_ERR_CUDA;                                                                                \
        indexer_logits_umma_kernel<RR><<<grid, kUmmaThreads, smem, st>>>(                                       \
            kmap, qp, weights, index_k_pool, num_pages, block_table, max_pages, seq_lens, cu_q, row_begin,      \
            row_end, logits, ld, rotate, chunk_tiles, dev_err);                                                 \
    } while (0)
    if (R == 1) DSA_LAUNCH_IDX(1);
    else if (R == 2) DSA_LAUNCH_IDX(2);
    else DSA_LAUNCH_IDX(4);
#undef DSA_LAUNCH_IDX
    return launch_status();
}
