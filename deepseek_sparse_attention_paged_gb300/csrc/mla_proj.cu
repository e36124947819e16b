// mla_proj.cu -- per-head projections around the absorbed sparse MLA (sm_103a): the absorbed
// latent query ql = q_nope W_UK_T and the value up-projection out = o_lat W_UV.
//
// Follows vllm mla/common.py, MLACommonImpl.forward decode branch and _q_proj_and_k_up_proj
// (bmm(q_nope as (N, B, P), W_UK_T (N, P, L)), W_UK_T = W_UK.permute(1, 2, 0)) and _v_up_proj
// (bmm(o_lat as (N, B, L), W_UV (N, L, V))).
//
// Both are, per head n, Y_n[T x M] = X_n[T x K] W_n[K x M] with the weight stored [N][K][M] (M
// contiguous): the absorb has K = 128, M = 512, the up-projection K = 512, M = 128.  The kernel
// forms the transposed product Y_n^T = W_n^T X_n^T on the tensor cores: A = W_n^T, 128 output
// dims per tile, read MN-major straight from the weight layout; B = X_n, a tile of TN rows,
// K-major; D in tensor memory, [128 output dims x TN rows] fp32.  Persistent CTAs walk the
// (head, 128-dim tile, row tile) work items: warp 0 streams 64-wide K chunks of the weight (two
// 64-dim atoms) and of the activation rows by TMA with the 128-byte swizzle through a ring;
// warp 1 issues tcgen05.mma.kind::f16 (bf16 operands, fp32 accumulation) into one of two TMEM
// accumulators; warps 2-5 (one per TMEM lane quadrant) round to bf16 and store while the next
// item accumulates.  At decode sizes the work is bound by the weight read (16.8 MB per
// projection for 128 heads).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dsa_common.cuh"
#include "sm100_ptx.cuh"

namespace dsa {
namespace {

constexpr int kProjThreads = 192;                  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kKChunk = 64;                        // K elements per stage: one 128-byte row
constexpr int kMTile = 128;                        // output dims per tile (the MMA's M)
constexpr int kAtomBytes = 64 * kKChunk * 2;       // 8192: 64 output dims x 64 K rows (MN-major atom)
constexpr int kAChunkBytes = 2 * kAtomBytes;       // 16384
constexpr int kRingBytes = 196608;
constexpr int kMaxStages = 8;

template <int TN>
struct ProjCfg {
    static constexpr int kBChunkBytes = TN * 128;                 // TN rows x 64 K elements
    static constexpr int kStageBytes = kAChunkBytes + kBChunkBytes;
    static constexpr int kStages = kRingBytes / kStageBytes < kMaxStages ? kRingBytes / kStageBytes : kMaxStages;
    static constexpr uint32_t kTmemCols = 2 * TN < 32 ? 32 : 2 * TN;   // two accumulators
    // up to 64 rows: one item's output tile as bf16 in shared memory, written out as 16-byte rows
    static constexpr int kOutBytes = TN <= 64 ? TN * kMTile * 2 : 0;
    static constexpr size_t kSmemBytes = 1024 + size_t(kStages) * kStageBytes + kOutBytes + 256;
    static_assert(kStages >= 2, "ring");
    static_assert(kTmemCols <= 512, "tensor memory");
};

struct ProjBars {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint32_t tmem_slot;
};
static_assert(sizeof(ProjBars) <= 256, "barrier block");

// Shared-memory matrix descriptor (sm_100 format): start, leading / stride byte offsets, layout.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(layout) << 61;
    return d;
}
constexpr uint32_t kSw128 = 2;

__device__ __forceinline__ uint16_t to_bf16_bits(float v) {
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    return *reinterpret_cast<const uint16_t*>(&b);
}

// Work item i -> (head, output-dim tile, row tile); heads vary fastest so that consecutive CTAs
// read different weight tiles.
struct Item {
    int n, mt, tt;
};
__device__ __forceinline__ Item item_of(int i, int heads, int mtiles) {
    Item it;
    it.n = i % heads;
    const int rest = i / heads;
    it.mt = rest % mtiles;
    it.tt = rest / mtiles;
    return it;
}

template <int TN>
__global__ void __launch_bounds__(kProjThreads, 1)
mla_proj_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap, int heads, int K,
                int M, int T, uint16_t* __restrict__ y, int64_t sy_t, int64_t sy_n, int vec, int32_t* err) {
    using C = ProjCfg<TN>;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    unsigned char* base = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint16_t* out_s = reinterpret_cast<uint16_t*>(base + C::kStages * C::kStageBytes);   // [TN][128] bf16
    ProjBars& bar = *reinterpret_cast<ProjBars*>(base + C::kStages * C::kStageBytes + C::kOutBytes);
    const uint32_t ring = ptx::smem_addr(base);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mtiles = M / kMTile;
    const int ttiles = (T + TN - 1) / TN;
    const int items = heads * mtiles * ttiles;
    const int kchunks = K / kKChunk;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(&bar.full[s], 1);
            ptx::mbar_init(&bar.empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&bar.acc_full[a], 1);
            ptx::mbar_init(&bar.acc_empty[a], 4);
        }
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(&bar.tmem_slot, C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = bar.tmem_slot;
    const uint64_t deadline = ptx::wait_deadline();
    bool timed_out = false;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            uint32_t c = 0;   // chunks issued
            for (int i = blockIdx.x; i < items && !timed_out; i += gridDim.x) {
                const Item it = item_of(i, heads, mtiles);
                for (int kc = 0; kc < kchunks; ++kc, ++c) {
                    const int s = static_cast<int>(c % C::kStages);
                    const uint32_t ph = (c / C::kStages) & 1u;
                    if (!ptx::mbar_wait(&bar.empty[s], ph ^ 1u, deadline)) { timed_out = true; break; }
                    ptx::mbar_arrive_expect_tx(&bar.full[s], C::kStageBytes);
                    unsigned char* st = base + s * C::kStageBytes;
                    const int m0 = it.mt * kMTile, k0 = kc * kKChunk;
                    ptx::tma_load_3d(st, &wmap, &bar.full[s], m0, k0, it.n);
                    ptx::tma_load_3d(st + kAtomBytes, &wmap, &bar.full[s], m0 + 64, k0, it.n);
                    ptx::tma_load_3d(st + kAChunkBytes, &xmap, &bar.full[s], k0, it.n, it.tt * TN);
                }
            }
            // copies still in flight land before the CTA may leave (bounded)
            const uint32_t last = c;
            for (uint32_t j = last > static_cast<uint32_t>(C::kStages) ? last - C::kStages : 0; j < last; ++j)
                if (!ptx::mbar_wait(&bar.full[j % C::kStages], (j / C::kStages) & 1u, ptx::wait_deadline(20000000ull)))
                    timed_out = true;
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::instr_desc(1, 1, kMTile, TN) | (1u << 15);   // A MN-major
            uint32_t c = 0;
            int local = 0;
            for (int i = blockIdx.x; i < items && !timed_out; i += gridDim.x, ++local) {
                const int a = local & 1;
                if (!ptx::mbar_wait(&bar.acc_empty[a], ((local >> 1) & 1) ^ 1u, deadline)) { timed_out = true; break; }
                ptx::tc_fence_after_sync();
                const uint32_t d = tmem + static_cast<uint32_t>(a * TN);
                for (int kc = 0; kc < kchunks; ++kc, ++c) {
                    const int s = static_cast<int>(c % C::kStages);
                    if (!ptx::mbar_wait(&bar.full[s], (c / C::kStages) & 1u, deadline)) { timed_out = true; break; }
                    ptx::tc_fence_after_sync();
                    const uint32_t sa = ring + s * C::kStageBytes;
                    const uint32_t sb = sa + kAChunkBytes;
#pragma unroll
                    for (int ks = 0; ks < kKChunk / 16; ++ks) {
                        const uint64_t da = smem_desc(sa + ks * 16 * 128, kAtomBytes, 1024, kSw128);
                        const uint64_t db = smem_desc(sb + ks * 32, 16, 1024, kSw128);
                        ptx::umma_f16(d, da, db, idesc, (kc | ks) != 0 ? 1u : 0u);
                    }
                    ptx::umma_commit(&bar.empty[s]);
                }
                if (timed_out) break;
                ptx::umma_commit(&bar.acc_full[a]);
            }
        }
    } else {
        // ---------------------------------------------------------------- epilogue (warps 2-5)
        const int quad = warp & 3;                              // TMEM lanes 32 quad .. +31
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        int local = 0;
        for (int i = blockIdx.x; i < items; i += gridDim.x, ++local) {
            const Item it = item_of(i, heads, mtiles);
            const int a = local & 1;
            // the same answer for the whole warp (a deadline could fall between its lanes' checks)
            const bool got = __all_sync(0xffffffffu, ptx::mbar_wait(&bar.acc_full[a], (local >> 1) & 1, deadline));
            const int m = it.mt * kMTile + quad * 32 + lane;
            const int t0 = it.tt * TN;
            if (C::kOutBytes > 0 && vec) {
                // the tile through shared memory: thread (dim quad * 32 + lane) writes its column of
                // bf16 values and the accumulator is released; once the four warps have met (and
                // leave together if any wait ran out), 16 threads per row store its 256 bytes as
                // 16-byte pieces
                if (got) {
                    ptx::tc_fence_after_sync();
#pragma unroll 1
                    for (int c0 = 0; c0 < TN; c0 += 32) {
                        uint32_t r[32];
                        ptx::tmem_ld_32x32b_x32(tmem + lane_base + static_cast<uint32_t>(a * TN + c0), r);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            out_s[(c0 + j) * kMTile + quad * 32 + lane] = to_bf16_bits(__uint_as_float(r[j]));
                    }
                    ptx::tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&bar.acc_empty[a]);
                }
                uint32_t any_late;
                asm volatile("{\n\t.reg .pred q, p;\n\tsetp.eq.u32 q, %1, 0;\n\tbar.red.or.pred p, 2, 128, q;\n\t"
                             "selp.u32 %0, 1, 0, p;\n\t}"
                             : "=r"(any_late) : "r"(got ? 1u : 0u) : "memory");
                if (any_late) { timed_out = true; break; }
                const int e = threadIdx.x - 64;   // 0 .. 127
                uint16_t* yrow = y + static_cast<int64_t>(it.n) * sy_n + it.mt * kMTile + (e & 15) * 8;
                for (int rr = e >> 4; rr < TN && t0 + rr < T; rr += 8)
                    *reinterpret_cast<uint4*>(yrow + static_cast<int64_t>(t0 + rr) * sy_t) =
                        *reinterpret_cast<const uint4*>(out_s + rr * kMTile + (e & 15) * 8);
                asm volatile("bar.sync 2, 128;" ::: "memory");   // read before the next item writes it
                continue;
            }
            if (!got) { timed_out = true; break; }
            ptx::tc_fence_after_sync();
            uint16_t* yb = y + static_cast<int64_t>(it.n) * sy_n + m;
#pragma unroll 1
            for (int c0 = 0; c0 < TN; c0 += 32) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(tmem + lane_base + static_cast<uint32_t>(a * TN + c0), r);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int t = t0 + c0 + j;
                    if (t < T) yb[static_cast<int64_t>(t) * sy_t] = to_bf16_bits(__uint_as_float(r[j]));
                }
            }
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bar.acc_empty[a]);
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

// ---------------------------------------------------------------------------------------------
// Row orientation for more than 64 rows: Y_n[128 rows x NT dims] = X_n[128 x K] W_n[K x NT] with
// the rows on the MMA's M.  A = the activation rows (K-major, as stored), B = the weight's NT
// output dims (MN-major, as stored), D = [128 rows x NT dims] fp32 in TMEM.  Each activation tile
// is loaded once per NT output dims, and a thread (= one row) writes NT contiguous bf16 values
// with 16-byte stores.
template <int NT>
struct RowsCfg {
    static constexpr int kAChunkBytes = 128 * 128;               // 128 rows x 64 K elements
    static constexpr int kBChunkBytes = (NT / 64) * kAtomBytes;  // NT / 64 atoms of 64 dims x 64 K rows
    static constexpr int kStageBytes = kAChunkBytes + kBChunkBytes;
    static constexpr int kStages = kRingBytes / kStageBytes < kMaxStages ? kRingBytes / kStageBytes : kMaxStages;
    static constexpr uint32_t kTmemCols = 2 * NT;
    static constexpr size_t kSmemBytes = 1024 + size_t(kStages) * kStageBytes + 256;
    static_assert(kStages >= 2 && kTmemCols <= 512, "budgets");
};

template <int NT>
__global__ void __launch_bounds__(kProjThreads, 1)
mla_proj_rows_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap, int heads,
                     int K, int M, int T, uint16_t* __restrict__ y, int64_t sy_t, int64_t sy_n, int32_t* err) {
    using C = RowsCfg<NT>;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    unsigned char* base = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    ProjBars& bar = *reinterpret_cast<ProjBars*>(base + C::kStages * C::kStageBytes);
    const uint32_t ring = ptx::smem_addr(base);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = M / NT;
    const int ttiles = (T + 127) / 128;
    const int items = heads * ntiles * ttiles;
    const int kchunks = K / kKChunk;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(&bar.full[s], 1);
            ptx::mbar_init(&bar.empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&bar.acc_full[a], 1);
            ptx::mbar_init(&bar.acc_empty[a], 4);
        }
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(&bar.tmem_slot, C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = bar.tmem_slot;
    const uint64_t deadline = ptx::wait_deadline();
    bool timed_out = false;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            uint32_t c = 0;
            for (int i = blockIdx.x; i < items && !timed_out; i += gridDim.x) {
                const Item it = item_of(i, heads, ntiles);   // mt: output-dim tile of NT
                for (int kc = 0; kc < kchunks; ++kc, ++c) {
                    const int s = static_cast<int>(c % C::kStages);
                    const uint32_t ph = (c / C::kStages) & 1u;
                    if (!ptx::mbar_wait(&bar.empty[s], ph ^ 1u, deadline)) { timed_out = true; break; }
                    ptx::mbar_arrive_expect_tx(&bar.full[s], C::kStageBytes);
                    unsigned char* st = base + s * C::kStageBytes;
                    const int k0 = kc * kKChunk;
                    ptx::tma_load_3d(st, &xmap, &bar.full[s], k0, it.n, it.tt * 128);
#pragma unroll
                    for (int j = 0; j < NT / 64; ++j)
                        ptx::tma_load_3d(st + C::kAChunkBytes + j * kAtomBytes, &wmap, &bar.full[s], it.mt * NT + 64 * j,
                                         k0, it.n);
                }
            }
            const uint32_t last = c;
            for (uint32_t j = last > static_cast<uint32_t>(C::kStages) ? last - C::kStages : 0; j < last; ++j)
                if (!ptx::mbar_wait(&bar.full[j % C::kStages], (j / C::kStages) & 1u, ptx::wait_deadline(20000000ull)))
                    timed_out = true;
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::instr_desc(1, 1, 128, NT) | (1u << 16);   // B MN-major
            uint32_t c = 0;
            int local = 0;
            for (int i = blockIdx.x; i < items && !timed_out; i += gridDim.x, ++local) {
                const int a = local & 1;
                if (!ptx::mbar_wait(&bar.acc_empty[a], ((local >> 1) & 1) ^ 1u, deadline)) { timed_out = true; break; }
                ptx::tc_fence_after_sync();
                const uint32_t d = tmem + static_cast<uint32_t>(a * NT);
                for (int kc = 0; kc < kchunks; ++kc, ++c) {
                    const int s = static_cast<int>(c % C::kStages);
                    if (!ptx::mbar_wait(&bar.full[s], (c / C::kStages) & 1u, deadline)) { timed_out = true; break; }
                    ptx::tc_fence_after_sync();
                    const uint32_t sa = ring + s * C::kStageBytes;
                    const uint32_t sb = sa + C::kAChunkBytes;
#pragma unroll
                    for (int ks = 0; ks < kKChunk / 16; ++ks) {
                        const uint64_t da = smem_desc(sa + ks * 32, 16, 1024, kSw128);
                        const uint64_t db = smem_desc(sb + ks * 16 * 128, kAtomBytes, 1024, kSw128);
                        ptx::umma_f16(d, da, db, idesc, (kc | ks) != 0 ? 1u : 0u);
                    }
                    ptx::umma_commit(&bar.empty[s]);
                }
                if (timed_out) break;
                ptx::umma_commit(&bar.acc_full[a]);
            }
        }
    } else {
        // ---------------------------------------------------------------- epilogue (warps 2-5)
        const int quad = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        int local = 0;
        for (int i = blockIdx.x; i < items; i += gridDim.x, ++local) {
            const Item it = item_of(i, heads, ntiles);
            const int a = local & 1;
            if (!ptx::mbar_wait(&bar.acc_full[a], (local >> 1) & 1, deadline)) { timed_out = true; break; }
            ptx::tc_fence_after_sync();
            const int t = it.tt * 128 + quad * 32 + lane;
            uint16_t* yr = y + static_cast<int64_t>(t) * sy_t + static_cast<int64_t>(it.n) * sy_n + it.mt * NT;
#pragma unroll 1
            for (int c0 = 0; c0 < NT; c0 += 32) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(tmem + lane_base + static_cast<uint32_t>(a * NT + c0), r);
                ptx::tmem_wait_ld();
                if (t < T) {
                    uint4* dst = reinterpret_cast<uint4*>(yr + c0);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const uint32_t lo = to_bf16_bits(__uint_as_float(r[8 * q4 + 2 * e]));
                            const uint32_t hi = to_bf16_bits(__uint_as_float(r[8 * q4 + 2 * e + 1]));
                            w[e] = lo | (hi << 16);
                        }
                        dst[q4] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bar.acc_empty[a]);
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
EncodeTiledFn proj_tensor_map_encoder() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<EncodeTiledFn>(fn);
}

// Y[t, n, 0:M] = X[t, n, 0:K] W[n] for every row t < T and head n < heads; W bf16 [heads][K][M].
dsa_status launch_proj(const void* x, int64_t sx_t, int64_t sx_n, const void* w, int K, int M, int T, int heads,
                       void* y, int64_t sy_t, int64_t sy_n, int32_t* dev_err, cudaStream_t stream) {
    if (T < 0 || heads < 0 || sx_t < 0 || sx_n < 0 || sy_t < 0 || sy_n < 0) return DSA_ERR_INVALID_ARG;
    if (T == 0 || heads == 0) return DSA_OK;
    if (!x || !w || !y) return DSA_ERR_INVALID_ARG;
    // TMA: 16-byte aligned bases and 16-byte multiples as strides
    if (!aligned16(x) || !aligned16(w) || (sx_t % 8) != 0 || (sx_n % 8) != 0) return DSA_ERR_INVALID_ARG;
    // distinct output vectors must not overlap
    if ((heads > 1 && sy_n < M) || (T > 1 && sy_t < M) || (heads > 1 && T > 1 && sy_t == sy_n))
        return DSA_ERR_INVALID_ARG;
    auto encode = proj_tensor_map_encoder();
    if (encode == nullptr) return DSA_ERR_CUDA;
    // row orientation (16-byte row stores) from 65 rows on, when the output allows vector stores
    const bool vec = aligned16(y) && (sy_t % 8) == 0 && (sy_n % 8) == 0;   // 16-byte output rows
    const bool rows = T > 64 && vec;
    const int NT = M >= 256 ? 256 : 128;   // output dims per row-orientation item
    const int TN = rows ? 128 : (T <= 64 ? 64 : (T <= 128 ? 128 : 256));
    CUtensorMap wmap, xmap;
    {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K),
                                    static_cast<cuuint64_t>(heads)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(M) * 2, static_cast<cuuint64_t>(K) * M * 2};
        const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kKChunk), 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DSA_ERR_CUDA;
    }
    {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(heads),
                                    static_cast<cuuint64_t>(T)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(sx_n) * 2, static_cast<cuuint64_t>(sx_t) * 2};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(kKChunk), 1, static_cast<cuuint32_t>(TN)};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DSA_ERR_CUDA;
    }
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return DSA_ERR_CUDA;
    const int64_t items = rows ? static_cast<int64_t>(heads) * (M / NT) * ((T + 127) / 128)
                               : static_cast<int64_t>(heads) * (M / kMTile) * ((T + TN - 1) / TN);
    if (items > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
    const int ctas = static_cast<int>(items < sms ? items : sms);
    uint16_t* yb = static_cast<uint16_t*>(y);
    if (rows) {
#define DSA_LAUNCH_ROWS(NTV)                                                                                   \
    do {                                                                                                       \
        const size_t smem = RowsCfg<NTV>::kSmemBytes;                                                          \
        if (cudaFuncSetAttribute(mla_proj_rows_kernel<NTV>, cudaFuncAttributeMaxDynamicSharedMemorySize,       \
                                 static_cast<int>(smem)) != cudaSuccess)                                       \
            return DSA_ERR_CUDA;                                                                               \
        mla_proj_rows_kernel<NTV><<<ctas, kProjThreads, smem, stream>>>(wmap, xmap, heads, K, M, T, yb, sy_t,   \
                                                                        sy_n, dev_err);                        \
    } while (0)
        if (NT == 256) DSA_LAUNCH_ROWS(256);
        else DSA_LAUNCH_ROWS(128);
#undef DSA_LAUNCH_ROWS
        return launch_status();
    }
#define DSA_LAUNCH_PROJ(TNV)                                                                                   \
    do {                                                                                                       \
        const size_t smem = ProjCfg<TNV>::kSmemBytes;                                                          \
        if (cudaFuncSetAttribute(mla_proj_kernel<TNV>, cudaFuncAttributeMaxDynamicSharedMemorySize,            \
                                 static_cast<int>(smem)) != cudaSuccess)                                       \
            return DSA_ERR_CUDA;                                                                               \
        mla_proj_kernel<TNV><<<ctas, kProjThreads, smem, stream>>>(wmap, xmap, heads, K, M, T, yb, sy_t, sy_n, \
                                                                   vec ? 1 : 0, dev_err);                      \
    } while (0)
    if (TN == 64) DSA_LAUNCH_PROJ(64);
    else if (TN == 128) DSA_LAUNCH_PROJ(128);
    else DSA_LAUNCH_PROJ(256);
#undef DSA_LAUNCH_PROJ
    return launch_status();
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_mla_absorb_q(const void* q_nope_bf16, int64_t q_row_stride, int64_t q_head_stride,
                                       const void* w_uk_t_bf16, int32_t T, int32_t H, void* ql_bf16,
                                       int64_t out_row_stride, int64_t out_head_stride, int32_t* dev_err,
                                       void* stream) {
    return dsa::launch_proj(q_nope_bf16, q_row_stride, q_head_stride, w_uk_t_bf16, 128, dsa::kValueDim, T, H, ql_bf16,
                            out_row_stride, out_head_stride, dev_err, static_cast<cudaStream_t>(stream));
}

extern "C" dsa_status dsa_mla_v_up(const void* o_lat_bf16, int64_t o_row_stride, int64_t o_head_stride,
                                   const void* w_uv_bf16, int32_t T, int32_t H, void* out_bf16, int64_t out_row_stride,
                                   int64_t out_head_stride, int32_t* dev_err, void* stream) {
    return dsa::launch_proj(o_lat_bf16, o_row_stride, o_head_stride, w_uv_bf16, dsa::kValueDim, 128, T, H, out_bf16,
                            out_row_stride, out_head_stride, dev_err, static_cast<cudaStream_t>(stream));
}
