// indexer_logits.cu -- lightning-indexer logits over the paged FP8 index-K cache.
//
// Follows sglang dsa_indexer.py, Indexer._get_topk_paged (paged MQA logits over block_tables and
// seqlens, kv cache viewed as [pages, 64, 1, 132]) with the head gate of _get_logits_head_gate
// (weights * q_scale) and the per-128 FP8 quantisation of the query in Indexer.forward_cuda:
//     I[r,s] = sum_h w[r,h] * q_scale[r,h] * ReLU(k_scale[s] * sum_d q_code[r,h,d] * k_code[s,d])
// for s < v_r.
//
// Two kernels.  The query prologue quantises every (row, head) vector exactly once into the
// caller's workspace, already in the shared-memory layout the tensor cores read.  The logits
// kernel is persistent: one CTA per SM takes an equal share of all 128-key tiles of all requests
// (tiles of one (request, row group) are consecutive), streams the key pages through a deep TMA
// ring, multiplies them with the resident query tile on the FP8 tensor cores (tcgen05, fp32
// accumulation in tensor memory) and reduces ReLU, head gates and head sum in the epilogue that
// reads the accumulator, so only the final fp32 logit of each (row, key) reaches global memory.
// The logits kernel is launched as a programmatic dependent of the prologue, so its setup and its
// first key pages overlap the prologue; only the query-tile loads wait for it.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "dsa_common.cuh"
#include "sm100_ptx.cuh"

namespace dsa {
namespace {

constexpr float kInvSqrt128 = 0x1.6a09e6p-4f;

// Quantise one 128-wide query head held as 4 values per lane (lane l: dims 4l .. 4l+3), with the
// optional Hadamard rotation first (same butterflies and rounding as the key store).  Returns the
// 4 codes packed little-endian and the fp32 scale.
// Scale format "ue8m0": the smallest power of two not below the fp32 scale s (s positive, normal).
__device__ __forceinline__ float pow2_at_least(float s) {
    const uint32_t u = __float_as_uint(s);
    return (u & 0x007fffffu) ? __uint_as_float((u & 0x7f800000u) + 0x00800000u) : s;
}

__device__ __forceinline__ uint32_t quantise_head(float x[4], bool rotate, bool ue8m0, int lane, float* scale_out) {
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
    float scale = __fdiv_rn(fmaxf(amax, 1e-4f), 448.0f);
    if (ue8m0) scale = pow2_at_least(scale);
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(__fdiv_rn(x[e], scale), __NV_SATFINITE, __NV_E4M3);
        packed |= static_cast<uint32_t>(c) << (8 * e);
    }
    *scale_out = scale;
    return packed;
}

// Per-row histogram of the top 12 bits of each logit's order key (HIST variant, for the fused
// indexer + top-k): the key maps larger floats to larger unsigned values, -0 and +0 to one key and
// NaN to the smallest key -- the mapping the top-k kernels select on.
constexpr int kTopBins = 4096;
__device__ __forceinline__ uint32_t logit_order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kTileKeys = 128;
constexpr int kTileCodeBytes = kTileKeys * kIndexDim;    // 16 KB: two pages of codes
constexpr int kQRowBytes = kIndexHeads * kIndexDim;       // 8 KB of codes per query row
constexpr int kQGateBytes = kIndexHeads * 4;              // 64 fp32 gates w' per query row
constexpr int kThreads = 352;                             // 11 warps
constexpr int kEpiWarp0 = 2;                              // warps 2..9: two epilogue warpgroups
constexpr int kLoaderWarp = 10;
constexpr int kWidenWarp0 = 11;                           // c8: warps 11..14 widen int8 key tiles to f16
constexpr int kProducer1Warp = 11;                        // two pipelines: key producer of pipeline 1
constexpr int kMma1Warp = 12;                             // two pipelines: MMA issuer of pipeline 1
constexpr int kQRowBytesC8 = kIndexHeads * kIndexDim * 2; // c8: 16 KB of f16 query codes per row
constexpr int kWTileBytes = kTileKeys * kIndexDim * 2;    // c8: 32 KB, one key tile widened to f16

// acc2 += gates2 * (ReLU(x0), ReLU(x1)) on two fp32 lanes at once (packed FMA, round to nearest)
__device__ __forceinline__ void fma2_relu(uint64_t& acc2, uint64_t gates2, uint32_t x0, uint32_t x1) {
    uint64_t x2;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x2) : "f"(fmaxf(__uint_as_float(x0), 0.0f)), "f"(fmaxf(__uint_as_float(x1), 0.0f)));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2) : "l"(gates2), "l"(x2));
}

// Bring the 128-byte line holding p into L2 (no register result, no memory change).
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// ---------------------------------------------------------------------------------------------
// Query prologue: one warp per (row, head) vector.  Writes the 128 codes of the vector into the
// row's 8 KB block of the workspace at the position the 128-byte swizzle gives B-operand row
// `head` (16-byte chunk c of row h lands at chunk c ^ (h & 7)), and w' = w * q_scale.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
indexer_q_prologue_kernel(const uint16_t* __restrict__ q, const float* __restrict__ w,
                          const int32_t* __restrict__ cu_q, int B, int row_begin, int row_end, int mode,
                          uint8_t* __restrict__ q_codes, float* __restrict__ q_gates, uint32_t* __restrict__ hist_zero,
                          const int32_t* __restrict__ seq_lens) {
    // Before anything else, L2 prefetches of what every CTA of the logits kernel reads in its setup:
    // the row offsets and the lengths.  A prefetch changes no memory and fills only L2, where any
    // later write of the previous kernel lands as well, so it may overlap that kernel.
    {
        const int64_t gt = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
        if (gt < (B + 32) / 32) prefetch_l2(cu_q + gt * 32);
        if (gt < (B + 31) / 32) prefetch_l2(seq_lens + gt * 32);
    }
    // launched as a programmatic dependent of the previous kernel on the stream: its CTAs are
    // resident early and start once that kernel has completed (nothing else is read or written
    // before).  Only then may the logits kernel be scheduled: it reads key pages before its own
    // wait, and the previous kernel may be the store writing them.
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    // the rows' top-12-bit histograms (one-call indexer) start at zero: block b clears words
    // 512 b .. 512 b + 511 (8 blocks per row, 4096 words per row).  The logits kernel adds into them
    // only after its query loads, which wait for this whole grid.
    if (hist_zero != nullptr) {
        hist_zero[blockIdx.x * 512 + threadIdx.x] = 0u;
        hist_zero[blockIdx.x * 512 + 256 + threadIdx.x] = 0u;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t v = static_cast<int64_t>(blockIdx.x) * 8 + warp;   // (row - row_begin) * 64 + head
    if (v >= static_cast<int64_t>(row_end - row_begin) * kIndexHeads) return;
    const int64_t r = row_begin + v / kIndexHeads;
    const int h = static_cast<int>(v % kIndexHeads);
    if (r >= __ldg(cu_q + B)) return;
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(q + (r * kIndexHeads + h) * kIndexDim) + lane);
    float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
    float scale;
    const uint32_t packed = quantise_head(x, (mode & 1) != 0, (mode & 2) != 0, lane, &scale);
    uint8_t* dst = q_codes + (v / kIndexHeads) * kQRowBytes;
    const uint32_t off = h * 128 + (((lane >> 2) ^ (h & 7)) << 4) + ((lane & 3) << 2);
    *reinterpret_cast<uint32_t*>(dst + off) = packed;
    if (lane == 0) q_gates[v] = __ldg(w + r * kIndexHeads + h) * scale;
}

// Query prologue of the int8 cache: one warp per (row, head) vector, rotated with the bf16 Hadamard
// / sqrt(128) and quantised to int8 with one scale (c8_rotate_quant), the codes written as f16
// (exact) into the row's 16 KB block: dim chunk c (dims 64 c ..) of head h at c * 8 KB + h * 128
// with the 128-byte swizzle; the gate w16 * q_scale16 (the weight and the scale rounded to fp16, as
// the c8 path casts weights and scales; their product is exact in fp32).
__global__ void __launch_bounds__(256)
indexer_q_prologue_c8_kernel(const uint16_t* __restrict__ q, const float* __restrict__ w,
                             const int32_t* __restrict__ cu_q, int B, int row_begin, int row_end,
                             uint8_t* __restrict__ q_codes, float* __restrict__ q_gates) {
    ptx::griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t v = static_cast<int64_t>(blockIdx.x) * 8 + warp;   // (row - row_begin) * 64 + head
    if (v >= static_cast<int64_t>(row_end - row_begin) * kIndexHeads) return;
    const int64_t r = row_begin + v / kIndexHeads;
    const int h = static_cast<int>(v % kIndexHeads);
    if (r >= __ldg(cu_q + B)) return;
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(q + (r * kIndexHeads + h) * kIndexDim) + lane);
    const float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
    float scale;
    const uint32_t packed = c8_rotate_quant(x, lane, &scale);
    uint32_t lo, hi;
    i8x4_to_f16x4(packed, lo, hi);
    // dims 4 lane .. + 3 = f16 bytes 8 lane .. + 7: chunk lane / 16, 16-byte piece (lane % 16) / 2
    uint8_t* dst = q_codes + (v / kIndexHeads) * kQRowBytesC8 + (lane >> 4) * 8192 + h * 128 +
                   ((((lane & 15) >> 1) ^ (h & 7)) << 4) + (lane & 1) * 8;
    *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
    if (lane == 0)
        q_gates[v] = __half2float(__float2half_rn(__ldg(w + r * kIndexHeads + h))) * __half2float(__float2half_rn(scale));
}

// ---------------------------------------------------------------------------------------------
// Work decomposition.  A segment is one (request b, group g of R consecutive query rows); its
// tiles are the 128-key tiles [0, ceil(vmax / 128)) of the group's longest visible prefix.  The
// segments are numbered b * G + g (G = groups of the longest request) and their tiles
// concatenated; CTA c of the grid takes the tiles [T c / grid, T (c+1) / grid).
// ---------------------------------------------------------------------------------------------
struct Seg {
    int sidx;     // b * G + g
    int b, L, q0, q_len, j0, nrows, vmax;
    int ntiles;   // tiles of the whole segment
    int tile;     // current tile within the segment
};

constexpr int kSegTab = 8;   // segments of a CTA's share kept in shared memory

struct SegArgs {
    const int32_t* seq_lens;
    const int32_t* cu_q;
    int B, G, R, row_begin, row_end;
    int shift;   // compressed keys: visible entries = visible tokens >> shift
    // the first segments of this CTA's share (tab_base .. tab_base + tab_n - 1), read from shared
    // memory instead of global memory during the stream
    const Seg* tab;
    int tab_base, tab_n;
};

__device__ __forceinline__ int seg_load(const SegArgs& a, int sidx, Seg& s) {
    if (a.tab != nullptr && sidx >= a.tab_base && sidx < a.tab_base + a.tab_n) {
        s = a.tab[sidx - a.tab_base];
        return s.ntiles;
    }
    s.sidx = sidx;
    s.ntiles = 0;
    const int b = sidx / a.G;
    const int g = sidx - b * a.G;
    if (b >= a.B) return 0;
    const int q0 = __ldg(a.cu_q + b);
    const int q_len = __ldg(a.cu_q + b + 1) - q0;
    const int j0 = g * a.R;
    if (j0 >= q_len) return 0;
    const int nrows = min(a.R, q_len - j0);
    if (q0 + j0 >= a.row_end || q0 + j0 + nrows <= a.row_begin) return 0;
    const int L = __ldg(a.seq_lens + b);
    s.b = b; s.L = L; s.q0 = q0; s.q_len = q_len; s.j0 = j0; s.nrows = nrows;
    s.vmax = visible_len(L, q_len, j0 + nrows - 1) >> a.shift;
    s.ntiles = (s.vmax + kTileKeys - 1) / kTileKeys;
    return s.ntiles;
}

// Move to the first tile of the next segment that has tiles (the caller knows one exists).
__device__ __forceinline__ void seg_next(const SegArgs& a, Seg& s) {
    int sidx = s.sidx;
    while (seg_load(a, ++sidx, s) == 0 && sidx < a.B * a.G) {
    }
    s.tile = 0;
}

// Block-wide (warps kEpiWarp0 .. kEpiWarp0 + 7, named barrier 1) inclusive scan of one int64 per
// thread; `scratch` holds 8 partials.  Returns this thread's inclusive prefix and the total.
__device__ __forceinline__ int64_t epi_scan(int64_t v, int64_t* scratch, int64_t* total) {
    const int t = threadIdx.x - kEpiWarp0 * 32;
    const int lane = t & 31, w = t >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int64_t o = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += o;
    }
    if (lane == 31) scratch[w] = v;
    asm volatile("bar.sync 1, 256;" ::: "memory");
    int64_t before = 0, all = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t x = scratch[i];
        if (i < w) before += x;
        all += x;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    *total = all;
    return before + v;
}

// ---------------------------------------------------------------------------------------------
// Logits kernel.  Per tile, with n = row_in_group * 64 + head:
//     D[key, n] = sum_d k_code[key, d] * q_code[n, d]
// is one M = 128 (keys) x N = 64 R x K = 128 FP8 UMMA (4 instructions of K = 32), the key tile
// (two 64-token pages, 8 KB of codes each) arriving by TMA with the 128-byte swizzle and the query
// tile of the segment (R rows x 8 KB, double-buffered across segments) by bulk copy from the
// prologue's workspace.
//
// Warp roles (352 threads): warp 0 = key producer, warp 1 = TMEM owner + MMA issuer, warps 2-9 =
// two epilogue warpgroups taking alternate tiles (warp w reads TMEM lanes 32 (w % 4) .. +31, one
// key per thread: ReLU, gates w', head sum, key scale, store), warp 10 = query-tile loader.  With
// two pipelines (416 threads) the alternate tiles form two independent streams: warps 0 / 1 /
// epilogue group 0 handle the even tiles with stage ring 0 and accumulators 0-1, warps 11 / 12 /
// epilogue group 1 the odd tiles with ring 1 and accumulators 2-3.
// ---------------------------------------------------------------------------------------------
template <int R, bool HIST = false, bool C8 = false>
struct IdxCfg {
    static_assert(!HIST || R <= 2, "the per-row histograms fit shared memory for row groups of up to 2 rows");
    static_assert(!C8 || (R <= 2 && !HIST), "the int8 cache: row groups of up to 2 rows, no histograms");
    static constexpr int N = 64 * R;
    // Independent pipelines per CTA: pipeline p takes the CTA's tiles i with i % kPipes == p and has
    // its own key producer, stage ring, MMA issuer, accumulators and epilogue warpgroup, so a key
    // page that is late stalls only its own pipeline (one in-order ring streams random pages ~12 %
    // slower: every stage behind a late page waits for it).
    static constexpr int kPipes = (C8 || R == 4) ? 1 : 2;
    static constexpr int kThreadsCfg = C8 ? kThreads + 4 * 32 : (kPipes == 2 ? kThreads + 2 * 32 : kThreads);
    // with HIST, the R 16 KB histograms take the place of R (or, for R = 2, two) key stages; with C8
    // the two 32 KB f16 key tiles and the f16 query take the place of key stages
    static constexpr int kStages =
        C8 ? (R == 1 ? 7 : 5) : ((R == 1) ? (HIST ? 10 : 12) : (R == 2 ? (HIST ? 8 : 10) : 9));
    static_assert(kStages % kPipes == 0, "equal rings");
    static constexpr int kStagesPipe = kStages / kPipes;
    static constexpr int kAcc = (R == 4) ? 2 : 4;                 // accumulators of N columns
    static constexpr int kAccPipe = kAcc / kPipes;
    static constexpr uint32_t kTmemCols = kAcc * N;               // 256 / 512 / 512
    static constexpr int kQRowB = C8 ? kQRowBytesC8 : kQRowBytes;
    static constexpr int kQBytes = R * kQRowB;
    static constexpr int kScaleElem = C8 ? 2 : 4;                 // fp16 / fp32 key scales
    static constexpr int kPoolPageBytes = C8 ? kC8PageBytes : kIndexPageBytes;
    static constexpr int kPoolScaleOff = C8 ? kC8ScaleOffset : kIndexScaleOffset;
    static constexpr size_t kCodesOff = 0;
    static constexpr size_t kQOff = kCodesOff + size_t(kStages) * kTileCodeBytes;
    static constexpr size_t kWOff = kQOff + 2 * size_t(kQBytes);
    static constexpr size_t kScalesOff = kWOff + (C8 ? 2 * size_t(kWTileBytes) : 0);
    static constexpr size_t kGatesOff = kScalesOff + size_t(kStages) * kTileKeys * kScaleElem;
    static constexpr size_t kBarOff = kGatesOff + 2 * size_t(R) * kQGateBytes;
    // full / empty per stage, tfull / tempty per accumulator, qfull / qempty, the epilogue warps'
    // histogram barrier, and with C8 wfull / wempty per f16 tile
    static constexpr int kBars = 2 * kStages + 2 * kAcc + 4 + 1 + (C8 ? 4 : 0);
    static constexpr size_t kMiscOff = kBarOff + size_t(kBars) * 8;   // tmem slot, partition, scan
    static constexpr size_t kSegTabOff = kMiscOff + 16 + 8 * 8;   // [kSegTab] Seg + the count
    static constexpr size_t kPageOkOff = kSegTabOff + kSegTab * sizeof(Seg) + 16;
    static constexpr size_t kHistOff = (kPageOkOff + 2 * kStages + 15) / 16 * 16;
    static constexpr size_t kHistBytes = HIST ? size_t(R) * kTopBins * 4 : 0;
    static constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + kHistOff + kHistBytes;
    static_assert(kSmemBytes <= 232448, "shared-memory budget");
};

template <int R, bool HIST, bool C8>
__global__ void __launch_bounds__(IdxCfg<R, HIST, C8>::kThreadsCfg, 1)
indexer_logits_umma_kernel(const __grid_constant__ CUtensorMap kmap, const uint8_t* __restrict__ q_codes,
                           const float* __restrict__ q_gates, const uint8_t* __restrict__ pool, int64_t num_pages,
                           const int32_t* __restrict__ block_table, int max_pages,
                           const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu_q, int B, int G,
                           int row_begin, int row_end, float* __restrict__ logits, int64_t ld, int32_t* err,
                           uint32_t* __restrict__ hist_g, int cmp_shift) {
    using C = IdxCfg<R, HIST, C8>;
    constexpr int S = C::kStages;
    constexpr int N = C::N;
    constexpr int NA = C::kAcc;
    constexpr int P = C::kPipes;
    constexpr int SP = C::kStagesPipe;
    constexpr int NAP = C::kAccPipe;
    // tile i of this CTA: pipeline i % P, stage and accumulator of that pipeline's ring, and the
    // parities of their barriers on this use
    auto stage_of = [](int i) { return (i % P) * SP + (i / P) % SP; };
    auto stage_ph = [](int i) { return static_cast<uint32_t>((i / P) / SP) & 1u; };
    auto acc_of = [](int i) { return (i % P) * NAP + (i / P) % NAP; };
    auto acc_ph = [](int i) { return static_cast<uint32_t>((i / P) / NAP) & 1u; };
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    unsigned char* base = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    unsigned char* codes = base + C::kCodesOff;                               // [S][16 KB]
    unsigned char* qtile = base + C::kQOff;                                   // [2][R * 8 KB] (C8: 16 KB)
    unsigned char* wtile = base + C::kWOff;                                   // C8: [2][32 KB] f16 key tiles
    unsigned char* scales_b = base + C::kScalesOff;                           // [S][128] fp32 (C8: fp16)
    float* scales = reinterpret_cast<float*>(scales_b);
    float* gates = reinterpret_cast<float*>(base + C::kGatesOff);             // [2][R * 64]
    uint64_t* full = reinterpret_cast<uint64_t*>(base + C::kBarOff);
    uint64_t* empty = full + S;
    uint64_t* tfull = empty + S;
    uint64_t* tempty = tfull + NA;
    uint64_t* qfull = tempty + NA;     // [2]
    uint64_t* qempty = qfull + 2;      // [2]
    uint64_t* hsync = qempty + 2;      // HIST: the 8 epilogue warps meet before / after a histogram flush
    uint64_t* wfull = hsync + 1;       // C8: [2] an f16 key tile is written (4 widen warps)
    uint64_t* wempty = wfull + 2;      // C8: [2] the MMAs that read it completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + C::kMiscOff);
    int32_t* part = reinterpret_cast<int32_t*>(base + C::kMiscOff + 4);      // start segment, tile, count
    int64_t* scan_scratch = reinterpret_cast<int64_t*>(base + C::kMiscOff + 16);
    Seg* segtab = reinterpret_cast<Seg*>(base + C::kSegTabOff);
    int32_t* segtab_n = reinterpret_cast<int32_t*>(base + C::kSegTabOff + kSegTab * sizeof(Seg));
    uint8_t* page_ok = base + C::kPageOkOff;                                  // [S][2]
    uint32_t* hist_s = reinterpret_cast<uint32_t*>(base + C::kHistOff);       // HIST: [R][4096]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const SegArgs sa{seq_lens, cu_q, B, G, R, row_begin, row_end, cmp_shift, nullptr, 0, 0};
    ptx::griddep_launch_dependents();   // the top-k kernel may be scheduled; it waits for this grid
    if (warp == kLoaderWarp) {
        // while the other warps set up: L2 prefetch of this CTA's slice of the block table (of its
        // first 8 MB), which the producers read right after the setup
        const int64_t bytes = static_cast<int64_t>(B) * max_pages * 4;
        const int64_t lines = (bytes < (int64_t(8) << 20) ? bytes : (int64_t(8) << 20)) / 128;
        const int64_t l1 = lines * (blockIdx.x + 1) / gridDim.x;
        for (int64_t l = lines * blockIdx.x / gridDim.x + lane; l < l1; l += 32) prefetch_l2(block_table + l * 32);
    }
    const int nseg = B * G;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(&full[s], 1);
            // the stage's readers: the MMA commit (C8: the 4 widen warps) + the 4 warps of the tile's
            // epilogue group (scales, page flags)
            ptx::mbar_init(&empty[s], (C8 ? 4 : 1) + 4);
        }
        if (C8) {
            for (int b2 = 0; b2 < 2; ++b2) {
                ptx::mbar_init(&wfull[b2], 4);
                ptx::mbar_init(&wempty[b2], 1);
            }
        }
        for (int a = 0; a < NA; ++a) {
            ptx::mbar_init(&tfull[a], 1);
            ptx::mbar_init(&tempty[a], 4);
        }
        for (int b2 = 0; b2 < 2; ++b2) {
            ptx::mbar_init(&qfull[b2], 1);
            ptx::mbar_init(&qempty[b2], P + 8);  // each MMA issuer's commit + every epilogue warp
        }
        ptx::mbar_init(hsync, 8);
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, C::kTmemCols);
        ptx::tmem_relinquish();
    }
    if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 8) {
        // This CTA's share of the work.  A segment of n > 0 tiles weighs n + kSegCost: with the
        // histogram, leaving a segment (both epilogue groups meet, flush the bins, meet again)
        // costs about two tiles' time, without it next to nothing.  The CTAs take equal ranges
        // [w0, w1) of the total weight, and a CTA's tiles are the tiles whose positions fall in its
        // range (the first kSegCost positions of a segment hold none).  Scans carry
        // (weight << 32) + tiles: one scan when every segment has its own thread, else a total pass
        // and a search pass over chunks of 256 segments.
        constexpr int kSegCost = HIST ? 2 : 0;
        const int t = threadIdx.x - kEpiWarp0 * 32;
        Seg tmp;
        auto packed = [&](int n) -> int64_t {
            return n > 0 ? ((static_cast<int64_t>(n) + kSegCost) << 32) + n : 0;
        };
        // (this thread's segment ends at packed prefix incl and holds n tiles) claim the share's
        // first tile and add / subtract the tile positions of w1 and w0 into the count
        auto claim = [&](int sidx, int n, int64_t incl, int64_t w0, int64_t w1) {
            if (n <= 0) return;
            const int64_t e = incl >> 32, s = e - (n + kSegCost);   // weight range [s, e)
            const int64_t tiles_before = (incl & 0xffffffffLL) - n;
            if (w1 > w0 && s <= w0 && w0 < e) {
                const int64_t k = w0 - s > kSegCost ? w0 - s - kSegCost : 0;
                part[0] = sidx;
                part[1] = static_cast<int32_t>(k);
                atomicSub(&part[2], static_cast<int32_t>(tiles_before + k));
            }
            if (w1 > w0 && s <= w1 && w1 < e)
                atomicAdd(&part[2], static_cast<int32_t>(tiles_before + (w1 - s > kSegCost ? w1 - s - kSegCost : 0)));
        };
        if (nseg <= 256) {
            const int n = (t < nseg) ? seg_load(sa, t, tmp) : 0;
            int64_t total;
            const int64_t incl = epi_scan(packed(n), scan_scratch, &total);
            const int64_t W = total >> 32;
            const int64_t w0 = W * blockIdx.x / gridDim.x;
            const int64_t w1 = W * (blockIdx.x + 1) / gridDim.x;
            if (t == 0) {
                part[0] = nseg;
                part[1] = 0;
                part[2] = (w1 > w0 && w1 == W) ? static_cast<int32_t>(total & 0xffffffffLL) : 0;
            }
            asm volatile("bar.sync 1, 256;" ::: "memory");   // the defaults above before the claims
            claim(t, n, incl, w0, w1);
            asm volatile("bar.sync 1, 256;" ::: "memory");   // the start segment is known
            // the share's first segments into the table (each thread holds its own segment)
            const int s0 = part[0];
            if (t >= s0 && t < s0 + kSegTab && t < nseg) segtab[t - s0] = tmp;
            if (t == 0) *segtab_n = s0 < nseg ? min(kSegTab, nseg - s0) : 0;
        } else {
            if (t == 0) *segtab_n = 0;
            int64_t mine = 0;
            for (int sidx = t; sidx < nseg; sidx += 256) mine += packed(seg_load(sa, sidx, tmp));
            int64_t total;
            epi_scan(mine, scan_scratch, &total);
            const int64_t W = total >> 32;
            const int64_t w0 = W * blockIdx.x / gridDim.x;
            const int64_t w1 = W * (blockIdx.x + 1) / gridDim.x;
            if (t == 0) {
                part[0] = nseg;
                part[1] = 0;
                part[2] = (w1 > w0 && w1 == W) ? static_cast<int32_t>(total & 0xffffffffLL) : 0;
            }
            asm volatile("bar.sync 1, 256;" ::: "memory");   // the defaults above before the claims
            if (w1 > w0) {
                int64_t seen = 0;   // packed sum over the chunks before
                for (int c0 = 0; c0 < nseg; c0 += 256) {
                    const int n = (c0 + t < nseg) ? seg_load(sa, c0 + t, tmp) : 0;
                    int64_t chunk_total;
                    const int64_t incl = epi_scan(packed(n), scan_scratch, &chunk_total) + seen;
                    claim(c0 + t, n, incl, w0, w1);
                    seen += chunk_total;
                    if ((seen >> 32) > w1) break;
                }
            }
        }
    }
    if (HIST && warp >= kEpiWarp0 && warp < kEpiWarp0 + 8)
        for (int i = threadIdx.x - kEpiWarp0 * 32; i < R * kTopBins; i += 256) hist_s[i] = 0u;
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int count = part[2];
    const uint64_t deadline = ptx::wait_deadline();
    bool timed_out = false;
    const SegArgs sat{seq_lens, cu_q, B, G, R, row_begin, row_end, cmp_shift, segtab, part[0], *segtab_n};
    Seg sg;
    if (count > 0) {
        seg_load(sat, part[0], sg);
        sg.tile = part[1];
    }

    if ((warp == 0 || (P == 2 && warp == kProducer1Warp)) && count > 0) {   // ---------------- key producer
        const int pipe = warp == 0 ? 0 : 1;   // issues the tiles i with i % P == pipe
        int32_t win = -1;           // block-table entries 2 * wbase + lane of segment wseg
        int wbase = -1, wseg = -1;
        for (int i = 0; i < count; ++i) {
          if (i % P == pipe) {
            const int s = stage_of(i);
            const uint32_t ph = stage_ph(i);
            const int wb = sg.tile & ~15;
            if (wb != wbase || sg.sidx != wseg) {
                wbase = wb;
                wseg = sg.sidx;
                const int e = 2 * wb + lane;
                win = (e < 2 * sg.ntiles && e < max_pages)
                          ? __ldg(block_table + static_cast<int64_t>(sg.b) * max_pages + e)
                          : -1;
            }
            const int32_t pg0 = __shfl_sync(0xffffffffu, win, 2 * (sg.tile - wb));
            const int32_t pg1 = __shfl_sync(0xffffffffu, win, 2 * (sg.tile - wb) + 1);
            if (lane == 0) {
                // (without the histograms) the rest of the ring after each pipeline's first tile goes
                // out 0.4 us later, so that the first tiles of all CTAs are served ahead of the
                // start-up burst (~25 MB): the CTAs then start together instead of up to ~2 us apart
                if (!HIST && i == P + pipe) __nanosleep(400);
                if (!ptx::mbar_wait(&empty[s], ph ^ 1u, deadline)) timed_out = true;
                if (!timed_out) {
                    const bool need1 = sg.tile * kTileKeys + kPage < sg.vmax;
                    const bool ok0 = pg0 >= 0 && pg0 < num_pages;
                    const bool ok1 = need1 && pg1 >= 0 && pg1 < num_pages;
                    if (!ok0 || (need1 && !ok1)) raise_error(err, DSA_DEVERR_PAGE_RANGE);
                    page_ok[2 * s] = ok0;
                    page_ok[2 * s + 1] = ok1;
                    const uint32_t bytes = (ok0 ? (kPage * kIndexDim + kPage * C::kScaleElem) : 0) +
                                           (ok1 ? (kPage * kIndexDim + kPage * C::kScaleElem) : 0);
                    ptx::mbar_arrive_expect_tx(&full[s], bytes);
                    unsigned char* dst = codes + s * kTileCodeBytes;
                    if (ok0) {
                        ptx::tma_load_3d(dst, &kmap, &full[s], 0, 0, pg0);
                        ptx::bulk_load(scales_b + s * kTileKeys * C::kScaleElem,
                                       pool + static_cast<int64_t>(pg0) * C::kPoolPageBytes + C::kPoolScaleOff,
                                       kPage * C::kScaleElem, &full[s]);
                    }
                    if (ok1) {
                        ptx::tma_load_3d(dst + kPage * kIndexDim, &kmap, &full[s], 0, 0, pg1);
                        ptx::bulk_load(scales_b + (s * kTileKeys + kPage) * C::kScaleElem,
                                       pool + static_cast<int64_t>(pg1) * C::kPoolPageBytes + C::kPoolScaleOff,
                                       kPage * C::kScaleElem, &full[s]);
                    }
                }
            }
            if (__shfl_sync(0xffffffffu, timed_out ? 1 : 0, 0)) { timed_out = true; break; }
          }
            if (++sg.tile == sg.ntiles && i + 1 < count) seg_next(sat, sg);
        }
    } else if (warp == kLoaderWarp && count > 0) {   // ---------------- query-tile loader
        if (lane == 0) {
            ptx::griddep_wait();   // the prologue's workspace is complete and visible
            int remaining = count;
            for (int n = 0; remaining > 0; ++n) {
                const int qb = n & 1;
                if (!ptx::mbar_wait(&qempty[qb], ((n >> 1) & 1) ^ 1u, deadline)) { timed_out = true; break; }
                uint32_t bytes = 0;
                for (int jj = 0; jj < sg.nrows; ++jj) {
                    const int r = sg.q0 + sg.j0 + jj;
                    if (r >= row_begin && r < row_end) bytes += C::kQRowB + kQGateBytes;
                }
                ptx::mbar_arrive_expect_tx(&qfull[qb], bytes);
                for (int jj = 0; jj < sg.nrows; ++jj) {
                    const int r = sg.q0 + sg.j0 + jj;
                    if (r < row_begin || r >= row_end) continue;
                    const int64_t rr = r - row_begin;
                    if (C8) {   // the row's two 8 KB dim chunks go to the two chunk columns of the tile
                        for (int c = 0; c < 2; ++c)
                            ptx::bulk_load(qtile + qb * C::kQBytes + c * (R * 8192) + jj * 8192,
                                           q_codes + rr * kQRowBytesC8 + c * 8192, 8192, &qfull[qb]);
                    } else {
                        ptx::bulk_load(qtile + qb * C::kQBytes + jj * kQRowBytes, q_codes + rr * kQRowBytes,
                                       kQRowBytes, &qfull[qb]);
                    }
                    ptx::bulk_load(gates + (qb * R + jj) * kIndexHeads, q_gates + rr * kIndexHeads, kQGateBytes,
                                   &qfull[qb]);
                }
                remaining -= sg.ntiles - sg.tile;
                if (remaining > 0) seg_next(sat, sg);
            }
        }
    } else if ((warp == 1 || (P == 2 && warp == kMma1Warp)) && count > 0) {   // ---------------- MMA issuer
        if (lane == 0) {
            const int pipe = warp == 1 ? 0 : 1;   // issues the tiles i with i % P == pipe
            constexpr uint32_t idesc = ptx::instr_desc(0, 0, kTileKeys, N);
            int n = 0;
            bool seg_start = true;
            for (int i = 0; i < count && !timed_out; ++i) {
                const int qb = n & 1;
                // every issuer meets every segment's query tile, so that each segment's release of
                // the tile (qempty) gets one commit per issuer after its last MMA on it
                if (seg_start && !ptx::mbar_wait(&qfull[qb], (n >> 1) & 1, deadline)) { timed_out = true; break; }
                seg_start = false;
              if (i % P == pipe) {
                const int s = stage_of(i);
                const uint32_t ph = stage_ph(i);
                const int a = acc_of(i);
                const uint32_t aph = acc_ph(i);
                if (C8) {
                    if (!ptx::mbar_wait(&wfull[i & 1], (i >> 1) & 1, deadline)) { timed_out = true; break; }
                } else if (!ptx::mbar_wait(&full[s], ph, deadline)) {
                    timed_out = true;
                    break;
                }
                if (!ptx::mbar_wait(&tempty[a], aph ^ 1u, deadline)) { timed_out = true; break; }
                ptx::tc_fence_after_sync();
                const uint32_t q_addr = ptx::smem_addr(qtile + qb * C::kQBytes);
                const uint32_t d = tmem + static_cast<uint32_t>(a * N);
                if (C8) {
                    // f16 x f16 (kind::f16, format code 0 for both): K = 16 per instruction, the 128
                    // dims in two 64-dim chunk columns of both operands
                    ptx::fence_proxy_async_smem();
                    const uint32_t a_addr = ptx::smem_addr(wtile + (i & 1) * kWTileBytes);
#pragma unroll
                    for (int k = 0; k < kIndexDim / 16; ++k) {
                        const uint32_t off = (k & 3) * 32;
                        ptx::umma_f16(d, ptx::sw128_kmajor_desc(a_addr + (k >> 2) * (kTileKeys * 128) + off),
                                      ptx::sw128_kmajor_desc(q_addr + (k >> 2) * (R * 8192) + off), idesc,
                                      k > 0 ? 1u : 0u);
                    }
                    ptx::umma_commit(&wempty[i & 1]);
                } else {
                    const uint32_t a_addr = ptx::smem_addr(codes + s * kTileCodeBytes);
#pragma unroll
                    for (int k = 0; k < kIndexDim / 32; ++k)
                        ptx::umma_f8f6f4(d, ptx::sw128_kmajor_desc(a_addr + k * 32),
                                         ptx::sw128_kmajor_desc(q_addr + k * 32), idesc, k > 0 ? 1u : 0u);
                    ptx::umma_commit(&empty[s]);
                }
                ptx::umma_commit(&tfull[a]);
              }
                if (++sg.tile == sg.ntiles || i + 1 == count) {   // last tile of the segment here
                    ptx::umma_commit(&qempty[qb]);
                    ++n;
                    seg_start = true;
                    if (i + 1 < count) seg_next(sat, sg);
                }
            }
        }
    } else if (C8 && warp >= kWidenWarp0 && warp < kWidenWarp0 + 4 && count > 0) {   // ------- int8 -> f16
        // thread t of the 4 warps owns key row t of every tile: its 8 swizzled 16-byte pieces of
        // int8 codes become 16 f16 pieces in the two 64-dim chunk columns of the f16 tile
        const int key = (warp - kWidenWarp0) * 32 + lane;
        int s = 0;
        uint32_t ph = 0;
        for (int i = 0; i < count; ++i) {
            const int wb = i & 1;
            if (!ptx::mbar_wait(&full[s], ph, deadline)) { timed_out = true; break; }
            if (!ptx::mbar_wait(&wempty[wb], ((i >> 1) & 1) ^ 1u, deadline)) { timed_out = true; break; }
            const unsigned char* src = codes + s * kTileCodeBytes + key * 128;
            unsigned char* dst = wtile + wb * kWTileBytes + key * 128;
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const uint4 c = *reinterpret_cast<const uint4*>(src + ((p ^ (key & 7)) << 4));
                uint4 lo, hi;
                i8x4_to_f16x4(c.x, lo.x, lo.y);
                i8x4_to_f16x4(c.y, lo.z, lo.w);
                i8x4_to_f16x4(c.z, hi.x, hi.y);
                i8x4_to_f16x4(c.w, hi.z, hi.w);
                unsigned char* row = dst + (p >> 2) * (kTileKeys * 128);
                const int j0 = 2 * (p & 3);
                *reinterpret_cast<uint4*>(row + ((j0 ^ (key & 7)) << 4)) = lo;
                *reinterpret_cast<uint4*>(row + (((j0 + 1) ^ (key & 7)) << 4)) = hi;
            }
            ptx::fence_proxy_async_smem();   // read by the tensor cores
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(&wfull[wb]);
                ptx::mbar_arrive(&empty[s]);
            }
            if (++s == S) { s = 0; ph ^= 1u; }
        }
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 8 && count > 0) {   // ---------------- epilogue
        const int grp = (warp - kEpiWarp0) >> 2;          // takes the tiles i with i % 2 == grp
        uint32_t hph = 0;                                  // HIST: next phase of hsync
        const int quad = warp & 3;
        const int key_in_tile = quad * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        int n = 0;
        bool seg_start = true;
        for (int i = 0; i < count; ++i) {
            const int qb = n & 1;
            if (seg_start && !ptx::mbar_wait(&qfull[qb], (n >> 1) & 1, deadline)) { timed_out = true; break; }
            seg_start = false;
            if ((i & 1) == grp) {   // with two pipelines: the tiles of pipeline grp
                const int s = stage_of(i);
                const uint32_t ph = stage_ph(i);
                const int a = acc_of(i);
                const uint32_t aph = acc_ph(i);
                if (!ptx::mbar_wait(&full[s], ph, deadline)) { timed_out = true; break; }
                if (!ptx::mbar_wait(&tfull[a], aph, deadline)) { timed_out = true; break; }
                ptx::tc_fence_after_sync();
                const bool ok = page_ok[2 * s + (key_in_tile >> 6)] != 0;
                float ks;
                if (C8) ks = __half2float(reinterpret_cast<const __half*>(scales_b)[s * kTileKeys + key_in_tile]);
                else ks = scales[s * kTileKeys + key_in_tile];
                const int key = sg.tile * kTileKeys + key_in_tile;
#pragma unroll 1
                for (int jj = 0; jj < sg.nrows; ++jj) {   // one query row at a time: 64 accumulator columns
                    uint32_t r0[32], r1[32];
                    const uint32_t col = tmem + lane_base + static_cast<uint32_t>(a * N + jj * kIndexHeads);
                    ptx::tmem_ld_32x32b_x32(col, r0);
                    ptx::tmem_ld_32x32b_x32(col + 32, r1);
                    ptx::tmem_wait_ld();
                    const float* g = gates + (qb * R + jj) * kIndexHeads;
                    float acc = 0.0f;
                    if constexpr (!C8) {
                        // the head sum as two interleaved partial sums (even / odd heads) with packed
                        // two-lane FMAs, added at the end: half the FMA instructions of the epilogue
                        // (with int8 keys, where the widen warps share the issue slots, it measured
                        // no better and keeps one sum in head order)
                        uint64_t acc2 = 0;   // the bit pattern of (0.0f, 0.0f)
                        const uint64_t* g2 = reinterpret_cast<const uint64_t*>(g);
#pragma unroll
                        for (int h = 0; h < 32; h += 2)
                            fma2_relu(acc2, g2[h / 2], r0[h], r0[h + 1]);
#pragma unroll
                        for (int h = 0; h < 32; h += 2)
                            fma2_relu(acc2, g2[16 + h / 2], r1[h], r1[h + 1]);
                        float lo, hi;
                        asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(acc2));
                        acc = lo + hi;
                    } else {
#pragma unroll
                        for (int h = 0; h < 32; ++h) acc = fmaf(g[h], fmaxf(__uint_as_float(r0[h]), 0.0f), acc);
#pragma unroll
                        for (int h = 0; h < 32; ++h) acc = fmaf(g[32 + h], fmaxf(__uint_as_float(r1[h]), 0.0f), acc);
                    }
                    const int r = sg.q0 + sg.j0 + jj;
                    const int v = visible_len(sg.L, sg.q_len, sg.j0 + jj) >> cmp_shift;
                    if (HIST) {
                        // every visible key gets a logit (-inf where its page id was bad) and is
                        // counted, so the histogram describes exactly the row the top-k reads
                        if (key < v && key < ld && r >= row_begin && r < row_end) {
                            const float val = ok ? acc * ks : -INFINITY;
                            logits[static_cast<int64_t>(r - row_begin) * ld + key] = val;
                            atomicAdd(&hist_s[jj * kTopBins + (logit_order_key(val) >> 20)], 1u);
                        }
                    } else if (ok && key < v && key < ld && r >= row_begin && r < row_end) {
                        logits[static_cast<int64_t>(r - row_begin) * ld + key] = acc * ks;
                    }
                }
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    ptx::mbar_arrive(&tempty[a]);
                    ptx::mbar_arrive(&empty[s]);
                }
            }
            if (++sg.tile == sg.ntiles || i + 1 == count) {   // leaving the segment: its gates are free
                if (HIST) {
                    // every epilogue warp's counts of this segment are in; add the non-empty bins to
                    // the rows' global histograms and clear them for the next segment
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(hsync);
                    if (!ptx::mbar_wait(hsync, hph, deadline)) { timed_out = true; break; }
                    hph ^= 1u;
                    const int t = threadIdx.x - kEpiWarp0 * 32;
                    for (int jj = 0; jj < sg.nrows; ++jj) {
                        const int r = sg.q0 + sg.j0 + jj;
                        const bool live = r >= row_begin && r < row_end;
                        uint32_t* hg = hist_g + static_cast<int64_t>(r - row_begin) * kTopBins;
                        for (int bin = t; bin < kTopBins; bin += 256) {
                            const uint32_t c = hist_s[jj * kTopBins + bin];
                            if (c != 0u) {
                                if (live) atomicAdd(hg + bin, c);
                                hist_s[jj * kTopBins + bin] = 0u;
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(hsync);
                    if (!ptx::mbar_wait(hsync, hph, deadline)) { timed_out = true; break; }
                    hph ^= 1u;
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&qempty[qb]);
                ++n;
                seg_start = true;
                if (i + 1 < count) seg_next(sat, sg);
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

extern "C" size_t dsa_indexer_logits_workspace_size(int32_t rows) {
    using namespace dsa;
    return rows <= 0 ? 0 : static_cast<size_t>(rows) * (kQRowBytes + kQGateBytes);
}

extern "C" size_t dsa_indexer_logits_c8_workspace_size(int32_t rows) {
    using namespace dsa;
    return rows <= 0 ? 0 : static_cast<size_t>(rows) * (kQRowBytesC8 + kQGateBytes);
}

namespace dsa {

// The logits call; with hist_g != nullptr (row groups of at most 2 rows) the kernel also adds each
// row's top-12-bit order-key histogram into hist_g[(r - row_begin) * 4096 ..] (zeroed here by the
// query prologue).
dsa_status indexer_logits_launch(const void* q_bf16, const float* weights, const uint8_t* index_k_pool,
                                 int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                 const int32_t* seq_lens, const int32_t* cu_q, int32_t B, int32_t max_seq_len,
                                 int32_t max_q_len, int32_t row_begin, int32_t row_end, float* logits, int64_t ld,
                                 uint32_t flags, void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream,
                                 uint32_t* hist_g) {
    if (B < 0 || max_seq_len < 0 || max_q_len < 0 || row_begin < 0 || row_end < row_begin || max_pages < 0 ||
        num_pages < 0)
        return DSA_ERR_INVALID_ARG;
    if ((flags & ~(DSA_Q_ROTATE | DSA_SCALE_UE8M0 | DSA_KEYS_CMP4)) != 0u) return DSA_ERR_INVALID_ARG;
    const int cmp_shift = (flags & DSA_KEYS_CMP4) != 0u ? 2 : 0;
    if (B == 0 || row_end == row_begin || max_seq_len == 0 || max_q_len == 0) return DSA_OK;
    if (!q_bf16 || !weights || !index_k_pool || !block_table || !seq_lens || !cu_q || !logits || !workspace)
        return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_bf16) || !aligned16(index_k_pool) || !aligned16(workspace)) return DSA_ERR_INVALID_ARG;
    if (ws_bytes < dsa_indexer_logits_workspace_size(row_end - row_begin)) return DSA_ERR_INVALID_ARG;
    if (ld < max_seq_len) return DSA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(max_pages) * kPage < max_seq_len) return DSA_ERR_INVALID_ARG;
    const int R = max_q_len >= 4 ? 4 : (max_q_len >= 2 ? 2 : 1);
    if (hist_g != nullptr && R > 2) return DSA_ERR_UNSUPPORTED;
    const int groups = (max_q_len + R - 1) / R;
    if (static_cast<int64_t>(groups) * B > 0x7fffffffLL - 1) return DSA_ERR_UNSUPPORTED;
    if (num_pages > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
    const int64_t tiles_per_seg = (max_seq_len + kTileKeys - 1) / kTileKeys;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return DSA_ERR_CUDA;
    const int64_t upper = tiles_per_seg * groups * B;   // bound on the tiles of all segments
    const int ctas = static_cast<int>(upper < sms ? upper : sms);

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
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // query prologue mode: bit 0 rotate, bit 1 power-of-two scales
    const int mode = ((flags & DSA_Q_ROTATE) != 0u ? 1 : 0) | ((flags & DSA_SCALE_UE8M0) != 0u ? 2 : 0);
    const int rows = row_end - row_begin;
    uint8_t* q_codes = static_cast<uint8_t*>(workspace);
    float* q_gates = reinterpret_cast<float*>(q_codes + static_cast<size_t>(rows) * kQRowBytes);

    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // query prologue: 8 vectors per 256-thread block; a programmatic dependent of the previous kernel
    // on the stream (it waits on the device for that kernel's completion before any access but its
    // L2 prefetches of the lengths and row offsets)
    {
        cudaLaunchConfig_t pcfg = {};
        pcfg.gridDim = dim3(static_cast<unsigned>(rows) * (kIndexHeads / 8), 1, 1);
        pcfg.blockDim = dim3(256, 1, 1);
        pcfg.stream = st;
        pcfg.attrs = attr;
        pcfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&pcfg, indexer_q_prologue_kernel, static_cast<const uint16_t*>(q_bf16), weights, cu_q,
                               static_cast<int>(B), static_cast<int>(row_begin), static_cast<int>(row_end), mode,
                               q_codes, q_gates, hist_g, seq_lens) != cudaSuccess)
            return DSA_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const uint8_t* qc = q_codes;
    const float* qg = q_gates;
#define DSA_LAUNCH_IDX(RR, HH)                                                                                  \
    do {                                                                                                        \
        const size_t smem = IdxCfg<RR, HH>::kSmemBytes;                                                         \
        cfg.blockDim = dim3(IdxCfg<RR, HH>::kThreadsCfg, 1, 1);                                                 \
        if (cudaFuncSetAttribute(indexer_logits_umma_kernel<RR, HH, false>,                                     \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess) \
            return DSA_ERR_CUDA;                                                                                \
        cfg.dynamicSmemBytes = smem;                                                                            \
        if (cudaLaunchKernelEx(&cfg, indexer_logits_umma_kernel<RR, HH, false>, kmap, qc, qg, index_k_pool, num_pages, \
                               block_table, static_cast<int>(max_pages), seq_lens, cu_q, static_cast<int>(B),  \
                               groups, static_cast<int>(row_begin), static_cast<int>(row_end), logits, ld,     \
                               dev_err, hist_g, cmp_shift) != cudaSuccess)                                      \
            return DSA_ERR_CUDA;                                                                                \
    } while (0)
    if (hist_g != nullptr) {
        if (R == 1) DSA_LAUNCH_IDX(1, true);
        else DSA_LAUNCH_IDX(2, true);
    } else if (R == 1) DSA_LAUNCH_IDX(1, false);
    else if (R == 2) DSA_LAUNCH_IDX(2, false);
    else DSA_LAUNCH_IDX(4, false);
#undef DSA_LAUNCH_IDX
    return launch_status();
}

}  // namespace dsa

extern "C" dsa_status dsa_indexer_logits(const void* q_bf16, const float* weights, const uint8_t* index_k_pool,
                                         int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                         const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                                         int32_t max_seq_len, int32_t max_q_len, int32_t row_begin,
                                         int32_t row_end, float* logits, int64_t ld, uint32_t flags,
                                         void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream) {
    return dsa::indexer_logits_launch(q_bf16, weights, index_k_pool, num_pages, block_table, max_pages, seq_lens,
                                      cu_q, B, max_seq_len, max_q_len, row_begin, row_end, logits, ld, flags,
                                      workspace, ws_bytes, dev_err, stream, nullptr);
}

namespace dsa {

// The logits call over the int8 ("c8") cache: query prologue (rotation, int8 quantisation, f16
// codes, fp16 gates), then the logits kernel with f16 tensor-core products of the int8 values.
dsa_status indexer_logits_c8_launch(const void* q_bf16, const float* weights, const uint8_t* pool,
                                    int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                    const int32_t* seq_lens, const int32_t* cu_q, int32_t B, int32_t max_seq_len,
                                    int32_t max_q_len, int32_t row_begin, int32_t row_end, float* logits, int64_t ld,
                                    void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream) {
    if (B < 0 || max_seq_len < 0 || max_q_len < 0 || row_begin < 0 || row_end < row_begin || max_pages < 0 ||
        num_pages < 0)
        return DSA_ERR_INVALID_ARG;
    if (B == 0 || row_end == row_begin || max_seq_len == 0 || max_q_len == 0) return DSA_OK;
    if (!q_bf16 || !weights || !pool || !block_table || !seq_lens || !cu_q || !logits || !workspace)
        return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_bf16) || !aligned16(pool) || !aligned16(workspace)) return DSA_ERR_INVALID_ARG;
    if (ws_bytes < dsa_indexer_logits_c8_workspace_size(row_end - row_begin)) return DSA_ERR_INVALID_ARG;
    if (ld < max_seq_len) return DSA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(max_pages) * kPage < max_seq_len) return DSA_ERR_INVALID_ARG;
    const int R = max_q_len >= 2 ? 2 : 1;
    const int groups = (max_q_len + R - 1) / R;
    if (static_cast<int64_t>(groups) * B > 0x7fffffffLL - 1) return DSA_ERR_UNSUPPORTED;
    if (num_pages > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
    const int64_t tiles_per_seg = (max_seq_len + kTileKeys - 1) / kTileKeys;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return DSA_ERR_CUDA;
    const int64_t upper = tiles_per_seg * groups * B;
    const int ctas = static_cast<int>(upper < sms ? upper : sms);

    // tensor map over the code bytes of the page-blocked int8 pool: (byte in row, row in page, page)
    CUtensorMap kmap;
    {
        auto encode = tensor_map_encoder();
        if (encode == nullptr) return DSA_ERR_CUDA;
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kIndexDim), static_cast<cuuint64_t>(kPage),
                                    static_cast<cuuint64_t>(num_pages)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kIndexDim), static_cast<cuuint64_t>(kC8PageBytes)};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(kIndexDim), static_cast<cuuint32_t>(kPage), 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(pool), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DSA_ERR_CUDA;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int rows = row_end - row_begin;
    uint8_t* q_codes = static_cast<uint8_t*>(workspace);
    float* q_gates = reinterpret_cast<float*>(q_codes + static_cast<size_t>(rows) * kQRowBytesC8);
    indexer_q_prologue_c8_kernel<<<static_cast<unsigned>(rows) * (kIndexHeads / 8), 256, 0, st>>>(
        static_cast<const uint16_t*>(q_bf16), weights, cu_q, B, row_begin, row_end, q_codes, q_gates);
    if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;

    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas, 1, 1);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const uint8_t* qc = q_codes;
    const float* qg = q_gates;
    uint32_t* no_hist = nullptr;
#define DSA_LAUNCH_IDX_C8(RR)                                                                                   \
    do {                                                                                                        \
        using Cfg = IdxCfg<RR, false, true>;                                                                    \
        if (cudaFuncSetAttribute(indexer_logits_umma_kernel<RR, false, true>,                                   \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,                                   \
                                 static_cast<int>(Cfg::kSmemBytes)) != cudaSuccess)                             \
            return DSA_ERR_CUDA;                                                                                \
        cfg.blockDim = dim3(Cfg::kThreadsCfg, 1, 1);                                                            \
        cfg.dynamicSmemBytes = Cfg::kSmemBytes;                                                                 \
        if (cudaLaunchKernelEx(&cfg, indexer_logits_umma_kernel<RR, false, true>, kmap, qc, qg, pool, num_pages, \
                               block_table, static_cast<int>(max_pages), seq_lens, cu_q, static_cast<int>(B),  \
                               groups, static_cast<int>(row_begin), static_cast<int>(row_end), logits, ld,     \
                               dev_err, no_hist, 0) != cudaSuccess)                                             \
            return DSA_ERR_CUDA;                                                                                \
    } while (0)
    if (R == 1) DSA_LAUNCH_IDX_C8(1);
    else DSA_LAUNCH_IDX_C8(2);
#undef DSA_LAUNCH_IDX_C8
    return launch_status();
}

}  // namespace dsa

extern "C" dsa_status dsa_indexer_logits_c8(const void* q_bf16, const float* weights, const uint8_t* index_k_pool_c8,
                                            int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                            const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                                            int32_t max_seq_len, int32_t max_q_len, int32_t row_begin,
                                            int32_t row_end, float* logits, int64_t ld, void* workspace,
                                            size_t ws_bytes, int32_t* dev_err, void* stream) {
    return dsa::indexer_logits_c8_launch(q_bf16, weights, index_k_pool_c8, num_pages, block_table, max_pages,
                                         seq_lens, cu_q, B, max_seq_len, max_q_len, row_begin, row_end, logits, ld,
                                         workspace, ws_bytes, dev_err, stream);
}
