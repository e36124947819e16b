// sparse_mla.cu -- absorbed sparse MLA decode over the top-k selected latent rows (sm_103a).
//
// Follows vllm_ascend sfa_v1.py, _execute_sparse_flash_attention_process
// (npu_sparse_flash_attention with query = ql_nope, key = value = latent cache, query_rope /
// key_rope, sparse_indices = top-k, sparse_block_size = 1, block_table) and vllm mla/common.py,
// MLACommonImpl.forward decode branch (absorbed 576-wide query, one shared KV head; _forward_decode
// returns (out, lse); merge_attn_states merges partial results by their log-sum-exp).
//
// Work split.  CTA = (query row r, split j of the k selected entries, rank c of a 2-CTA cluster).
// Rank c owns the value dims 256 c .. 256 c + 255 (latent chunks 4c .. 4c+3 of 64 dims) and half of
// the rope dims, 512 + 32 c .. 512 + 32 c + 31: 288 of the 576 dims each.  A CTA reads only its own
// dims of every selected row (16-byte cp.async straight into the tensor-core operand layouts),
// keeps only its own query dims, computes the partial score tile over them, and the two CTAs swap
// partial score tiles through distributed shared memory (st.async, counted as transaction bytes on
// the receiver's mbarrier; the receiver returns a 4-byte st.async per warp once it has read them).
// Both then hold the full scores, run the same softmax (identical P: the fp32 sum is commutative)
// and each accumulates its 256 output dims from its own value chunks.  Nothing of a latent row is
// read twice or copied between the CTAs.
//
// Pipelining.  Score tiles are double-buffered in tensor memory and the swap buffers in shared
// memory, so the score MMAs of tile t+1 and the swap of its partial scores overlap the softmax of
// tile t; P is written back over its score tile in tensor memory (bf16) and read from there by the
// PV MMA, which leaves shared memory for a 4-deep load ring.
//
// Tensor memory (512 columns x 128 lanes, lane = head):
//   [0, 256)    O, this CTA's 256 output dims (fp32)
//   [256, 320)  score tile buffer 0 (fp32, 64 keys); P of that tile over its first 32 columns
//   [320, 384)  score tile buffer 1
//   [384, 512)  this CTA's 4 value-dim query chunks, the A operand of the score MMA (two bf16 per column)
// Shared memory: 4 stages of 64 keys x (4 chunks of 128 B, 128-byte swizzle, K-major; they double as
// the MN-major value operand) + (32 rope dims, no swizzle); 2 buffers of the peer's partial scores
// (32 KB each); the query's rope half (8 KB, no swizzle).
//
// Roles (416 threads), for tiles of 64 selected entries:
//   warps 0-7 (softmax): warp w reads TMEM lanes 32 (w % 4) .. +31 (head = lane), keys 32 (w / 4) ..
//           +31 of each tile.  Query into TMEM / shared memory; per tile: read its partial scores,
//           send them to the peer, add the peer's, tile max shared with the warp holding the other
//           keys of the same heads, online softmax in the log2 domain with lazy rescaling (O and l
//           are rescaled only when the running max grows by more than 8, so p <= 2^8 otherwise), P
//           into tensor memory as bf16; O / l and lse at the end (each warp 128 of the 256 dims);
//   warp 8 (MMA):  S = Q_c K_c^T (M = 128 heads, N = 64 keys, K = 288) and O += P V_c (M = 128,
//           N = 256 dims, K = 64 keys), bf16 in, fp32 accumulate in TMEM; issues whichever of the
//           next score MMA and the next PV is ready first;
//   warps 9-12 (producers): warp 9 + w resolves entries 16 w .. 16 w + 15 of each tile to latent
//           rows two batches ahead (independent loads) and copies this CTA's dims of those rows
//           (padding / invalid entries read row 0 and get probability 0).
// With one split the CTA writes bf16 output directly; with several, normalised fp32 partials and
// their lse go to the workspace and a combine kernel merges them.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "dsa_common.cuh"
#include "sm100_ptx.cuh"

namespace dsa {
namespace {

constexpr int kHeadsPerCta = 128;                 // M of both MMAs (fewer heads: rows unused)
constexpr int kKeysPerTile = 64;
constexpr int kOwnChunks = 4;                     // value chunks per CTA (64 dims, 128 B each)
constexpr int kRopeHalf = 32;                     // rope dims per CTA
constexpr int kHalfDims = kValueDim / 2;          // 256 output dims per CTA
constexpr int kKvChunkBytes = kKeysPerTile * 128;               // 8192
constexpr int kRopeBytes = kKeysPerTile * kRopeHalf * 2;        // 4096
constexpr int kKvStageBytes = kOwnChunks * kKvChunkBytes + kRopeBytes;   // 36864 (1024-aligned)
constexpr int kKvStages = 4;
constexpr int kXBytes = kHeadsPerCta * kKeysPerTile * 4;        // 32768: the peer's partial scores
constexpr int kQRopeBytes = kHeadsPerCta * kRopeHalf * 2;       // 8192
constexpr int kSoftmaxWarps = 8;
constexpr int kMmaWarp = 8;
constexpr int kProducerWarp0 = 9;
constexpr int kProducerWarps = 4;
constexpr int kMlaThreads = 32 * (kProducerWarp0 + kProducerWarps);   // 416
constexpr int kKeysPerProducer = kKeysPerTile / kProducerWarps;       // 16
static_assert(kKeysPerProducer == 8 || kKeysPerProducer == 16, "copy lane maps");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = kHalfDims;                          // score buffers at columns 256 and 320
constexpr uint32_t kTmemQ = kTmemS + 2 * kKeysPerTile;          // query chunks at columns 384 .. 511
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;                       // log2 units
constexpr int kBatch = 4;                                       // tiles resolved per batch
constexpr size_t kBarBytes = 4096;
constexpr size_t kMlaSmemBytes = 1024 + size_t(kKvStages) * kKvStageBytes + 2 * size_t(kXBytes) + kQRopeBytes +
                                 kBarBytes;

static_assert(kKvStageBytes % 1024 == 0, "stages keep the 1024-byte alignment of the swizzled chunks");
static_assert(kTmemQ + kOwnChunks * 32 == kTmemCols, "tensor-memory budget");
static_assert(kMlaSmemBytes <= 232448, "shared-memory budget");
// Shared-memory matrix descriptor (sm_100 format): start, leading / stride byte offsets, layout.
__device__ __forceinline__ uint64_t make_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(layout) << 61;
    return d;
}
constexpr uint32_t kLayoutNone = 0;
constexpr uint32_t kLayoutSw128 = 2;

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Arrive on `bar` (without raising its expected count) once all cp.async of this thread so far landed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(ptx::smem_addr(bar)) : "memory");
}

// Shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}

// 16-byte store into another CTA's shared memory, counted as transaction bytes on that CTA's
// mbarrier (no fence needed: the receiver's wait on the mbarrier orders the data).
__device__ __forceinline__ void st_async_v4(uint32_t addr, float a, float b, float c, float d, uint32_t bar_cluster) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     addr),
                 "f"(a), "f"(b), "f"(c), "f"(d), "r"(bar_cluster)
                 : "memory");
}

__device__ __forceinline__ void st_async_b32(uint32_t addr, uint32_t v, uint32_t bar_cluster) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr), "r"(v),
                 "r"(bar_cluster)
                 : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// 2^x on the special-function unit (PTX ex2.approx; relative error about 2^-22, ample for P in bf16).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// D[tmem] (+)= A[tmem] x B[smem]^T, bf16 operands, fp32 accumulate (one thread issues).
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Byte offset of 16-byte piece j (dims 8 j .. 8 j + 7) of row i in a K-major operand without
// swizzle whose rows hold 4 pieces (64 bytes): 8-row core matrices of 128 contiguous bytes, the 4
// core matrices of a row group 128 bytes apart (leading byte offset), row groups 512 bytes apart
// (stride byte offset).
__device__ __forceinline__ uint32_t rope_off(int i, int j) {
    return static_cast<uint32_t>((i >> 3) * 512 + j * 128 + (i & 7) * 16);
}

// Bit i: entry 32 kh + i of a tile is real, from the valid words of its producer warps.
__device__ __forceinline__ uint32_t half_valid_bits(const uint32_t (&words)[kProducerWarps], int kh) {
    constexpr int per_half = 32 / kKeysPerProducer;
    uint32_t v = 0;
#pragma unroll
    for (int w = 0; w < per_half; ++w) v |= words[kh * per_half + w] << (w * kKeysPerProducer);
    return v;
}

struct MlaBars {
    uint64_t q_full;               // query in TMEM / shared memory (8 softmax warps)
    uint64_t kv_full[kKvStages];   // every producer thread's cp.async landed + one arrive per producer warp
    uint64_t kv_empty[kKvStages];  // PV of the stage's tile completed
    uint64_t s_full[2];            // score MMAs of the buffer's tile completed
    uint64_t s_free[2];            // PV that read P from the buffer completed (buffer reusable)
    uint64_t p_full[2];            // P of the buffer's tile in TMEM (8 softmax warps)
    uint64_t x_full[2];            // the peer's partial scores are in x[b] (local arm + the peer's 32 KB)
    uint64_t x_free[2];            // the peer read the scores this CTA sent into its x[b] (local arm + 8 x 4 B)
    uint64_t o_full;               // last PV completed
    uint64_t pair[4];              // the two softmax warps of lane quadrant q (all 64 threads arrive)
    uint32_t x_sink[2][kSoftmaxWarps];   // targets of the peer's 4-byte consumed signals
    uint32_t tmem_slot;
    uint32_t pad;
    uint32_t valid[kKvStages][kProducerWarps];   // bit i: entry kKeysPerProducer w + i of the stage's tile is real
    float tmax[2][2][kHeadsPerCta];   // [tile parity][key half]: this tile's maximum (shared by the warp pair)
    float lsum[2][kHeadsPerCta];   // per key half: the final partial row sums
};
static_assert(sizeof(MlaBars) <= kBarBytes, "barrier block");

// The second source of entries of the compressed-KV attention (TWO = true): entries [0, win) of a
// row are the window positions v - win .. v - 1 of the main cache, entries [win, win + k2) the
// listed compressed entries of cache 2 (visible while < v >> shift2).  An entry's source travels
// in bit 30 of its position and of its row id (both caches hold fewer than 2^30 rows).
struct TwoSrc {
    const uint16_t* kv2;
    int64_t num_pages2;
    const int32_t* block_table2;
    int max_pages2;
    int shift2;
    const int32_t* idx2;
    int k2;
    int win;
    const float* sinks;   // [H] sink logits, folded into the softmax denominator (one split)
};
constexpr int kSrc2 = 1 << 30;

template <bool TWO>
__global__ void __launch_bounds__(kMlaThreads, 1)
sparse_mla_umma_kernel(const uint16_t* __restrict__ kv, const uint16_t* __restrict__ q, int64_t num_pages,
                       const int32_t* __restrict__ block_table, int max_pages, const int32_t* __restrict__ seq_lens,
                       const int32_t* __restrict__ cu_q, int B, const int32_t* __restrict__ idx, int k, int H,
                       float scale, int splits, int cmp_shift, int part_stride, int part_base,
                       uint16_t* __restrict__ out, float* __restrict__ lse_out, float* __restrict__ part_o,
                       float* __restrict__ part_lse, int32_t* err, TwoSrc ts) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    unsigned char* base = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    unsigned char* kvs = base;                                         // [4][4 chunks x 8 KB | rope 4 KB]
    float* xs = reinterpret_cast<float*>(kvs + kKvStages * kKvStageBytes);   // [2][2 halves][8 quads][128 heads][4]
    unsigned char* qrope = reinterpret_cast<unsigned char*>(xs) + 2 * kXBytes;   // [128 heads x 32 dims], no swizzle
    MlaBars& bar = *reinterpret_cast<MlaBars*>(qrope + kQRopeBytes);

    const int split = blockIdx.y;
    const int r = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = row_request(cu_q, B, r);
    const int q0 = __ldg(cu_q + b);
    const int v = visible_len(__ldg(seq_lens + b), __ldg(cu_q + b + 1) - q0, r - q0) >> cmp_shift;
    const int per_split = (k + splits - 1) / splits;
    const int e_begin = split * per_split;
    const int e_end = min(k, e_begin + per_split);
    const int ntiles = e_end > e_begin ? (e_end - e_begin + kKeysPerTile - 1) / kKeysPerTile : 0;
    const uint32_t crank = cluster_ctarank();
    const uint32_t peer = crank ^ 1u;
    const int half = static_cast<int>(crank);   // output dims 256 half .., rope dims 512 + 32 half ..

    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar.q_full, kSoftmaxWarps);
        for (int s = 0; s < kKvStages; ++s) {
            ptx::mbar_init(&bar.kv_full[s], kProducerWarps * 32 + kProducerWarps);
            ptx::mbar_init(&bar.kv_empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&bar.s_full[a], 1);
            ptx::mbar_init(&bar.s_free[a], 1);
            ptx::mbar_init(&bar.p_full[a], kSoftmaxWarps);
            ptx::mbar_init(&bar.x_full[a], 1);
            ptx::mbar_init(&bar.x_free[a], 1);
        }
        ptx::mbar_init(&bar.o_full, 1);
        for (int qd = 0; qd < 4; ++qd) ptx::mbar_init(&bar.pair[qd], 64);
        ptx::fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(&bar.tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    cluster_sync_all();   // both CTAs' barriers exist before the peer signals or writes into them
    ptx::tc_fence_after_sync();
    const uint32_t tmem = bar.tmem_slot;
    const uint64_t deadline = ptx::wait_deadline();
    bool timed_out = false;
    const uint32_t kv_addr0 = ptx::smem_addr(kvs);

    if (warp >= kProducerWarp0) {
        // ---------------------------------------------------------------- producers
        const int pw = warp - kProducerWarp0;
        ptx::griddep_wait();   // launched as a programmatic dependent: the top-k indices are complete
        // lane l < 16 owns entry 16 pw + l of every tile.  Batches of kBatch tiles: positions are
        // loaded two batches ahead and page ids one batch ahead, so no load waits on another on the
        // critical path.
        const int my_entry = pw * kKeysPerProducer + lane;
        auto load_pos = [&](int tile) -> int {
            const int e = e_begin + tile * kKeysPerTile + my_entry;
            if (!(lane < kKeysPerProducer && tile < ntiles && e < e_end)) return -1;
            if (TWO) {
                if (e < ts.win) return v - ts.win + e;   // the window (negative: before the first token)
                const int p2 = __ldg(ts.idx2 + static_cast<int64_t>(r) * ts.k2 + (e - ts.win));
                return p2 >= 0 ? (p2 | kSrc2) : -1;
            }
            return __ldg(idx + static_cast<int64_t>(r) * k + e);
        };
        auto pos_ok = [&](int pos) -> bool {
            if (pos < 0) return false;
            if (TWO && (pos & kSrc2)) {
                const int p = pos & (kSrc2 - 1);
                return p < (v >> ts.shift2) && (p >> 6) < ts.max_pages2;
            }
            return pos >= 0 && pos < v && (pos >> 6) < max_pages;
        };
        auto load_page = [&](int pos) -> int {
            if (!pos_ok(pos)) return -1;
            if (TWO && (pos & kSrc2))
                return __ldg(ts.block_table2 + static_cast<int64_t>(b) * ts.max_pages2 + ((pos & (kSrc2 - 1)) >> 6));
            return __ldg(block_table + static_cast<int64_t>(b) * max_pages + (pos >> 6));
        };
        auto to_row = [&](int pos, int page) -> int {   // -1: padding or invalid (reported)
            if (pos < 0) return -1;
            if (!pos_ok(pos)) { raise_error(err, DSA_DEVERR_INDEX_RANGE); return -1; }
            const bool two = TWO && (pos & kSrc2);
            if (page < 0 || page >= (two ? ts.num_pages2 : num_pages)) { raise_error(err, DSA_DEVERR_PAGE_RANGE); return -1; }
            return (page * kPage + (pos & 63)) | (two ? kSrc2 : 0);
        };
        int pos1[kBatch], page1[kBatch], pos2[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) pos1[u] = load_pos(u);
#pragma unroll
        for (int u = 0; u < kBatch; ++u) page1[u] = load_page(pos1[u]);
#pragma unroll
        for (int u = 0; u < kBatch; ++u) pos2[u] = load_pos(kBatch + u);
        // value chunks: lane = 8 * (key % 4) + 16-byte piece of a 128-byte chunk row;
        // rope half: lane = 4 * (key % 8) + 16-byte piece of the 64-byte rope row
        const int piece = lane & 7;
        const int rpiece = lane & 3;
        const uint16_t* kv_val = kv + half * kHalfDims + piece * 8;
        const uint16_t* kv_rope = kv + kValueDim + half * kRopeHalf + rpiece * 8;
        const uint16_t* kv2_val = TWO ? ts.kv2 + half * kHalfDims + piece * 8 : nullptr;
        const uint16_t* kv2_rope = TWO ? ts.kv2 + kValueDim + half * kRopeHalf + rpiece * 8 : nullptr;
        for (int t0 = 0; t0 < ntiles && !timed_out; t0 += kBatch) {
            int rows[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) rows[u] = to_row(pos1[u], page1[u]);
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                pos1[u] = pos2[u];
                page1[u] = load_page(pos2[u]);
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) pos2[u] = load_pos(t0 + 2 * kBatch + u);
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int t = t0 + u;
                if (t >= ntiles) break;
                const int s = t % kKvStages;
                const uint32_t ph = (t / kKvStages) & 1;
                const uint32_t vbits = __ballot_sync(0xffffffffu, rows[u] >= 0) & ((1u << kKeysPerProducer) - 1u);
                const int row_src = rows[u] >= 0 ? rows[u] : 0;
                // the stage is free once PV of its previous tile completed
                if (lane == 0 && !ptx::mbar_wait(&bar.kv_empty[s], ph ^ 1u, deadline)) timed_out = true;
                timed_out = __shfl_sync(0xffffffffu, timed_out ? 1 : 0, 0) != 0;
                if (timed_out) break;
                const uint32_t stage = kv_addr0 + s * kKvStageBytes;
#pragma unroll
                for (int kq = 0; kq < kKeysPerProducer / 4; ++kq) {
                    const int kl = kq * 4 + (lane >> 3);                 // key within this warp's 16
                    const int key = pw * kKeysPerProducer + kl;
                    const int rr = __shfl_sync(0xffffffffu, row_src, kl);
                    const uint16_t* src = (TWO && (rr & kSrc2)) ? kv2_val + static_cast<int64_t>(rr & (kSrc2 - 1)) * kLatentDim
                                                                : kv_val + static_cast<int64_t>(rr) * kLatentDim;
#pragma unroll
                    for (int j = 0; j < kOwnChunks; ++j)
                        cp_async_16(stage + j * kKvChunkBytes + key * 128 + ((piece ^ (key & 7)) << 4), src + j * 64);
                }
#pragma unroll
                for (int kq = 0; kq < kKeysPerProducer / 8; ++kq) {
                    const int kl = kq * 8 + (lane >> 2);
                    const int key = pw * kKeysPerProducer + kl;
                    const int rr = __shfl_sync(0xffffffffu, row_src, kl);
                    const uint16_t* src = (TWO && (rr & kSrc2)) ? kv2_rope + static_cast<int64_t>(rr & (kSrc2 - 1)) * kLatentDim
                                                                : kv_rope + static_cast<int64_t>(rr) * kLatentDim;
                    cp_async_16(stage + kOwnChunks * kKvChunkBytes + rope_off(key, rpiece), src);
                }
                cp_async_arrive_noinc(&bar.kv_full[s]);
                if (lane == 0) {
                    bar.valid[s][pw] = vbits;
                    ptx::mbar_arrive(&bar.kv_full[s]);
                }
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = ptx::instr_desc(1, 1, kHeadsPerCta, kKeysPerTile);
            constexpr uint32_t idesc_pv = ptx::instr_desc(1, 1, kHeadsPerCta, kHalfDims) | (1u << 16);  // B MN-major
            const uint32_t qrope_addr = ptx::smem_addr(qrope);
            bool ok = ptx::mbar_wait(&bar.q_full, 0, deadline);
            int tq = 0, tp = 0;   // next score tile, next PV tile
            while (ok && tp < ntiles) {
                bool issued = false;
                // score MMAs of tile tq: its dims landed and its score buffer's previous PV completed
                if (tq < ntiles && ptx::mbar_test_wait(&bar.kv_full[tq % kKvStages], (tq / kKvStages) & 1) &&
                    ptx::mbar_test_wait(&bar.s_free[tq & 1], ((tq >> 1) & 1) ^ 1u)) {
                    ptx::fence_proxy_async_smem();   // rows written by cp.async, read by the tensor cores
                    ptx::tc_fence_after_sync();
                    const uint32_t kb = kv_addr0 + (tq % kKvStages) * kKvStageBytes;
                    const uint32_t d = tmem + kTmemS + (tq & 1) * kKeysPerTile;
#pragma unroll 1
                    for (int j = 0; j < kOwnChunks; ++j) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t db = make_desc(kb + j * kKvChunkBytes + kk * 32, 16, 1024, kLayoutSw128);
                            umma_f16_ts(d, tmem + kTmemQ + j * 32 + kk * 8, db, idesc_qk, (j | kk) != 0 ? 1u : 0u);
                        }
                    }
#pragma unroll
                    for (int kk = 0; kk < kRopeHalf / 16; ++kk) {
                        const uint64_t da = make_desc(qrope_addr + kk * 256, 128, 512, kLayoutNone);
                        const uint64_t db = make_desc(kb + kOwnChunks * kKvChunkBytes + kk * 256, 128, 512, kLayoutNone);
                        ptx::umma_f16(d, da, db, idesc_qk, 1u);
                    }
                    ptx::umma_commit(&bar.s_full[tq & 1]);
                    ++tq;
                    issued = true;
                }
                // O += P(tp) V(tp), P read from its score buffer in TMEM
                if (tp < tq && ptx::mbar_test_wait(&bar.p_full[tp & 1], (tp >> 1) & 1)) {
                    ptx::tc_fence_after_sync();
                    const int s = tp % kKvStages;
                    const uint32_t vb = kv_addr0 + s * kKvStageBytes;   // own chunks 0-3 = this CTA's value dims
                    const uint32_t pa = tmem + kTmemS + (tp & 1) * kKeysPerTile;
#pragma unroll
                    for (int ks = 0; ks < kKeysPerTile / 16; ++ks) {
                        const uint64_t db = make_desc(vb + ks * 16 * 128, kKvChunkBytes, 1024, kLayoutSw128);
                        umma_f16_ts(tmem, pa + ks * 8, db, idesc_pv, (tp | ks) != 0 ? 1u : 0u);
                    }
                    ptx::umma_commit(&bar.kv_empty[s]);
                    ptx::umma_commit(&bar.s_free[tp & 1]);
                    ++tp;
                    issued = true;
                }
                if (!issued && static_cast<uint64_t>(clock64()) > deadline) ok = false;
            }
            if (ok && ntiles > 0) ptx::umma_commit(&bar.o_full);
            if (!ok) timed_out = true;
        }
    } else {
        // ---------------------------------------------------------------- query, softmax, epilogue
        const int quad = warp & 3;                  // TMEM lanes 32 quad .. +31
        const int kh = warp >> 2;                   // keys 32 kh .. 32 kh + 31 of every tile
        const int head = quad * 32 + lane;          // TMEM lane = head
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        {
            // value chunks 2 kh, 2 kh + 1 of this CTA into TMEM; rope pieces 2 kh, 2 kh + 1 into
            // shared memory
            const uint4* src = reinterpret_cast<const uint4*>(q + (static_cast<int64_t>(r) * H + head) * kLatentDim);
            const bool live = head < H;
#pragma unroll 1
            for (int jj = 0; jj < 2; ++jj) {
                const int j = 2 * kh + jj;
                const int c = 4 * half + j;           // global chunk
                uint4 raw[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) raw[i] = live ? __ldg(src + c * 8 + i) : make_uint4(0u, 0u, 0u, 0u);
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    w[4 * i + 0] = raw[i].x;
                    w[4 * i + 1] = raw[i].y;
                    w[4 * i + 2] = raw[i].z;
                    w[4 * i + 3] = raw[i].w;
                }
                tmem_st_32x32b_x32(tmem + lane_base + kTmemQ + j * 32, w);
            }
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int j = 2 * kh + jj;
                const uint4 pr = live ? __ldg(src + (kValueDim + half * kRopeHalf) / 8 + j) : make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(qrope + rope_off(head, j)) = pr;
            }
            ptx::fence_proxy_async_smem();
            tmem_wait_st();
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bar.q_full);
        }
        const float cscale = scale * kLog2e;
        // the peer's x[b] for this thread's 32 scores: [b][kh][8 quads][128 heads][4]
        const uint32_t x_peer0 = map_to_rank(ptx::smem_addr(xs), peer) + (kh * 8 * kHeadsPerCta + head) * 16;
        float m_run = -INFINITY, l_run = 0.0f;
        // Tile u's partial scores: wait for its score MMAs, read this warp's 32 columns, send them to
        // the peer's x[u & 1] (once the peer has read what this CTA sent there for tile u - 2).  Tile
        // t + 1 is fetched and sent right after P(t), so its transfer overlaps the peer finishing
        // tile t and this warp's next receive finds the data there.
        uint32_t sr[32];
        auto fetch_send = [&](int u) -> bool {
            const int su = u % kKvStages;
            const int bu = u & 1;
            const uint32_t pu = (u >> 1) & 1;
            if (threadIdx.x == 0) ptx::mbar_arrive_expect_tx(&bar.x_full[bu], kXBytes);   // the peer's tile-u scores
            if (!ptx::mbar_wait(&bar.s_full[bu], pu, deadline)) return false;
            // the stage's tile landed (orders the producers' valid-bit words before they are read)
            if (!ptx::mbar_wait(&bar.kv_full[su], (u / kKvStages) & 1, deadline)) return false;
            ptx::tc_fence_after_sync();
            ptx::tmem_ld_32x32b_x32(tmem + lane_base + kTmemS + bu * kKeysPerTile + kh * 32, sr);
            ptx::tmem_wait_ld();
            if (u >= 2 && !ptx::mbar_wait(&bar.x_free[bu], pu ^ 1u, deadline)) return false;
            // arm the next phase (the peer's consumed signals of tile u) after the previous one completed
            if (threadIdx.x == 0) ptx::mbar_arrive_expect_tx(&bar.x_free[bu], kSoftmaxWarps * 4);
            const uint32_t xp = x_peer0 + bu * kXBytes;
            const uint32_t xf_peer = map_to_rank(ptx::smem_addr(&bar.x_full[bu]), peer);
#pragma unroll
            for (int kq = 0; kq < 8; ++kq)
                st_async_v4(xp + kq * (kHeadsPerCta * 16), __uint_as_float(sr[4 * kq]), __uint_as_float(sr[4 * kq + 1]),
                            __uint_as_float(sr[4 * kq + 2]), __uint_as_float(sr[4 * kq + 3]), xf_peer);
            return true;
        };
        if (ntiles > 0 && !fetch_send(0)) timed_out = true;
        for (int t = 0; t < ntiles && !timed_out; ++t) {
            const int s = t % kKvStages;
            const int bb = t & 1;
            const uint32_t ph = (t >> 1) & 1;
            if (!ptx::mbar_wait(&bar.x_full[bb], ph, deadline)) { timed_out = true; break; }
            {
                const float* xr = xs + bb * (kXBytes / 4) + (kh * 8 * kHeadsPerCta + head) * 4;
#pragma unroll
                for (int kq = 0; kq < 8; ++kq) {
                    const float4 o = *reinterpret_cast<const float4*>(xr + kq * (kHeadsPerCta * 4));
                    sr[4 * kq + 0] = __float_as_uint(__uint_as_float(sr[4 * kq + 0]) + o.x);
                    sr[4 * kq + 1] = __float_as_uint(__uint_as_float(sr[4 * kq + 1]) + o.y);
                    sr[4 * kq + 2] = __float_as_uint(__uint_as_float(sr[4 * kq + 2]) + o.z);
                    sr[4 * kq + 3] = __float_as_uint(__uint_as_float(sr[4 * kq + 3]) + o.w);
                }
            }
            __syncwarp();   // every lane's reads of x have returned (their values are in sr)
            if (lane == 0)
                st_async_b32(map_to_rank(ptx::smem_addr(&bar.x_sink[bb][warp]), peer), 1u,
                             map_to_rank(ptx::smem_addr(&bar.x_free[bb]), peer));
            const uint32_t vbits = half_valid_bits(bar.valid[s], kh);
            float tmax = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float sv = ((vbits >> i) & 1u) ? __uint_as_float(sr[i]) * cscale : -INFINITY;
                sr[i] = __float_as_uint(sv);
                tmax = fmaxf(tmax, sv);
            }
            // the tile maximum of this head over all 64 keys: shared with the other key half's warp
            // (phase t of the pair barrier; the values double-buffered by tile parity, so a value is
            // overwritten only after the partner has passed the next phase, i.e. has read it)
            bar.tmax[bb][kh][head] = tmax;
            ptx::mbar_arrive(&bar.pair[quad]);
            if (!ptx::mbar_wait(&bar.pair[quad], t & 1, deadline)) { timed_out = true; break; }
            tmax = fmaxf(tmax, bar.tmax[bb][kh ^ 1][head]);
            // lazy rescale: move the reference max only when the tile max exceeds it by > 8
            const bool grow = tmax > m_run + kRescaleThreshold || (m_run == -INFINITY && tmax > -INFINITY);
            const float m_new = grow ? tmax : m_run;
            const float alpha = grow ? ((m_run == -INFINITY) ? 0.0f : exp2f(m_run - m_new)) : 1.0f;
            if (t > 0 && __any_sync(0xffffffffu, grow)) {
                // O may only be rescaled once PV(t-1) has completed; this warp rescales its 128 columns
                if (!ptx::mbar_wait(&bar.s_free[(t - 1) & 1], ((t - 1) >> 1) & 1, deadline)) { timed_out = true; break; }
                ptx::tc_fence_after_sync();
#pragma unroll 1
                for (int cc = kh * 128; cc < kh * 128 + 128; cc += 32) {
                    uint32_t o[32];
                    ptx::tmem_ld_32x32b_x32(tmem + lane_base + cc, o);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st_32x32b_x32(tmem + lane_base + cc, o);
                }
                tmem_wait_st();
            }
            l_run *= alpha;
            m_run = m_new;
            float psum = 0.0f;
            uint32_t pk[16];
            const bool any = m_run != -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const float p0 = any ? fast_exp2(__uint_as_float(sr[i]) - m_run) : 0.0f;
                const float p1 = any ? fast_exp2(__uint_as_float(sr[i + 1]) - m_run) : 0.0f;
                psum += p0 + p1;
                pk[i / 2] = pack_bf16x2(p0, p1);
            }
            l_run += psum;
            // P of keys 32 kh .. +31 over columns 16 kh .. +15 of this tile's score buffer (both
            // warps of the pair read their scores before the pair barrier above)
            tmem_st_32x32b_x16(tmem + lane_base + kTmemS + bb * kKeysPerTile + kh * 16, pk);
            tmem_wait_st();
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bar.p_full[bb]);
            if (t + 1 < ntiles && !fetch_send(t + 1)) { timed_out = true; break; }
        }
        // the peer's last consumed signals land here before this CTA may finish
        if (!timed_out) {
            for (int t = (ntiles >= 2 ? ntiles - 2 : 0); t < ntiles; ++t)
                if (!ptx::mbar_wait(&bar.x_free[t & 1], (t >> 1) & 1, deadline)) { timed_out = true; break; }
        }
        // ---------------- epilogue: O / l, lse
        bar.lsum[kh][head] = l_run;
        ptx::mbar_arrive(&bar.pair[quad]);
        if (!timed_out && !ptx::mbar_wait(&bar.pair[quad], ntiles & 1, deadline)) timed_out = true;
        const float l_tot = l_run + bar.lsum[kh ^ 1][head];
        bool have_o = ntiles > 0 && !timed_out;
        if (have_o && !ptx::mbar_wait(&bar.o_full, 0, deadline)) { timed_out = true; have_o = false; }
        ptx::tc_fence_after_sync();
        float inv_l = l_tot > 0.0f ? 1.0f / l_tot : 0.0f;
        float lse = l_tot > 0.0f ? (m_run + log2f(l_tot)) / kLog2e : -INFINITY;
        const bool write_head = head < H;
        const int64_t rh = static_cast<int64_t>(r) * H + head;
        if (TWO && part_o == nullptr) {
            // the head's sink logit joins the denominator: D = l 2^m + 2^sink (log2 units)
            const float sl2 = (write_head ? __ldg(ts.sinks + head) : -INFINITY) * kLog2e;
            const float m_run_eff = l_tot > 0.0f ? m_run : -INFINITY;
            const float mf = fmaxf(m_run_eff, sl2);
            if (mf == -INFINITY) {
                inv_l = 0.0f;
                lse = -INFINITY;
            } else {
                const float a = l_tot > 0.0f ? l_tot * exp2f(m_run_eff - mf) : 0.0f;
                const float d = a + exp2f(sl2 - mf);
                inv_l = l_tot > 0.0f ? exp2f(m_run_eff - mf) / d : 0.0f;
                lse = (mf + log2f(d)) / kLog2e;
            }
        }
        if (part_o == nullptr) {
            uint16_t* dst = out + rh * kValueDim + half * kHalfDims;
#pragma unroll 1
            for (int cc = kh * 128; cc < kh * 128 + 128; cc += 32) {
                uint32_t o[32];
                if (have_o) {
                    ptx::tmem_ld_32x32b_x32(tmem + lane_base + cc, o);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                if (write_head) {
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(o[i]) * inv_l, __uint_as_float(o[i + 1]) * inv_l);
                        w.y = pack_bf16x2(__uint_as_float(o[i + 2]) * inv_l, __uint_as_float(o[i + 3]) * inv_l);
                        w.z = pack_bf16x2(__uint_as_float(o[i + 4]) * inv_l, __uint_as_float(o[i + 5]) * inv_l);
                        w.w = pack_bf16x2(__uint_as_float(o[i + 6]) * inv_l, __uint_as_float(o[i + 7]) * inv_l);
                        *reinterpret_cast<uint4*>(dst + cc + i) = w;
                    }
                }
            }
            if (write_head && half == 0 && kh == 0 && lse_out != nullptr) lse_out[rh] = lse;
        } else {
            float* dst = part_o + (rh * part_stride + part_base + split) * kValueDim + half * kHalfDims;
#pragma unroll 1
            for (int cc = kh * 128; cc < kh * 128 + 128; cc += 32) {
                uint32_t o[32];
                if (have_o) {
                    ptx::tmem_ld_32x32b_x32(tmem + lane_base + cc, o);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                if (write_head) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4*>(dst + cc + i) =
                            make_float4(__uint_as_float(o[i]) * inv_l, __uint_as_float(o[i + 1]) * inv_l,
                                        __uint_as_float(o[i + 2]) * inv_l, __uint_as_float(o[i + 3]) * inv_l);
                }
            }
            if (write_head && half == 0 && kh == 0) part_lse[rh * part_stride + part_base + split] = lse;
        }
    }
    if (timed_out) raise_error(err, DSA_DEVERR_TIMEOUT);
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
    cluster_sync_all();   // neither CTA leaves while its peer may still signal or write into it
}

// ---------------------------------------------------------------------------------------------
// FP8 latent cache (vllm mla/common.py, MLACommonImpl.forward with kv_cache_dtype "fp8": the cache
// rows are E4M3 codes of x / k_scale, the decode query is quantised by ops.scaled_fp8_quant with
// q_scale, and _forward_decode runs on the FP8 query and cache).  Same work split, swap and
// softmax as the bf16 kernel; the differences:
//   * a code stage (5 in a ring) holds this CTA's FP8 codes of the 64 selected rows -- value dims
//     256 c .. + 255 as two 128-byte swizzled K-major chunks, rope dims 512 + 32 c .. + 31 without
//     swizzle; the score MMA starts as soon as they land;
//   * the value dims are widened to bf16 (exact: E4M3 values are bf16 values) into one of two value
//     buffers in the MN-major value layout by two widen warps (one thread per key), as soon as the
//     codes have landed and the PV that read the buffer before has completed; the producers only
//     issue copies;
//   * the score MMA is E4M3 x E4M3 (kind::f8f6f4, K = 32) with the query's codes in tensor memory
//     (quantised there by the softmax warps with q_scale); S is scaled by scale * q_scale * k_scale;
//   * P stays bf16 and PV stays bf16 x bf16; O is scaled by k_scale at the end.
// ---------------------------------------------------------------------------------------------
constexpr int kF8ChunkBytes = kKeysPerTile * 128;                        // 128 value codes per row
constexpr int kF8RopeBytes = kKeysPerTile * kRopeHalf;                   // 32 rope codes per row
constexpr int kF8CodeBytes = 2 * kF8ChunkBytes + kF8RopeBytes;           // 18432
constexpr int kF8VBytes = kOwnChunks * kKvChunkBytes;                    // 32768: bf16 value dims
constexpr int kF8Stages = 5;                                             // code stages (tiles in flight)
constexpr int kF8VBufs = 2;                                              // bf16 value buffers
constexpr int kF8WidenWarp0 = kProducerWarp0 + kProducerWarps;          // warps 13, 14 widen the value codes
constexpr int kF8WidenWarps = 2;
constexpr int kF8Threads = 32 * (kF8WidenWarp0 + kF8WidenWarps);         // 480
constexpr uint32_t kF8TmemQRope = kTmemQ + 64;                           // query codes: value 64 + rope 8 columns
constexpr size_t kF8SmemBytes = 1024 + size_t(kF8Stages) * kF8CodeBytes + size_t(kF8VBufs) * kF8VBytes +
                                2 * size_t(kXBytes) + kBarBytes;
static_assert(kF8CodeBytes % 1024 == 0 && kF8VBytes % 1024 == 0, "1024-byte alignment of the swizzled parts");
static_assert(kF8WidenWarps * 32 == kKeysPerTile, "one widen thread per key of a tile");
static_assert(kF8SmemBytes <= 232448, "shared-memory budget");

struct Mla8Bars {
    uint64_t q_full;               // query codes in TMEM (8 softmax warps)
    uint64_t k_full[kF8Stages];    // every producer thread's cp.async landed + one arrive per producer warp
    uint64_t k_empty[kF8Stages];   // score MMAs done (1), codes widened (2 widen warps), valid bits read (8 warps)
    uint64_t v_full[kF8VBufs];     // values widened to bf16 (2 widen warps)
    uint64_t v_empty[kF8VBufs];    // PV that read the buffer completed
    uint64_t s_full[2], s_free[2], p_full[2], x_full[2], x_free[2];   // as in the bf16 kernel
    uint64_t o_full;
    uint64_t pair[4];
    uint32_t x_sink[2][kSoftmaxWarps];
    uint32_t tmem_slot;
    uint32_t pad;
    uint32_t valid[kF8Stages][kProducerWarps];
    float tmax[2][2][kHeadsPerCta];
    float lsum[2][kHeadsPerCta];
};
static_assert(sizeof(Mla8Bars) <= kBarBytes, "barrier block");

// Byte offset of 16-byte piece p (codes 16 p .. 16 p + 15) of row i of the rope codes: K-major without
// swizzle, rows of 32 bytes = two core matrices, 8-row groups 256 bytes apart.
__device__ __forceinline__ uint32_t rope8_off(int i, int p) {
    return static_cast<uint32_t>((i >> 3) * 256 + p * 128 + (i & 7) * 16);
}

// D[tmem] (+)= A[tmem] x B[smem]^T, E4M3 operands, fp32 accumulate (one thread issues).
__device__ __forceinline__ void umma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, const uint32_t (&r)[4]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
                 "r"(r[2]), "r"(r[3])
                 : "memory");
}

// Four bf16 -> E4M3 codes of x / qs (one IEEE division each, round to nearest even, saturating).
__device__ __forceinline__ uint32_t quant4_e4m3(uint32_t lo, uint32_t hi, float qs) {
    const float v[4] = {bf16_lo(lo), bf16_hi(lo), bf16_lo(hi), bf16_hi(hi)};
    uint32_t w = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e)
        w |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(__fdiv_rn(v[e], qs), __NV_SATFINITE, __NV_E4M3)) << (8 * e);
    return w;
}

// Two E4M3 codes -> two bf16 (exact) with one conversion instruction.  The codes are widened to
// f16 (exact); every finite E4M3 value is a normal f16 whose low 7 mantissa bits are zero, so
// moving each half's exponent and mantissa right by 3 bits gives the bf16 bits of value * 2^-112
// (a normal bf16, smallest 2^-121), and one bf16 multiply by 2^112 (exact) restores the value.
// Zeros keep their sign.  The NaN codes 0x7F / 0xFF are never written by the latent store
// (saturating quantisation) and are not decoded faithfully here.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t two) {
    uint32_t h, d;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(two));
    const uint32_t t = ((h & 0x7fff7fffu) >> 3) | (h & 0x80008000u);
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(t), "r"(0x77807780u));   // 2^112 = bf16 0x7780
    return d;
}

__global__ void __launch_bounds__(kF8Threads, 1)
sparse_mla_fp8_kernel(const uint8_t* __restrict__ kv8, float k_scale, const uint16_t* __restrict__ q, float q_scale,
                      int64_t num_pages, const int32_t* __restrict__ block_table, int max_pages,
                      const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ cu_q, int B,
                      const int32_t* __restrict__ idx, int k, int H, float scale, int splits, uint16_t* __restrict__ out,
                      float* __restrict__ lse_out, float* __restrict__ part_o, float* __restrict__ part_lse, int32_t* err) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    unsigned char* base = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    unsigned char* kvs = base;                                                   // [5][codes 18 KB]
    unsigned char* vbs = kvs + kF8Stages * kF8CodeBytes;                         // [2][bf16 values 32 KB]
    float* xs = reinterpret_cast<float*>(vbs + kF8VBufs * kF8VBytes);            // [2][2 halves][8 quads][128 heads][4]
    Mla8Bars& bar = *reinterpret_cast<Mla8Bars*>(reinterpret_cast<unsigned char*>(xs) + 2 * kXBytes);

    const int split = blockIdx.y;
    const int r = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = row_request(cu_q, B, r);
    const int q0 = __ldg(cu_q + b);
    const int v = visible_len(__ldg(seq_lens + b), __ldg(cu_q + b + 1) - q0, r - q0);
    const int per_split = (k + splits - 1) / splits;
    const int e_begin = split * per_split;
    const int e_end = min(k, e_begin + per_split);
    const int ntiles = e_end > e_begin ? (e_end - e_begin + kKeysPerTile - 1) / kKeysPerTile : 0;
    const uint32_t crank = cluster_ctarank();
    const uint32_t peer = crank ^ 1u;
    const int half = static_cast<int>(crank);

    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar.q_full, kSoftmaxWarps);
        for (int s = 0; s < kF8Stages; ++s) {
            ptx::mbar_init(&bar.k_full[s], kProducerWarps * 32 + kProducerWarps);
            ptx::mbar_init(&bar.k_empty[s], 1 + kF8WidenWarps + kSoftmaxWarps);
        }
        for (int s = 0; s < kF8VBufs; ++s) {
            ptx::mbar_init(&bar.v_full[s], kF8WidenWarps);
            ptx::mbar_init(&bar.v_empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&bar.s_full[a], 1);
            ptx::mbar_init(&bar.s_free[a], 1);
            ptx::mbar_init(&bar.p_full[a], kSoftmaxWarps);
            ptx::mbar_init(&bar.x_full[a], 1);
            ptx::mbar_init(&bar.x_free[a], 1);
        }
        ptx::mbar_init(&bar.o_full, 1);
        for (int qd = 0; qd < 4; ++qd) ptx::mbar_init(&bar.pair[qd], 64);
        ptx::fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(&bar.tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    cluster_sync_all();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = bar.tmem_slot;
    const uint64_t deadline = ptx::wait_deadline();
    bool timed_out = false;
    const uint32_t kv_addr0 = ptx::smem_addr(kvs);

    if (warp >= kF8WidenWarp0) {
        // ---------------------------------------------------------------- widen warps
        // thread t owns key t of every tile: once the tile's codes landed and the PV that read
        // value buffer u % 2 before completed, its 256 value codes (16 swizzled 16-byte pieces in
        // two 128-byte chunks) become 32 bf16 pieces in the MN-major value layout
        const int key = (warp - kF8WidenWarp0) * 32 + lane;
        for (int u = 0; u < ntiles; ++u) {
            const int s = u % kF8Stages;
            const int vi = u % kF8VBufs;
            const bool ok = ptx::mbar_wait(&bar.k_full[s], (u / kF8Stages) & 1, deadline) &&
                            ptx::mbar_wait(&bar.v_empty[vi], ((u / kF8VBufs) & 1) ^ 1u, deadline);
            if (__any_sync(0xffffffffu, !ok)) { timed_out = true; break; }
            const unsigned char* sp = kvs + s * kF8CodeBytes + key * 128;
            unsigned char* vp = vbs + vi * kF8VBytes + key * 128;
#pragma unroll
            for (int p = 0; p < 16; ++p) {
                const uint4 c = *reinterpret_cast<const uint4*>(sp + (p >> 3) * kF8ChunkBytes + (((p & 7) ^ (key & 7)) << 4));
                uint4 lo, hi;
                lo.x = e4m3x2_to_bf16x2(static_cast<uint16_t>(c.x));
                lo.y = e4m3x2_to_bf16x2(static_cast<uint16_t>(c.x >> 16));
                lo.z = e4m3x2_to_bf16x2(static_cast<uint16_t>(c.y));
                lo.w = e4m3x2_to_bf16x2(static_cast<uint16_t>(c.y >> 16));
                hi.x = e4m3x2_to_bf16x2(static_cast<uint16_t>(c.z));
                hi.y = e4m3x2_to_bf16x2(static_cast<uint16_t>(c.z >> 16));
                hi.z = e4m3x2_to_bf16x2(static_cast<uint16_t>(c.w));
                hi.w = e4m3x2_to_bf16x2(static_cast<uint16_t>(c.w >> 16));
                // dims 16 p .. 16 p + 15: chunk p / 4 of 64 dims, pieces 2 (p % 4) and 2 (p % 4) + 1
                unsigned char* vrow = vp + (p >> 2) * kKvChunkBytes;
                *reinterpret_cast<uint4*>(vrow + (((2 * (p & 3)) ^ (key & 7)) << 4)) = lo;
                *reinterpret_cast<uint4*>(vrow + (((2 * (p & 3) + 1) ^ (key & 7)) << 4)) = hi;
            }
            ptx::fence_proxy_async_smem();   // the bf16 values are read by the tensor cores
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(&bar.v_full[vi]);
                ptx::mbar_arrive(&bar.k_empty[s]);
            }
        }
    } else if (warp >= kProducerWarp0) {
        // ---------------------------------------------------------------- producers
        const int pw = warp - kProducerWarp0;
        ptx::griddep_wait();
        const int my_entry = pw * kKeysPerProducer + lane;
        auto load_pos = [&](int tile) -> int {
            const int e = e_begin + tile * kKeysPerTile + my_entry;
            return (lane < kKeysPerProducer && tile < ntiles && e < e_end) ? __ldg(idx + static_cast<int64_t>(r) * k + e)
                                                                          : -1;
        };
        auto pos_ok = [&](int pos) -> bool { return pos >= 0 && pos < v && (pos >> 6) < max_pages; };
        auto load_page = [&](int pos) -> int {
            return pos_ok(pos) ? __ldg(block_table + static_cast<int64_t>(b) * max_pages + (pos >> 6)) : -1;
        };
        auto to_row = [&](int pos, int page) -> int {
            if (pos < 0) return -1;
            if (!pos_ok(pos)) { raise_error(err, DSA_DEVERR_INDEX_RANGE); return -1; }
            if (page < 0 || page >= num_pages) { raise_error(err, DSA_DEVERR_PAGE_RANGE); return -1; }
            return page * kPage + (pos & 63);
        };
        int pos1[kBatch], page1[kBatch], pos2[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) pos1[u] = load_pos(u);
#pragma unroll
        for (int u = 0; u < kBatch; ++u) page1[u] = load_page(pos1[u]);
#pragma unroll
        for (int u = 0; u < kBatch; ++u) pos2[u] = load_pos(kBatch + u);
        const uint8_t* kv_val = kv8 + half * kHalfDims + (lane & 15) * 16;
        const uint8_t* kv_rope = kv8 + kValueDim + half * kRopeHalf + (lane & 1) * 16;
        for (int t0 = 0; t0 < ntiles && !timed_out; t0 += kBatch) {
            int rows[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) rows[u] = to_row(pos1[u], page1[u]);
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                pos1[u] = pos2[u];
                page1[u] = load_page(pos2[u]);
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) pos2[u] = load_pos(t0 + 2 * kBatch + u);
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int t = t0 + u;
                if (t >= ntiles) break;
                const int s = t % kF8Stages;
                const uint32_t ph = (t / kF8Stages) & 1;
                const uint32_t vbits = __ballot_sync(0xffffffffu, rows[u] >= 0) & ((1u << kKeysPerProducer) - 1u);
                const int row_src = rows[u] >= 0 ? rows[u] : 0;
                if (lane == 0 && !ptx::mbar_wait(&bar.k_empty[s], ph ^ 1u, deadline)) timed_out = true;
                timed_out = __shfl_sync(0xffffffffu, timed_out ? 1 : 0, 0) != 0;
                if (timed_out) break;
                const uint32_t stage = kv_addr0 + s * kF8CodeBytes;
#pragma unroll
                for (int kq = 0; kq < kKeysPerProducer / 2; ++kq) {
                    const int kl = 2 * kq + (lane >> 4);
                    const int key = pw * kKeysPerProducer + kl;
                    const int64_t row = __shfl_sync(0xffffffffu, row_src, kl);
                    const int j = lane & 15;
                    cp_async_16(stage + (j >> 3) * kF8ChunkBytes + key * 128 + (((j & 7) ^ (key & 7)) << 4),
                                kv_val + row * kLatentDim);
                }
                {
                    const int kl = lane >> 1;   // two 16-byte rope pieces per key
                    const int key = pw * kKeysPerProducer + kl;
                    const int64_t row = __shfl_sync(0xffffffffu, row_src, kl & (kKeysPerProducer - 1));
                    if (kl < kKeysPerProducer)
                        cp_async_16(stage + 2 * kF8ChunkBytes + rope8_off(key, lane & 1), kv_rope + row * kLatentDim);
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
                cp_async_arrive_noinc(&bar.k_full[s]);
                if (lane == 0) {
                    bar.valid[s][pw] = vbits;
                    ptx::mbar_arrive(&bar.k_full[s]);
                }
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = ptx::instr_desc(0, 0, kHeadsPerCta, kKeysPerTile);   // E4M3 x E4M3
            constexpr uint32_t idesc_pv = ptx::instr_desc(1, 1, kHeadsPerCta, kHalfDims) | (1u << 16);
            bool ok = ptx::mbar_wait(&bar.q_full, 0, deadline);
            int tq = 0, tp = 0;
            while (ok && tp < ntiles) {
                bool issued = false;
                if (tq < ntiles && ptx::mbar_test_wait(&bar.k_full[tq % kF8Stages], (tq / kF8Stages) & 1) &&
                    ptx::mbar_test_wait(&bar.s_free[tq & 1], ((tq >> 1) & 1) ^ 1u)) {
                    ptx::fence_proxy_async_smem();
                    ptx::tc_fence_after_sync();
                    const uint32_t kb = kv_addr0 + (tq % kF8Stages) * kF8CodeBytes;
                    const uint32_t d = tmem + kTmemS + (tq & 1) * kKeysPerTile;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t db = make_desc(kb + (kk >> 2) * kF8ChunkBytes + (kk & 3) * 32, 16, 1024, kLayoutSw128);
                        umma_f8_ts(d, tmem + kTmemQ + kk * 8, db, idesc_qk, kk != 0 ? 1u : 0u);
                    }
                    umma_f8_ts(d, tmem + kF8TmemQRope, make_desc(kb + 2 * kF8ChunkBytes, 128, 256, kLayoutNone), idesc_qk,
                               1u);
                    ptx::umma_commit(&bar.s_full[tq & 1]);
                    ptx::umma_commit(&bar.k_empty[tq % kF8Stages]);
                    ++tq;
                    issued = true;
                }
                if (tp < tq && ptx::mbar_test_wait(&bar.p_full[tp & 1], (tp >> 1) & 1) &&
                    ptx::mbar_test_wait(&bar.v_full[tp % kF8VBufs], (tp / kF8VBufs) & 1)) {
                    ptx::tc_fence_after_sync();
                    const uint32_t vb = ptx::smem_addr(vbs) + (tp % kF8VBufs) * kF8VBytes;
                    const uint32_t pa = tmem + kTmemS + (tp & 1) * kKeysPerTile;
#pragma unroll
                    for (int ks = 0; ks < kKeysPerTile / 16; ++ks) {
                        const uint64_t db = make_desc(vb + ks * 16 * 128, kKvChunkBytes, 1024, kLayoutSw128);
                        umma_f16_ts(tmem, pa + ks * 8, db, idesc_pv, (tp | ks) != 0 ? 1u : 0u);
                    }
                    ptx::umma_commit(&bar.v_empty[tp % kF8VBufs]);
                    ptx::umma_commit(&bar.s_free[tp & 1]);
                    ++tp;
                    issued = true;
                }
                if (!issued && static_cast<uint64_t>(clock64()) > deadline) ok = false;
            }
            if (ok && ntiles > 0) ptx::umma_commit(&bar.o_full);
            if (!ok) timed_out = true;
        }
    } else {
        // ---------------------------------------------------------------- query, softmax, epilogue
        const int quad = warp & 3;
        const int kh = warp >> 2;
        const int head = quad * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        {
            // the query's codes (x / q_scale): value dims 128 kh .. + 127 of this CTA -> columns
            // 384 + 32 kh .., rope dims 16 kh .. + 15 of this CTA -> columns 448 + 4 kh ..
            const uint4* src = reinterpret_cast<const uint4*>(q + (static_cast<int64_t>(r) * H + head) * kLatentDim);
            const bool live = head < H;
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint4 raw = live ? __ldg(src + (half * kHalfDims + kh * 128) / 8 + i) : make_uint4(0u, 0u, 0u, 0u);
                w[2 * i] = quant4_e4m3(raw.x, raw.y, q_scale);
                w[2 * i + 1] = quant4_e4m3(raw.z, raw.w, q_scale);
            }
            tmem_st_32x32b_x32(tmem + lane_base + kTmemQ + 32 * kh, w);
            uint32_t wr[4];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const uint4 raw =
                    live ? __ldg(src + (kValueDim + half * kRopeHalf + kh * 16) / 8 + i) : make_uint4(0u, 0u, 0u, 0u);
                wr[2 * i] = quant4_e4m3(raw.x, raw.y, q_scale);
                wr[2 * i + 1] = quant4_e4m3(raw.z, raw.w, q_scale);
            }
            tmem_st_32x32b_x4(tmem + lane_base + kF8TmemQRope + 4 * kh, wr);
            tmem_wait_st();
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bar.q_full);
        }
        const float cscale = scale * q_scale * k_scale * kLog2e;
        const uint32_t x_peer0 = map_to_rank(ptx::smem_addr(xs), peer) + (kh * 8 * kHeadsPerCta + head) * 16;
        float m_run = -INFINITY, l_run = 0.0f;
        uint32_t sr[32];
        uint32_t vbits_next = 0;   // valid bits of the fetched tile, read before its code stage is released
        auto fetch_send = [&](int u) -> bool {
            const int su = u % kF8Stages;
            const int bu = u & 1;
            const uint32_t pu = (u >> 1) & 1;
            if (threadIdx.x == 0) ptx::mbar_arrive_expect_tx(&bar.x_full[bu], kXBytes);
            if (!ptx::mbar_wait(&bar.s_full[bu], pu, deadline)) return false;
            if (!ptx::mbar_wait(&bar.k_full[su], (u / kF8Stages) & 1, deadline)) return false;
            vbits_next = half_valid_bits(bar.valid[su], kh);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bar.k_empty[su]);
            ptx::tc_fence_after_sync();
            ptx::tmem_ld_32x32b_x32(tmem + lane_base + kTmemS + bu * kKeysPerTile + kh * 32, sr);
            ptx::tmem_wait_ld();
            if (u >= 2 && !ptx::mbar_wait(&bar.x_free[bu], pu ^ 1u, deadline)) return false;
            if (threadIdx.x == 0) ptx::mbar_arrive_expect_tx(&bar.x_free[bu], kSoftmaxWarps * 4);
            const uint32_t xp = x_peer0 + bu * kXBytes;
            const uint32_t xf_peer = map_to_rank(ptx::smem_addr(&bar.x_full[bu]), peer);
#pragma unroll
            for (int kq = 0; kq < 8; ++kq)
                st_async_v4(xp + kq * (kHeadsPerCta * 16), __uint_as_float(sr[4 * kq]), __uint_as_float(sr[4 * kq + 1]),
                            __uint_as_float(sr[4 * kq + 2]), __uint_as_float(sr[4 * kq + 3]), xf_peer);
            return true;
        };
        if (ntiles > 0 && !fetch_send(0)) timed_out = true;
        for (int t = 0; t < ntiles && !timed_out; ++t) {
            const int bb = t & 1;
            const uint32_t ph = (t >> 1) & 1;
            const uint32_t vbits = vbits_next;
            if (!ptx::mbar_wait(&bar.x_full[bb], ph, deadline)) { timed_out = true; break; }
            {
                const float* xr = xs + bb * (kXBytes / 4) + (kh * 8 * kHeadsPerCta + head) * 4;
#pragma unroll
                for (int kq = 0; kq < 8; ++kq) {
                    const float4 o = *reinterpret_cast<const float4*>(xr + kq * (kHeadsPerCta * 4));
                    sr[4 * kq + 0] = __float_as_uint(__uint_as_float(sr[4 * kq + 0]) + o.x);
                    sr[4 * kq + 1] = __float_as_uint(__uint_as_float(sr[4 * kq + 1]) + o.y);
                    sr[4 * kq + 2] = __float_as_uint(__uint_as_float(sr[4 * kq + 2]) + o.z);
                    sr[4 * kq + 3] = __float_as_uint(__uint_as_float(sr[4 * kq + 3]) + o.w);
                }
            }
            __syncwarp();
            if (lane == 0)
                st_async_b32(map_to_rank(ptx::smem_addr(&bar.x_sink[bb][warp]), peer), 1u,
                             map_to_rank(ptx::smem_addr(&bar.x_free[bb]), peer));
            float tmax = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float sv = ((vbits >> i) & 1u) ? __uint_as_float(sr[i]) * cscale : -INFINITY;
                sr[i] = __float_as_uint(sv);
                tmax = fmaxf(tmax, sv);
            }
            bar.tmax[bb][kh][head] = tmax;
            ptx::mbar_arrive(&bar.pair[quad]);
            if (!ptx::mbar_wait(&bar.pair[quad], t & 1, deadline)) { timed_out = true; break; }
            tmax = fmaxf(tmax, bar.tmax[bb][kh ^ 1][head]);
            const bool grow = tmax > m_run + kRescaleThreshold || (m_run == -INFINITY && tmax > -INFINITY);
            const float m_new = grow ? tmax : m_run;
            const float alpha = grow ? ((m_run == -INFINITY) ? 0.0f : exp2f(m_run - m_new)) : 1.0f;
            if (t > 0 && __any_sync(0xffffffffu, grow)) {
                if (!ptx::mbar_wait(&bar.s_free[(t - 1) & 1], ((t - 1) >> 1) & 1, deadline)) { timed_out = true; break; }
                ptx::tc_fence_after_sync();
#pragma unroll 1
                for (int cc = kh * 128; cc < kh * 128 + 128; cc += 32) {
                    uint32_t o[32];
                    ptx::tmem_ld_32x32b_x32(tmem + lane_base + cc, o);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st_32x32b_x32(tmem + lane_base + cc, o);
                }
                tmem_wait_st();
            }
            l_run *= alpha;
            m_run = m_new;
            float psum = 0.0f;
            uint32_t pk[16];
            const bool any = m_run != -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const float p0 = any ? fast_exp2(__uint_as_float(sr[i]) - m_run) : 0.0f;
                const float p1 = any ? fast_exp2(__uint_as_float(sr[i + 1]) - m_run) : 0.0f;
                psum += p0 + p1;
                pk[i / 2] = pack_bf16x2(p0, p1);
            }
            l_run += psum;
            tmem_st_32x32b_x16(tmem + lane_base + kTmemS + bb * kKeysPerTile + kh * 16, pk);
            tmem_wait_st();
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bar.p_full[bb]);
            if (t + 1 < ntiles && !fetch_send(t + 1)) { timed_out = true; break; }
        }
        if (!timed_out) {
            for (int t = (ntiles >= 2 ? ntiles - 2 : 0); t < ntiles; ++t)
                if (!ptx::mbar_wait(&bar.x_free[t & 1], (t >> 1) & 1, deadline)) { timed_out = true; break; }
        }
        bar.lsum[kh][head] = l_run;
        ptx::mbar_arrive(&bar.pair[quad]);
        if (!timed_out && !ptx::mbar_wait(&bar.pair[quad], ntiles & 1, deadline)) timed_out = true;
        const float l_tot = l_run + bar.lsum[kh ^ 1][head];
        bool have_o = ntiles > 0 && !timed_out;
        if (have_o && !ptx::mbar_wait(&bar.o_full, 0, deadline)) { timed_out = true; have_o = false; }
        ptx::tc_fence_after_sync();
        const float inv_l = l_tot > 0.0f ? k_scale / l_tot : 0.0f;   // the values are codes times k_scale
        const float lse = l_tot > 0.0f ? (m_run + log2f(l_tot)) / kLog2e : -INFINITY;
        const bool write_head = head < H;
        const int64_t rh = static_cast<int64_t>(r) * H + head;
        if (splits == 1) {
            uint16_t* dst = out + rh * kValueDim + half * kHalfDims;
#pragma unroll 1
            for (int cc = kh * 128; cc < kh * 128 + 128; cc += 32) {
                uint32_t o[32];
                if (have_o) {
                    ptx::tmem_ld_32x32b_x32(tmem + lane_base + cc, o);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                if (write_head) {
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        uint4 wv;
                        wv.x = pack_bf16x2(__uint_as_float(o[i]) * inv_l, __uint_as_float(o[i + 1]) * inv_l);
                        wv.y = pack_bf16x2(__uint_as_float(o[i + 2]) * inv_l, __uint_as_float(o[i + 3]) * inv_l);
                        wv.z = pack_bf16x2(__uint_as_float(o[i + 4]) * inv_l, __uint_as_float(o[i + 5]) * inv_l);
                        wv.w = pack_bf16x2(__uint_as_float(o[i + 6]) * inv_l, __uint_as_float(o[i + 7]) * inv_l);
                        *reinterpret_cast<uint4*>(dst + cc + i) = wv;
                    }
                }
            }
            if (write_head && half == 0 && kh == 0 && lse_out != nullptr) lse_out[rh] = lse;
        } else {
            float* dst = part_o + (rh * splits + split) * kValueDim + half * kHalfDims;
#pragma unroll 1
            for (int cc = kh * 128; cc < kh * 128 + 128; cc += 32) {
                uint32_t o[32];
                if (have_o) {
                    ptx::tmem_ld_32x32b_x32(tmem + lane_base + cc, o);
                    ptx::tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                if (write_head) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4*>(dst + cc + i) =
                            make_float4(__uint_as_float(o[i]) * inv_l, __uint_as_float(o[i + 1]) * inv_l,
                                        __uint_as_float(o[i + 2]) * inv_l, __uint_as_float(o[i + 3]) * inv_l);
                }
            }
            if (write_head && half == 0 && kh == 0) part_lse[rh * splits + split] = lse;
        }
    }
    if (timed_out) raise_error(err, DSA_DEVERR_TIMEOUT);
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
    cluster_sync_all();
}

__global__ void __launch_bounds__(128)
sparse_mla_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse, int splits,
                          uint16_t* __restrict__ out, float* __restrict__ lse, const float* __restrict__ sinks,
                          int H) {
    const int64_t rh = blockIdx.x;   // row * H + head
    const float* pl = part_lse + rh * splits;
    const float sink = sinks != nullptr ? __ldg(sinks + rh % H) : -INFINITY;   // joins the denominator
    float m = sink;
    for (int j = 0; j < splits; ++j) m = fmaxf(m, __ldg(pl + j));
    float wsum = (sink == -INFINITY || m == -INFINITY) ? 0.0f : expf(sink - m);
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
        uint2 packed;
        packed.x = pack_bf16x2(acc.x, acc.y);
        packed.y = pack_bf16x2(acc.z, acc.w);
        reinterpret_cast<uint2*>(out + rh * kValueDim + d)[0] = packed;
    }
    if (lse != nullptr && threadIdx.x == 0) lse[rh] = (m == -INFINITY) ? -INFINITY : m + logf(wsum);
}

// Splits of the k entries per row: the largest power of two (<= 8) for which the (row, split,
// half) grid still fits one wave of one CTA per SM and every split keeps >= 256 entries.
int mla_splits(int T, int k) {
    const int sms = device_sm_count();
    int s = 1;
    while (2 * T * (2 * s) <= sms && k / (2 * s) >= 256 && s < 8) s *= 2;
    return s;
}

}  // namespace
}  // namespace dsa

extern "C" size_t dsa_sparse_mla_workspace_size(int32_t T, int32_t H, int32_t k) {
    if (T <= 0 || H <= 0 || k <= 0) return 0;
    const size_t splits = static_cast<size_t>(dsa::mla_splits(T, k));
    if (splits == 1) return 0;
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
    if (num_pages < 1) return DSA_ERR_INVALID_ARG;
    if (B == 0 || !q_bf16 || !kv_pool || !block_table || !seq_lens || !cu_q || !idx || !out_bf16) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_bf16) || !aligned16(kv_pool) || !aligned16(out_bf16)) return DSA_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || T > 65535) return DSA_ERR_INVALID_ARG;
    if (num_pages * kPage >= 0x7fffffffLL || static_cast<int64_t>(T) * H >= 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
    const size_t ws_need = dsa_sparse_mla_workspace_size(T, H, k);
    if (ws_need > 0 && (workspace == nullptr || !aligned16(workspace) || workspace_bytes < ws_need))
        return DSA_ERR_INVALID_ARG;
    const int splits = mla_splits(T, k);
    float* part_o = static_cast<float*>(workspace);
    float* part_lse = splits > 1 ? part_o + static_cast<size_t>(T) * H * splits * kValueDim : nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaFuncSetAttribute(sparse_mla_umma_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kMlaSmemBytes)) != cudaSuccess)
        return DSA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, splits, T);   // x: the two ranks of a (row, split) = one cluster
    cfg.blockDim = dim3(kMlaThreads, 1, 1);
    cfg.dynamicSmemBytes = kMlaSmemBytes;
    cfg.stream = s;
    // clusters of 2; a programmatic dependent of the previous kernel on the stream (top-k): barrier
    // setup, TMEM allocation and the query load overlap it, the index reads wait for it
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, sparse_mla_umma_kernel<false>, static_cast<const uint16_t*>(kv_pool),
                           static_cast<const uint16_t*>(q_bf16), num_pages, block_table, static_cast<int>(max_pages),
                           seq_lens, cu_q, static_cast<int>(B), idx, static_cast<int>(k), static_cast<int>(H), scale,
                           splits, 0, splits, 0, static_cast<uint16_t*>(out_bf16), lse,
                           splits > 1 ? part_o : nullptr, part_lse, dev_err, TwoSrc{}) != cudaSuccess)
        return DSA_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
    if (splits > 1) {
        sparse_mla_combine_kernel<<<static_cast<unsigned>(static_cast<int64_t>(T) * H), 128, 0, s>>>(
            part_o, part_lse, splits, static_cast<uint16_t*>(out_bf16), lse, nullptr, H);
        if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

extern "C" dsa_status dsa_sparse_mla_decode_fp8(const void* q_bf16, float q_scale, const uint8_t* kv_pool_fp8,
                                                float k_scale, int64_t num_pages, const int32_t* block_table,
                                                int32_t max_pages, const int32_t* seq_lens, const int32_t* cu_q,
                                                int32_t B, const int32_t* idx, int32_t k, int32_t T, int32_t H,
                                                float scale, void* out_bf16, float* lse, void* workspace,
                                                size_t workspace_bytes, int32_t* dev_err, void* stream) {
    using namespace dsa;
    if (k < 1 || k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
    if (H != 16 && H != 32 && H != 64 && H != 128) return DSA_ERR_UNSUPPORTED;
    if (T < 0 || B < 0 || max_pages < 0 || num_pages < 0) return DSA_ERR_INVALID_ARG;
    if (T == 0) return DSA_OK;
    if (num_pages < 1) return DSA_ERR_INVALID_ARG;
    if (B == 0 || !q_bf16 || !kv_pool_fp8 || !block_table || !seq_lens || !cu_q || !idx || !out_bf16)
        return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_bf16) || !aligned16(kv_pool_fp8) || !aligned16(out_bf16)) return DSA_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !(q_scale > 0.0f) || !(k_scale > 0.0f) || !(q_scale < INFINITY) || !(k_scale < INFINITY) ||
        T > 65535)
        return DSA_ERR_INVALID_ARG;
    if (num_pages * kPage >= 0x7fffffffLL || static_cast<int64_t>(T) * H >= 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
    const size_t ws_need = dsa_sparse_mla_workspace_size(T, H, k);
    if (ws_need > 0 && (workspace == nullptr || !aligned16(workspace) || workspace_bytes < ws_need))
        return DSA_ERR_INVALID_ARG;
    const int splits = mla_splits(T, k);
    float* part_o = static_cast<float*>(workspace);
    float* part_lse = splits > 1 ? part_o + static_cast<size_t>(T) * H * splits * kValueDim : nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaFuncSetAttribute(sparse_mla_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kF8SmemBytes)) != cudaSuccess)
        return DSA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, splits, T);
    cfg.blockDim = dim3(kF8Threads, 1, 1);
    cfg.dynamicSmemBytes = kF8SmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, sparse_mla_fp8_kernel, kv_pool_fp8, k_scale, static_cast<const uint16_t*>(q_bf16),
                           q_scale, num_pages, block_table, static_cast<int>(max_pages), seq_lens, cu_q,
                           static_cast<int>(B), idx, static_cast<int>(k), static_cast<int>(H), scale, splits,
                           static_cast<uint16_t*>(out_bf16), lse, part_o, part_lse, dev_err) != cudaSuccess)
        return DSA_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
    if (splits > 1) {
        sparse_mla_combine_kernel<<<static_cast<unsigned>(static_cast<int64_t>(T) * H), 128, 0, s>>>(
            part_o, part_lse, splits, static_cast<uint16_t*>(out_bf16), lse, nullptr, H);
        if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
    }
    return DSA_OK;
}

extern "C" size_t dsa_sparse_attn_swa_cmp_workspace_size(int32_t T, int32_t H, int32_t window, int32_t k) {
    if (T <= 0 || H <= 0 || window <= 0 || k <= 0) return 0;
    const size_t splits = static_cast<size_t>(dsa::mla_splits(T, window + k));
    if (splits == 1) return 0;
    return static_cast<size_t>(T) * H * splits * (dsa::kValueDim + 1) * sizeof(float);
}

extern "C" dsa_status dsa_sparse_attn_swa_cmp(const void* q_bf16, const void* swa_kv, int64_t swa_num_pages,
                                              const int32_t* swa_block_table, int32_t swa_max_pages, const void* cmp_kv,
                                              int64_t cmp_num_pages, const int32_t* cmp_block_table,
                                              int32_t cmp_max_pages, const int32_t* seq_lens, const int32_t* cu_q,
                                              int32_t B, const int32_t* cmp_idx, int32_t k, int32_t window,
                                              int32_t cmp_ratio, const float* sinks, int32_t T, int32_t H, float scale,
                                              void* out_bf16, float* lse, void* workspace, size_t workspace_bytes,
                                              int32_t* dev_err, void* stream) {
    using namespace dsa;
    if (k < 1 || k > DSA_MAX_TOPK || window < 1 || window > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
    if (H != 16 && H != 32 && H != 64 && H != 128) return DSA_ERR_UNSUPPORTED;
    int shift = 0;
    while (shift < 8 && (1 << shift) < cmp_ratio) ++shift;
    if (cmp_ratio < 1 || (1 << shift) != cmp_ratio || shift > 7) return DSA_ERR_UNSUPPORTED;
    if (T < 0 || B < 0 || swa_max_pages < 0 || cmp_max_pages < 0 || swa_num_pages < 0 || cmp_num_pages < 0)
        return DSA_ERR_INVALID_ARG;
    if (T == 0) return DSA_OK;
    if (swa_num_pages < 1 || cmp_num_pages < 1 || B == 0) return DSA_ERR_INVALID_ARG;
    if (!q_bf16 || !swa_kv || !swa_block_table || !cmp_kv || !cmp_block_table || !seq_lens || !cu_q || !cmp_idx ||
        !sinks || !out_bf16)
        return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_bf16) || !aligned16(swa_kv) || !aligned16(cmp_kv) || !aligned16(out_bf16)) return DSA_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || T > 65535) return DSA_ERR_INVALID_ARG;
    // rows of both caches carry their source in bit 30
    if (swa_num_pages * kPage >= kSrc2 || cmp_num_pages * kPage >= kSrc2 || static_cast<int64_t>(T) * H >= 0x7fffffffLL)
        return DSA_ERR_UNSUPPORTED;
    const int ktot = window + k;
    const size_t ws_need = dsa_sparse_attn_swa_cmp_workspace_size(T, H, window, k);
    if (ws_need > 0 && (workspace == nullptr || !aligned16(workspace) || workspace_bytes < ws_need))
        return DSA_ERR_INVALID_ARG;
    const int splits = mla_splits(T, ktot);
    float* part_o = static_cast<float*>(workspace);
    float* part_lse = splits > 1 ? part_o + static_cast<size_t>(T) * H * splits * kValueDim : nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaFuncSetAttribute(sparse_mla_umma_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kMlaSmemBytes)) != cudaSuccess)
        return DSA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, splits, T);
    cfg.blockDim = dim3(kMlaThreads, 1, 1);
    cfg.dynamicSmemBytes = kMlaSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const TwoSrc ts{static_cast<const uint16_t*>(cmp_kv), cmp_num_pages, cmp_block_table, static_cast<int>(cmp_max_pages),
                    shift, cmp_idx, static_cast<int>(k), static_cast<int>(window), sinks};
    if (cudaLaunchKernelEx(&cfg, sparse_mla_umma_kernel<true>, static_cast<const uint16_t*>(swa_kv),
                           static_cast<const uint16_t*>(q_bf16), swa_num_pages, swa_block_table,
                           static_cast<int>(swa_max_pages), seq_lens, cu_q, static_cast<int>(B),
                           static_cast<const int32_t*>(nullptr), ktot, static_cast<int>(H), scale, splits, 0, splits, 0,
                           static_cast<uint16_t*>(out_bf16), lse, splits > 1 ? part_o : nullptr, part_lse, dev_err,
                           ts) != cudaSuccess)
        return DSA_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
    if (splits > 1) {
        sparse_mla_combine_kernel<<<static_cast<unsigned>(static_cast<int64_t>(T) * H), 128, 0, s>>>(
            part_o, part_lse, splits, static_cast<uint16_t*>(out_bf16), lse, sinks, H);
        if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
    }
    return DSA_OK;
}
