// topk.cu -- per-row top-k of the indexer logits, deterministic.
//
// Follows sglang dsa_indexer.py, forward_indexer (topk(min(topk, seq_len)) of the row's logits,
// then -1 padding) and Indexer._get_topk_paged (topk_transform over the paged logits).  The kept
// set is the k largest of I[r, 0:v_r) with ties broken toward the lower index; it is written in
// ascending index order and padded with -1.
//
// One 1024-thread CTA per row.  Logits map to order-preserving 32-bit keys (larger float ->
// larger key; -0 and +0 share a key; NaN gets the smallest key).  A 3-digit MSB-first radix
// select (11 + 11 + 10 bits, histograms in shared memory) finds the exact k-th largest key K and
// how many of the keys equal to K are kept; a final pass in index order writes every index with
// key > K plus the first (by index) of those equal to K.  The row is read 4 times, from L2.
#include "dsa_common.cuh"
#include "sm100_ptx.cuh"

namespace dsa {
namespace {

constexpr int kTopkThreads = 1024;
constexpr int kWarps = kTopkThreads / 32;

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;   // NaN: never preferred
    if (u == 0x80000000u) u = 0u;                      // -0 == +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Positions whose logit counts as +inf (the forced initial and local tokens): [0, init_end) and
// [local_begin, v).  With nothing forced, init_end = 0 and local_begin = v.
// ON = false (nothing forced) compiles the test away.
template <bool ON>
struct Forced {
    int init_end, local_begin;
    __device__ __forceinline__ uint32_t operator()(int s, uint32_t key) const {
        if (!ON) return key;
        return (s < init_end || s >= local_begin) ? 0xFF800000u : key;   // order key of +inf
    }
};
template <bool ON>
__device__ __forceinline__ Forced<ON> make_forced(int v, int n_init, int n_local) {
    Forced<ON> f;
    f.init_end = min(n_init, v);
    f.local_begin = max(0, v - n_local);
    return f;
}

// Block-wide inclusive scan of one uint32 per thread; also returns the block total.
__device__ __forceinline__ uint32_t block_inclusive_scan(uint32_t v, uint32_t* warp_tot, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += o;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        uint32_t t = warp_tot[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t o = __shfl_up_sync(0xffffffffu, t, d);
            if (lane >= d) t += o;
        }
        warp_tot[lane] = t;   // inclusive prefix of warp totals
    }
    __syncthreads();
    const uint32_t before = warp == 0 ? 0u : warp_tot[warp - 1];
    *total = warp_tot[kWarps - 1];
    __syncthreads();   // warp_tot may be reused by the caller's next scan
    return v + before;
}

struct TopkSmem {
    uint32_t hist[2048];
    uint32_t warp_tot[kWarps];
    uint32_t sel_digit;
    uint32_t sel_remaining;
};

// Given a histogram over `bins` digits (bins = 2048 or 1024), find the digit d such that
// (# keys with digit > d) < need <= (# keys with digit >= d); store d and
// need - (# keys with digit > d).
__device__ void select_digit(TopkSmem& sm, int bins, uint32_t need) {
    // thread t covers the digits (from the top) bins-1-2t and bins-2-2t (bins/1024 digits each)
    const int per = bins / kTopkThreads;   // 2 or 1
    uint32_t local = 0;
    for (int i = 0; i < per; ++i) local += sm.hist[bins - 1 - (threadIdx.x * per + i)];
    uint32_t total;
    const uint32_t incl = block_inclusive_scan(local, sm.warp_tot, &total);
    uint32_t above = incl - local;   // keys with digit greater than this thread's first digit
    for (int i = 0; i < per; ++i) {
        const int d = bins - 1 - (threadIdx.x * per + i);
        const uint32_t c = sm.hist[d];
        if (above < need && need <= above + c) {
            sm.sel_digit = static_cast<uint32_t>(d);
            sm.sel_remaining = need - above;
        }
        above += c;
    }
    __syncthreads();
}

template <bool FORCED>
__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(const float* __restrict__ logits, int64_t ld, const int32_t* __restrict__ seq_lens,
            const int32_t* __restrict__ cu_q, int B, int row_begin, int k, int n_init, int n_local, int cmp_shift,
            int32_t* __restrict__ idx) {
    __shared__ TopkSmem sm;
    // launched as a programmatic dependent of the logits kernel: the row's request is looked up in
    // the inputs (not written by that kernel) while it finishes, the logits are read after the wait
    ptx::griddep_launch_dependents();
    const int rl = blockIdx.x;                  // local row
    const int r = row_begin + rl;
    const int b = row_request(cu_q, B, r);
    const int q0 = __ldg(cu_q + b);
    int v = visible_len(__ldg(seq_lens + b), __ldg(cu_q + b + 1) - q0, r - q0) >> cmp_shift;
    ptx::griddep_wait();
    if (v > ld) v = static_cast<int>(ld);       // never read past the row
    const float* row = logits + static_cast<int64_t>(rl) * ld;
    const Forced<FORCED> F = make_forced<FORCED>(v, n_init, n_local);
    int32_t* out = idx + static_cast<int64_t>(rl) * k;

    if (v <= k) {   // short row: keep everything in index order
        for (int j = threadIdx.x; j < k; j += kTopkThreads) out[j] = j < v ? j : -1;
        return;
    }

    // ---- radix select of the k-th largest key
    uint32_t prefix = 0, need = static_cast<uint32_t>(k);
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    for (int pass = 0; pass < 3; ++pass) {
        const int bins = 1 << widths[pass];
        for (int i = threadIdx.x; i < bins; i += kTopkThreads) sm.hist[i] = 0;
        __syncthreads();
        const int hi_shift = shifts[pass] + widths[pass];   // bits above this digit must match
        for (int s = threadIdx.x; s < v; s += kTopkThreads) {
            const uint32_t key = F(s, order_key(__ldg(row + s)));
            const bool match = hi_shift >= 32 || (key >> hi_shift) == (prefix >> hi_shift);
            if (match) atomicAdd(&sm.hist[(key >> shifts[pass]) & (bins - 1)], 1u);
        }
        __syncthreads();
        select_digit(sm, bins, need);
        prefix |= sm.sel_digit << shifts[pass];
        need = sm.sel_remaining;
        __syncthreads();
    }
    const uint32_t kth = prefix;
    const uint32_t take_equal = need;           // keys equal to kth that are kept (lowest indices)

    // ---- index-ordered compaction
    uint32_t gt_base = 0, eq_base = 0;
    for (int base = 0; base < v; base += kTopkThreads) {
        const int s = base + threadIdx.x;
        uint32_t key = 0;
        bool valid = s < v;
        if (valid) key = F(s, order_key(__ldg(row + s)));
        const uint32_t gt = (valid && key > kth) ? 1u : 0u;
        const uint32_t eq = (valid && key == kth) ? 1u : 0u;
        uint32_t total;
        const uint32_t incl = block_inclusive_scan((gt << 16) | eq, sm.warp_tot, &total);
        const uint32_t excl = incl - ((gt << 16) | eq);
        const uint32_t gt_before = gt_base + (excl >> 16);
        const uint32_t eq_before = eq_base + (excl & 0xffffu);
        if (gt) out[gt_before + min(eq_before, take_equal)] = s;
        else if (eq && eq_before < take_equal) out[gt_before + eq_before] = s;
        gt_base += total >> 16;
        eq_base += total & 0xffffu;
    }
}

// ---------------------------------------------------------------------------------------------
// Two-read kernel for rows of up to kMaxBitmapWords * 32 keys.  Read 1: histogram of the top 12
// key bits.  Read 2: keys in bins above the threshold bin are marked in a shared-memory bitmap;
// keys in the threshold bin are collected (key, index) as candidates in shared memory.  The low 20
// bits are then resolved on the candidates (two 10-bit digits), the selected candidates marked,
// and a scan over the bitmap words writes the indices in ascending order.  If the threshold bin
// holds more candidates than fit, the low digits are resolved by re-reading the row instead.
// ---------------------------------------------------------------------------------------------
constexpr int kTopBins = 4096;                 // top 12 bits of the key
constexpr int kMaxBitmapWords = 4096;          // rows up to 131072 keys
constexpr int kCandidateCap = 8192;

struct BitmapSmem {
    uint32_t hist[kTopBins];
    uint32_t warp_tot[kWarps];
    uint32_t warp_tot2[kWarps];
    uint32_t sel_digit;
    uint32_t sel_remaining;
    uint32_t cand_count;
    int32_t row_v;
};
static_assert(sizeof(BitmapSmem) % 16 == 0, "16-byte alignment of the buffers after BitmapSmem");

// Visible length of global row r, looked up by all threads at once: thread t < B tests whether r
// falls in request t (one round of independent loads instead of a chain of dependent ones).
__device__ __forceinline__ int locate_visible(const int32_t* __restrict__ cu_q, const int32_t* __restrict__ seq_lens,
                                              int B, int r, int cmp_shift, BitmapSmem& sm) {
    if (threadIdx.x == 0) sm.row_v = 0;
    __syncthreads();
    for (int t = threadIdx.x; t < B; t += kTopkThreads) {
        const int a = __ldg(cu_q + t), e = __ldg(cu_q + t + 1), L = __ldg(seq_lens + t);
        if (a <= r && r < e) sm.row_v = visible_len(L, e - a, r - a) >> cmp_shift;
    }
    __syncthreads();
    return sm.row_v;
}

// Block-wide exclusive scans of two uint32 per thread at once (one set of barriers); also the
// block totals.
__device__ __forceinline__ void block_exclusive_scan2(uint32_t& a, uint32_t& b, BitmapSmem& sm, uint32_t* tot_a,
                                                      uint32_t* tot_b) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t ia = a, ib = b;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t oa = __shfl_up_sync(0xffffffffu, ia, d), ob = __shfl_up_sync(0xffffffffu, ib, d);
        if (lane >= d) { ia += oa; ib += ob; }
    }
    if (lane == 31) { sm.warp_tot[warp] = ia; sm.warp_tot2[warp] = ib; }
    __syncthreads();
    if (warp == 0) {
        uint32_t ta = sm.warp_tot[lane], tb = sm.warp_tot2[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t oa = __shfl_up_sync(0xffffffffu, ta, d), ob = __shfl_up_sync(0xffffffffu, tb, d);
            if (lane >= d) { ta += oa; tb += ob; }
        }
        sm.warp_tot[lane] = ta;
        sm.warp_tot2[lane] = tb;
    }
    __syncthreads();
    const uint32_t ba = warp == 0 ? 0u : sm.warp_tot[warp - 1], bb = warp == 0 ? 0u : sm.warp_tot2[warp - 1];
    *tot_a = sm.warp_tot[kWarps - 1];
    *tot_b = sm.warp_tot2[kWarps - 1];
    a = ia - a + ba;
    b = ib - b + bb;
    __syncthreads();
}

// Digit d (from the top) of `bins` histogram bins such that (# keys with digit > d) < need <=
// (# keys with digit >= d); stores d and need - (# keys with digit > d).  bins: 1024 or 4096.
__device__ void select_bin(uint32_t* hist, BitmapSmem& sm, int bins, uint32_t need) {
    const int per = bins / kTopkThreads;
    uint32_t local = 0;
    for (int i = 0; i < per; ++i) local += hist[bins - 1 - (threadIdx.x * per + i)];
    uint32_t total;
    const uint32_t incl = block_inclusive_scan(local, sm.warp_tot, &total);
    uint32_t above = incl - local;
    for (int i = 0; i < per; ++i) {
        const int d = bins - 1 - (threadIdx.x * per + i);
        const uint32_t c = hist[d];
        if (above < need && need <= above + c) {
            sm.sel_digit = static_cast<uint32_t>(d);
            sm.sel_remaining = need - above;
        }
        above += c;
    }
    __syncthreads();
}

// The row's top-12-bit histogram produced by the logits kernel (fused indexer + top-k) into
// hist[0, 4096): counts of the order keys of every visible logit of the row.  Positions forced to
// +inf leave their own bin for the +inf bin (the same mapping the key visits apply).  `issued`
// runs once the histogram's loads are in flight (work queued behind them, not ahead).
template <bool FORCED, class Issued>
__device__ void load_row_histogram(uint32_t* hist, const uint32_t* __restrict__ hist_row, const float* __restrict__ row,
                                   const Forced<FORCED>& Fg, int v, Issued&& issued) {
    constexpr int kPer = kTopBins / kTopkThreads;
    uint32_t h[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) h[j] = __ldg(hist_row + threadIdx.x + j * kTopkThreads);
    issued();
#pragma unroll
    for (int j = 0; j < kPer; ++j) hist[threadIdx.x + j * kTopkThreads] = h[j];
    __syncthreads();
    if (FORCED) {
        const int n1 = Fg.init_end;                    // [0, init_end)
        const int s2 = max(Fg.local_begin, Fg.init_end);   // [s2, v), not counted twice
        const int nf = n1 + (v - s2);
        for (int t = threadIdx.x; t < nf; t += kTopkThreads) {
            const int s = t < n1 ? t : s2 + (t - n1);
            atomicSub(&hist[order_key(__ldg(row + s)) >> 20], 1u);
            atomicAdd(&hist[0xFF800000u >> 20], 1u);
        }
        __syncthreads();
    }
}

template <bool FORCED, bool PREHIST>
__global__ void __launch_bounds__(kTopkThreads)
topk_bitmap_kernel(const float* __restrict__ logits, int64_t ld, const int32_t* __restrict__ seq_lens,
                   const int32_t* __restrict__ cu_q, int B, int row_begin, int k, int n_init, int n_local, int cmp_shift,
                   int32_t* __restrict__ idx,
                   int words_cap, const uint32_t* __restrict__ hist_g, int row_cap) {
    extern __shared__ __align__(16) unsigned char dsm[];
    BitmapSmem& sm = *reinterpret_cast<BitmapSmem*>(dsm);
    uint32_t* sel = reinterpret_cast<uint32_t*>(dsm + sizeof(BitmapSmem));   // key > k-th: kept
    uint32_t* tie = sel + words_cap;                                         // key == k-th
    uint32_t* ckey = tie + words_cap;
    int32_t* cidx = reinterpret_cast<int32_t*>(ckey + kCandidateCap);
    // with the histograms given (PREHIST) and row_cap > 0: a copy of the row, fetched while the
    // threshold bin is found (16-byte aligned: words_cap is then a multiple of 4 words)
    float* rowbuf = reinterpret_cast<float*>(cidx + kCandidateCap);

    // launched as a programmatic dependent of the logits kernel: the row's request is looked up in
    // the inputs (not written by that kernel) while it finishes, the logits are read after the wait
    ptx::griddep_launch_dependents();
    const int rl = blockIdx.x;
    const int r = row_begin + rl;
    int v = locate_visible(cu_q, seq_lens, B, r, cmp_shift, sm);
    ptx::griddep_wait();
    if (v > ld) v = static_cast<int>(ld);
    if (v > words_cap * 32) v = words_cap * 32;   // the launcher guarantees this never clips
    const float* row = logits + static_cast<int64_t>(rl) * ld;
    int32_t* out = idx + static_cast<int64_t>(rl) * k;
    if (v <= k) {
        for (int j = threadIdx.x; j < k; j += kTopkThreads) out[j] = j < v ? j : -1;
        return;
    }
    const int W = (v + 31) / 32;
    const Forced<FORCED> F = make_forced<FORCED>(v, n_init, n_local);

    // Visit every (index, key) of the row: 16-byte loads when the row is 16-byte aligned (several
    // loads in flight per thread), scalar otherwise and for the tail.
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
    const int v4 = vec ? (v >> 2) : 0;
    auto for_each_key = [&](auto&& fn) {
        const float4* row4 = reinterpret_cast<const float4*>(row);
        constexpr int U = 4;   // 16-byte loads in flight per thread
        int i = threadIdx.x;
        for (; i + (U - 1) * kTopkThreads < v4; i += U * kTopkThreads) {
            float4 a[U];
#pragma unroll
            for (int u = 0; u < U; ++u) a[u] = __ldg(row4 + i + u * kTopkThreads);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = i + u * kTopkThreads;
                fn(4 * j, F(4 * j, order_key(a[u].x))); fn(4 * j + 1, F(4 * j + 1, order_key(a[u].y)));
                fn(4 * j + 2, F(4 * j + 2, order_key(a[u].z))); fn(4 * j + 3, F(4 * j + 3, order_key(a[u].w)));
            }
        }
        for (; i < v4; i += kTopkThreads) {
            const float4 a = __ldg(row4 + i);
            fn(4 * i, F(4 * i, order_key(a.x))); fn(4 * i + 1, F(4 * i + 1, order_key(a.y)));
            fn(4 * i + 2, F(4 * i + 2, order_key(a.z))); fn(4 * i + 3, F(4 * i + 3, order_key(a.w)));
        }
        for (int s = 4 * v4 + threadIdx.x; s < v; s += kTopkThreads) fn(s, F(s, order_key(__ldg(row + s))));
    };

    // PREHIST: the row into shared memory (16-byte copies by every thread, issued right after the
    // histogram's loads and in flight while the threshold bin is found): its whole 16-byte groups,
    // so nothing at or past the visible length is read; the last < 4 keys come from global memory
    const bool use_row = PREHIST && vec && row_cap > 0 && v <= row_cap;
    auto copy_row = [&] {
        if (!use_row) return;
        const uint32_t dst0 = ptx::smem_addr(rowbuf);
        const float4* src4 = reinterpret_cast<const float4*>(row);
        for (int i = threadIdx.x; i < v4; i += kTopkThreads)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst0 + 16u * i), "l"(src4 + i) : "memory");
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    // ---- read 1: top-12-bit histogram (given by the logits kernel in the fused call)
    if (PREHIST) {
        load_row_histogram<FORCED>(sm.hist, hist_g + static_cast<int64_t>(rl) * kTopBins, row, F, v, copy_row);
    } else {
        for (int i = threadIdx.x; i < kTopBins; i += kTopkThreads) sm.hist[i] = 0;
        __syncthreads();
        for_each_key([&](int, uint32_t key) { atomicAdd(&sm.hist[key >> 20], 1u); });
        __syncthreads();
    }
    select_bin(sm.hist, sm, kTopBins, static_cast<uint32_t>(k));
    const uint32_t b1 = sm.sel_digit;
    uint32_t need = sm.sel_remaining;

    // ---- read 2: mark keys above the threshold bin, collect the threshold bin
    for (int w = threadIdx.x; w < W; w += kTopkThreads) sel[w] = tie[w] = 0u;
    if (threadIdx.x == 0) sm.cand_count = 0;
    if (use_row) asm volatile("cp.async.wait_all;" ::: "memory");   // this thread's copies landed
    __syncthreads();   // (and with them every thread's)
    auto mark = [&](int s, uint32_t key) {
        const uint32_t bin = key >> 20;
        if (bin > b1) {
            atomicOr(&sel[s >> 5], 1u << (s & 31));
        } else if (bin == b1) {
            const uint32_t p = atomicAdd(&sm.cand_count, 1u);
            if (p < static_cast<uint32_t>(kCandidateCap)) {
                ckey[p] = key;
                cidx[p] = s;
            }
        }
    };
    if (use_row) {
        const float4* r4 = reinterpret_cast<const float4*>(rowbuf);
        for (int i = threadIdx.x; i < v4; i += kTopkThreads) {
            const float4 a = r4[i];
            mark(4 * i, F(4 * i, order_key(a.x))); mark(4 * i + 1, F(4 * i + 1, order_key(a.y)));
            mark(4 * i + 2, F(4 * i + 2, order_key(a.z))); mark(4 * i + 3, F(4 * i + 3, order_key(a.w)));
        }
        for (int s = 4 * v4 + threadIdx.x; s < v; s += kTopkThreads) mark(s, F(s, order_key(__ldg(row + s))));
    } else {
        for_each_key(mark);
    }
    __syncthreads();
    const uint32_t n = sm.cand_count;
    const bool in_smem = n <= static_cast<uint32_t>(kCandidateCap);
    // ---- low digits: bits [19:10], then [9:0], of the threshold-bin keys
    uint32_t prefix = b1 << 20;
    for (int pass = 0; pass < 2; ++pass) {
        const int shift = pass == 0 ? 10 : 0;
        const int hi = shift + 10;   // bits above the digit must equal the prefix
        for (int i = threadIdx.x; i < 1024; i += kTopkThreads) sm.hist[i] = 0;
        __syncthreads();
        if (in_smem) {
            for (uint32_t i = threadIdx.x; i < n; i += kTopkThreads) {
                const uint32_t key = ckey[i];
                if ((key >> hi) == (prefix >> hi)) atomicAdd(&sm.hist[(key >> shift) & 1023u], 1u);
            }
        } else {
            for (int s = threadIdx.x; s < v; s += kTopkThreads) {
                const uint32_t key = F(s, order_key(__ldg(row + s)));
                if ((key >> hi) == (prefix >> hi)) atomicAdd(&sm.hist[(key >> shift) & 1023u], 1u);
            }
        }
        __syncthreads();
        select_bin(sm.hist, sm, 1024, need);
        prefix |= sm.sel_digit << shift;
        need = sm.sel_remaining;
        __syncthreads();
    }
    const uint32_t kth = prefix;
    const uint32_t take_equal = need;   // keys equal to kth that are kept (lowest indices first)
    if (in_smem) {
        for (uint32_t i = threadIdx.x; i < n; i += kTopkThreads) {
            const uint32_t key = ckey[i];
            const int s = cidx[i];
            if (key > kth) atomicOr(&sel[s >> 5], 1u << (s & 31));
            else if (key == kth) atomicOr(&tie[s >> 5], 1u << (s & 31));
        }
    } else {
        for (int s = threadIdx.x; s < v; s += kTopkThreads) {
            const uint32_t key = F(s, order_key(__ldg(row + s)));
            if ((key >> 20) != b1) continue;
            if (key > kth) atomicOr(&sel[s >> 5], 1u << (s & 31));
            else if (key == kth) atomicOr(&tie[s >> 5], 1u << (s & 31));
        }
    }
    __syncthreads();

    // ---- index-ordered output: thread t scans a contiguous range of bitmap words
    const int wpt = (W + kTopkThreads - 1) / kTopkThreads;
    const int w0 = min(W, threadIdx.x * wpt), w1 = min(W, w0 + wpt);
    uint32_t gt = 0, eq = 0;
    for (int w = w0; w < w1; ++w) {
        gt += __popc(sel[w]);
        eq += __popc(tie[w]);
    }
    uint32_t gt_before = gt, eq_before = eq, tot_gt, tot_eq;
    block_exclusive_scan2(gt_before, eq_before, sm, &tot_gt, &tot_eq);
    for (int w = w0; w < w1; ++w) {
        const uint32_t sw = sel[w], tw = tie[w];
        uint32_t bits = sw | tw;
        while (bits) {
            const int bit = __ffs(bits) - 1;
            bits &= bits - 1;
            const int s = w * 32 + bit;
            // positions stay below k whenever the selection counts are consistent; the guard keeps
            // every store inside the row regardless
            if ((sw >> bit) & 1u) {
                const uint32_t p = gt_before + min(eq_before, take_equal);
                if (p < static_cast<uint32_t>(k)) out[p] = s;
                ++gt_before;
            } else {
                const uint32_t p = gt_before + eq_before;
                if (eq_before < take_equal && p < static_cast<uint32_t>(k)) out[p] = s;
                ++eq_before;
            }
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Cluster kernel: the same two-read scheme with each long row split over a cluster of N = 2 or 4
// CTAs (for batches with few rows: N rows' worth of CTAs fit the GPU at once).  CTA c takes the
// keys [c w, (c + 1) w) of the row (clipped to v), w = ceil(v / N) rounded up to a multiple of 128.
// Every histogram (the 12-bit top digit, then each 10-bit low digit, each in a buffer of its own)
// is built locally in shared memory and summed over the cluster through distributed shared memory
// after one cluster barrier (16-byte remote reads, no remote atomics), so every CTA takes the same
// digit decisions; each marks its own part's bitmaps and writes its kept indices, offset by the
// kept counts of the CTAs before it.  Given the histogram (the fused indexer), each CTA copies its
// part of the row into shared memory (16-byte cp.async by every thread) while it loads the
// histogram and finds the threshold bin, and its pass over the keys reads that copy (when the part
// fits beside the other buffers: up to ~29 K keys on this GPU).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The 16 bytes at the same shared-memory offset as `p` (16-byte aligned) in CTA `rank`.
__device__ __forceinline__ uint4 ld_rank_v4(const uint32_t* p, uint32_t rank) {
    uint32_t a;
    uint4 v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(ptx::smem_addr(p)), "r"(rank));
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}

// The 4 bytes at the same shared-memory offset as `p` in CTA `rank`.
__device__ __forceinline__ uint32_t ld_rank_u32(const uint32_t* p, uint32_t rank) {
    uint32_t a, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(ptx::smem_addr(p)), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}

// total[b] = the sum over the cluster's CTAs of their hist[b], b < bins (a multiple of 4).  Every
// CTA's histogram is complete on entry.  A histogram buffer is never written again after it has
// been summed, and the kernel ends with a cluster barrier, so no barrier is needed after the reads.
template <int NC>
__device__ __forceinline__ void sum_over_cluster(const uint32_t* hist, uint32_t* total, int bins, uint32_t rank) {
    cluster_sync();   // every CTA's histogram is complete and visible
    for (int q = threadIdx.x; q < bins / 4; q += kTopkThreads) {
        uint4 acc = reinterpret_cast<const uint4*>(hist)[q];
#pragma unroll
        for (int j = 1; j < NC; ++j) {
            const uint4 o = ld_rank_v4(hist + 4 * q, (rank + j) % NC);
            acc.x += o.x; acc.y += o.y; acc.z += o.z; acc.w += o.w;
        }
        reinterpret_cast<uint4*>(total)[q] = acc;
    }
    __syncthreads();
}

template <bool FORCED, bool PREHIST, int NC>
__global__ void __launch_bounds__(kTopkThreads)
topk_cluster_kernel(const float* __restrict__ logits, int64_t ld, const int32_t* __restrict__ seq_lens,
                    const int32_t* __restrict__ cu_q, int B, int row_begin, int k, int n_init, int n_local, int cmp_shift,
                    int32_t* __restrict__ idx,
                    int words_cap, const uint32_t* __restrict__ hist_g, int cand_cap, int row_cap) {
    extern __shared__ __align__(16) unsigned char dsm[];
    BitmapSmem& sm = *reinterpret_cast<BitmapSmem*>(dsm);                      // hist: the top digit
    uint32_t* total = reinterpret_cast<uint32_t*>(dsm + sizeof(BitmapSmem));   // summed histogram
    uint32_t* lo_hist = total + kTopBins;                                        // [2][1024]: low digits
    uint32_t* xcnt = lo_hist + 2 * 1024;                                         // this part's kept counts
    uint32_t* sel = xcnt + 4;
    uint32_t* tie = sel + words_cap;
    uint32_t* ckey = tie + words_cap;
    int32_t* cidx = reinterpret_cast<int32_t*>(ckey + cand_cap);
    // with the histograms given (PREHIST) and row_cap > 0: a copy of this CTA's part of the row, fetched
    // while the threshold bin is found, so that the pass over the keys reads shared memory (16-byte
    // aligned: BitmapSmem's size, cand_cap and words_cap are multiples of 16 bytes / 4 words)
    float* rowbuf = reinterpret_cast<float*>(cidx + cand_cap);

    // launched as a programmatic dependent of the logits kernel: shared buffers are cleared and the
    // row's request is looked up in the inputs (not written by that kernel) while it finishes, the
    // logits and histograms are read after the wait
    ptx::griddep_launch_dependents();
    const uint32_t rank = cluster_rank();
    constexpr uint32_t ncta = NC;   // CTAs in the cluster (the launch's cluster size)
    const int rl = blockIdx.y;
    const int r = row_begin + rl;
    // histogram buffers zeroed while the row's request is looked up
    for (int i = threadIdx.x; i < kTopBins; i += kTopkThreads) sm.hist[i] = 0;
    for (int i = threadIdx.x; i < 2 * 1024; i += kTopkThreads) lo_hist[i] = 0;
    if (threadIdx.x == 0) sm.cand_count = 0;
    int v = locate_visible(cu_q, seq_lens, B, r, cmp_shift, sm);
    ptx::griddep_wait();
    if (v > ld) v = static_cast<int>(ld);
    // every CTA's part fits its bitmaps (the launcher guarantees this never clips)
    const int v_fit = static_cast<int>(ncta) * (words_cap * 32 - 256);
    if (v > v_fit) v = v_fit;
    const float* row = logits + static_cast<int64_t>(rl) * ld;
    int32_t* out = idx + static_cast<int64_t>(rl) * k;
    if (v <= k) {   // every CTA leaves here, before any cluster barrier
        if (rank == 0)
            for (int j = threadIdx.x; j < k; j += kTopkThreads) out[j] = j < v ? j : -1;
        return;
    }
    const int chunk = ((v + static_cast<int>(ncta) - 1) / static_cast<int>(ncta) + 127) & ~127;
    const int lo = min(v, static_cast<int>(rank) * chunk);
    const int nloc = min(v, lo + chunk) - lo;
    const int W = (nloc + 31) / 32;
    const float* part = row + lo;
    const Forced<FORCED> Fg = make_forced<FORCED>(v, n_init, n_local);
    const Forced<FORCED> F = {Fg.init_end - lo, Fg.local_begin - lo};   // in this part's local indices
    for (int w = threadIdx.x; w < W; w += kTopkThreads) sel[w] = tie[w] = 0u;

    const bool vec = (reinterpret_cast<uintptr_t>(part) & 15u) == 0;
    const int v4 = vec ? (nloc >> 2) : 0;
    // PREHIST: this part of the row into shared memory (16-byte copies by every thread, issued right
    // after the histogram's loads and in flight while the threshold bin is found): its whole 16-byte
    // groups, so nothing at or past the row's visible length is read; the last < 4 keys are read
    // from global memory in the pass over the keys
    const bool use_row = PREHIST && vec && row_cap > 0 && nloc <= row_cap;
    auto copy_row = [&] {
        if (!use_row) return;
        const uint32_t dst0 = ptx::smem_addr(rowbuf);
        const float4* src4 = reinterpret_cast<const float4*>(part);
        for (int i = threadIdx.x; i < v4; i += kTopkThreads)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst0 + 16u * i), "l"(src4 + i) : "memory");
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    auto for_each_key = [&](auto&& fn) {   // (local index, key) of this part
        const float4* p4 = reinterpret_cast<const float4*>(part);
        constexpr int U = 4;
        int i = threadIdx.x;
        for (; i + (U - 1) * kTopkThreads < v4; i += U * kTopkThreads) {
            float4 a[U];
#pragma unroll
            for (int u = 0; u < U; ++u) a[u] = __ldg(p4 + i + u * kTopkThreads);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = i + u * kTopkThreads;
                fn(4 * j, F(4 * j, order_key(a[u].x))); fn(4 * j + 1, F(4 * j + 1, order_key(a[u].y)));
                fn(4 * j + 2, F(4 * j + 2, order_key(a[u].z))); fn(4 * j + 3, F(4 * j + 3, order_key(a[u].w)));
            }
        }
        for (; i < v4; i += kTopkThreads) {
            const float4 a = __ldg(p4 + i);
            fn(4 * i, F(4 * i, order_key(a.x))); fn(4 * i + 1, F(4 * i + 1, order_key(a.y)));
            fn(4 * i + 2, F(4 * i + 2, order_key(a.z))); fn(4 * i + 3, F(4 * i + 3, order_key(a.w)));
        }
        for (int s = 4 * v4 + threadIdx.x; s < nloc; s += kTopkThreads) fn(s, F(s, order_key(__ldg(part + s))));
    };

    // ---- read 1: top-12-bit histogram of this part, summed over the cluster (in the fused call: the
    // whole row's histogram from the logits kernel, the same in every CTA)
    if (PREHIST) {
        load_row_histogram<FORCED>(total, hist_g + static_cast<int64_t>(rl) * kTopBins, row, Fg, v, copy_row);
    } else {
        for_each_key([&](int, uint32_t key) { atomicAdd(&sm.hist[key >> 20], 1u); });
        __syncthreads();
        sum_over_cluster<NC>(sm.hist, total, kTopBins, rank);
    }
    select_bin(total, sm, kTopBins, static_cast<uint32_t>(k));
    const uint32_t b1 = sm.sel_digit;
    uint32_t need = sm.sel_remaining;

    // ---- read 2: mark keys above the threshold bin, collect the threshold bin (this part)
    if (use_row) {   // every thread's copies landed, then all of them are visible
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();
    }
    auto mark = [&](int s, uint32_t key) {
        const uint32_t bin = key >> 20;
        if (bin > b1) {
            atomicOr(&sel[s >> 5], 1u << (s & 31));
        } else if (bin == b1) {
            const uint32_t p = atomicAdd(&sm.cand_count, 1u);
            if (p < static_cast<uint32_t>(cand_cap)) {
                ckey[p] = key;
                cidx[p] = s;
            }
        }
    };
    if (use_row) {
        const float4* r4 = reinterpret_cast<const float4*>(rowbuf);
        for (int i = threadIdx.x; i < v4; i += kTopkThreads) {
            const float4 a = r4[i];
            mark(4 * i, F(4 * i, order_key(a.x))); mark(4 * i + 1, F(4 * i + 1, order_key(a.y)));
            mark(4 * i + 2, F(4 * i + 2, order_key(a.z))); mark(4 * i + 3, F(4 * i + 3, order_key(a.w)));
        }
        for (int s = 4 * v4 + threadIdx.x; s < nloc; s += kTopkThreads) mark(s, F(s, order_key(__ldg(part + s))));
    } else {
        for_each_key(mark);
    }
    __syncthreads();
    const uint32_t n = sm.cand_count;
    const bool in_smem = n <= static_cast<uint32_t>(cand_cap);
    // ---- low digits: bits [19:10], then [9:0], over the cluster's threshold-bin keys
    uint32_t prefix = b1 << 20;
    // When every CTA's candidates are in its shared memory and together fit 4096 keys, each CTA
    // copies all of them (its peers' by distributed shared-memory loads) into `total` (free once
    // the threshold bin is known) and finds both digits alone: one cluster barrier instead of one
    // per digit with the digit histograms summed across the cluster.  Every CTA sees the same
    // counts, so all take the same branch.
    cluster_sync();   // every CTA's candidates and count are complete and visible
    uint32_t coff[NC];
    uint32_t ntot = 0;
    bool all_in = true;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const uint32_t nc = static_cast<uint32_t>(c) == rank ? n : ld_rank_u32(&sm.cand_count, c);
        coff[c] = ntot;
        ntot += nc;
        all_in = all_in && nc <= static_cast<uint32_t>(cand_cap);
    }
    const bool gathered = all_in && ntot <= static_cast<uint32_t>(kTopBins);
    if (gathered) {
        uint32_t* ukey = total;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const uint32_t nc = (c + 1 < NC ? coff[c + 1] : ntot) - coff[c];
            if (static_cast<uint32_t>(c) == rank) {
                for (uint32_t i = threadIdx.x; i < nc; i += kTopkThreads) ukey[coff[c] + i] = ckey[i];
            } else {   // 16-byte loads (ckey is 16-byte aligned and cand_cap a multiple of 4)
                for (uint32_t q = threadIdx.x; 4 * q < nc; q += kTopkThreads) {
                    const uint4 v4 = ld_rank_v4(ckey + 4 * q, c);
                    const uint32_t i = 4 * q;
                    ukey[coff[c] + i] = v4.x;
                    if (i + 1 < nc) ukey[coff[c] + i + 1] = v4.y;
                    if (i + 2 < nc) ukey[coff[c] + i + 2] = v4.z;
                    if (i + 3 < nc) ukey[coff[c] + i + 3] = v4.w;
                }
            }
        }
        __syncthreads();
        for (int pass = 0; pass < 2; ++pass) {
            const int shift = pass == 0 ? 10 : 0;
            const int hi = shift + 10;
            uint32_t* h = lo_hist + pass * 1024;
            for (uint32_t i = threadIdx.x; i < ntot; i += kTopkThreads) {
                const uint32_t key = ukey[i];
                if ((key >> hi) == (prefix >> hi)) atomicAdd(&h[(key >> shift) & 1023u], 1u);
            }
            __syncthreads();
            select_bin(h, sm, 1024, need);
            prefix |= sm.sel_digit << shift;
            need = sm.sel_remaining;
            __syncthreads();
        }
    }
    for (int pass = 0; pass < 2 && !gathered; ++pass) {
        const int shift = pass == 0 ? 10 : 0;
        const int hi = shift + 10;
        uint32_t* h = lo_hist + pass * 1024;
        if (in_smem) {
            for (uint32_t i = threadIdx.x; i < n; i += kTopkThreads) {
                const uint32_t key = ckey[i];
                if ((key >> hi) == (prefix >> hi)) atomicAdd(&h[(key >> shift) & 1023u], 1u);
            }
        } else {
            for (int s = threadIdx.x; s < nloc; s += kTopkThreads) {
                const uint32_t key = F(s, order_key(__ldg(part + s)));
                if ((key >> hi) == (prefix >> hi)) atomicAdd(&h[(key >> shift) & 1023u], 1u);
            }
        }
        __syncthreads();
        sum_over_cluster<NC>(h, total, 1024, rank);
        select_bin(total, sm, 1024, need);
        prefix |= sm.sel_digit << shift;
        need = sm.sel_remaining;
        __syncthreads();
    }
    const uint32_t kth = prefix;
    const uint32_t take_equal = need;   // keys equal to kth that are kept (lowest indices first)
    if (in_smem) {
        for (uint32_t i = threadIdx.x; i < n; i += kTopkThreads) {
            const uint32_t key = ckey[i];
            const int s = cidx[i];
            if (key > kth) atomicOr(&sel[s >> 5], 1u << (s & 31));
            else if (key == kth) atomicOr(&tie[s >> 5], 1u << (s & 31));
        }
    } else {
        for (int s = threadIdx.x; s < nloc; s += kTopkThreads) {
            const uint32_t key = F(s, order_key(__ldg(part + s)));
            if ((key >> 20) != b1) continue;
            if (key > kth) atomicOr(&sel[s >> 5], 1u << (s & 31));
            else if (key == kth) atomicOr(&tie[s >> 5], 1u << (s & 31));
        }
    }
    __syncthreads();

    // ---- index-ordered output; each part starts after the kept keys of the parts before it
    const int wpt = (W + kTopkThreads - 1) / kTopkThreads;
    const int w0 = min(W, threadIdx.x * wpt), w1 = min(W, w0 + wpt);
    uint32_t gt_before = 0, eq_before = 0;
    for (int w = w0; w < w1; ++w) {
        gt_before += __popc(sel[w]);
        eq_before += __popc(tie[w]);
    }
    uint32_t gt_tot, eq_tot;
    block_exclusive_scan2(gt_before, eq_before, sm, &gt_tot, &eq_tot);
    if (threadIdx.x == 0) {
        xcnt[0] = gt_tot;
        xcnt[1] = eq_tot;
    }
    __syncthreads();
    cluster_sync();   // every CTA's counts are visible
    for (uint32_t c = 0; c < rank; ++c) {
        const uint4 cc = ld_rank_v4(xcnt, c);
        gt_before += cc.x;
        eq_before += cc.y;
    }
    for (int w = w0; w < w1; ++w) {
        const uint32_t sw = sel[w], tw = tie[w];
        uint32_t bits = sw | tw;
        while (bits) {
            const int bit = __ffs(bits) - 1;
            bits &= bits - 1;
            const int s = lo + w * 32 + bit;
            // positions stay below k whenever the selection counts are consistent; the guard keeps
            // every store inside the row regardless
            if ((sw >> bit) & 1u) {
                const uint32_t p = gt_before + min(eq_before, take_equal);
                if (p < static_cast<uint32_t>(k)) out[p] = s;
                ++gt_before;
            } else {
                const uint32_t p = gt_before + eq_before;
                if (eq_before < take_equal && p < static_cast<uint32_t>(k)) out[p] = s;
                ++eq_before;
            }
        }
    }
    cluster_sync();   // every CTA has read this CTA's histograms and counts before any leaves
}

size_t cluster_smem_bytes(int words, int cand_cap, int row_cap) {
    return sizeof(BitmapSmem) + static_cast<size_t>(kTopBins) * 4 + 2 * 1024 * 4 + 16 +
           2 * static_cast<size_t>(words) * 4 + static_cast<size_t>(cand_cap) * 8 + static_cast<size_t>(row_cap) * 4;
}

size_t bitmap_smem_bytes(int words) {
    return sizeof(BitmapSmem) + 2 * static_cast<size_t>(words) * 4 + static_cast<size_t>(kCandidateCap) * 8;
}

}  // namespace
}  // namespace dsa

extern "C" size_t dsa_topk_workspace_size(int32_t rows, int32_t k, int32_t max_seq_len) {
    (void)rows; (void)k; (void)max_seq_len;
    return 0;
}

namespace dsa {

template <bool F, bool P, int NC>
void* topk_cluster_fn() { return reinterpret_cast<void*>(topk_cluster_kernel<F, P, NC>); }
template <bool F, bool P>
void* topk_bitmap_fn() { return reinterpret_cast<void*>(topk_bitmap_kernel<F, P>); }

// The top-k call; with hist_g != nullptr (the fused indexer + top-k) every row's top-12-bit key
// histogram comes from hist_g[(r - row_begin) * 4096 ..] instead of a first read of the row.
dsa_status topk_launch(const float* logits, int64_t ld, const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                       int32_t max_seq_len, int32_t row_begin, int32_t row_end, int32_t k, int32_t n_init,
                       int32_t n_local, int32_t* idx, void* stream, const uint32_t* hist_g, int32_t cmp_shift) {
    if (k < 1 || k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
    if (n_init < 0 || n_local < 0 || cmp_shift < 0 || cmp_shift > 7) return DSA_ERR_INVALID_ARG;
    const bool forced = n_init > 0 || n_local > 0;
    if (B < 0 || row_begin < 0 || row_end < row_begin || max_seq_len < 0) return DSA_ERR_INVALID_ARG;
    if (row_end == row_begin) return DSA_OK;
    if (B == 0 || !logits || !seq_lens || !cu_q || !idx) return DSA_ERR_INVALID_ARG;
    if (ld < max_seq_len) return DSA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int words = (max_seq_len + 31) / 32;
    // a programmatic dependent of the previous kernel on the stream (the logits kernel): its CTAs
    // may be scheduled early and wait on the device for that kernel's results
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(row_end - row_begin), 1, 1);
    cfg.blockDim = dim3(dsa::kTopkThreads, 1, 1);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return DSA_ERR_CUDA;
    const bool pre = hist_g != nullptr;
    if (pre && words > dsa::kMaxBitmapWords) return DSA_ERR_UNSUPPORTED;
    if (words <= dsa::kMaxBitmapWords && max_seq_len >= 16384 && (row_end - row_begin) <= sms / 2) {
        // long rows, fewer rows than SM pairs: each row on a cluster of ncta CTAs -- 4 when the
        // clusters of all rows fit 128 SMs at once and every CTA keeps at least 4096 keys of the
        // longest row, else 2 (8-CTA clusters measured slower: 16 rows of 128K keys 75 us
        // against 61 us with 4)
        const int rows = row_end - row_begin;
        const int ncta = (rows * 4 <= 128 && max_seq_len >= 4 * 4096) ? 4 : 2;
        const int part_keys = ((max_seq_len + ncta - 1) / ncta + 127) & ~127;
        int words_cap = ((part_keys + 256 + 31) / 32 + 3) & ~3;
        if (words_cap < 32) words_cap = 32;
        // with the histograms given: each CTA's part of the row in shared memory as well when it
        // fits (the threshold-bin candidates then get 4096 slots instead of 8192; more fall back to
        // reading the row)
        int cand_cap = dsa::kCandidateCap, row_cap = 0;
        int smem_max = 0;
        if (cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return DSA_ERR_CUDA;
        const int row_keys = (part_keys + 3) & ~3;
        if (pre && dsa::cluster_smem_bytes(words_cap, 4096, row_keys) <= static_cast<size_t>(smem_max)) {
            cand_cap = 4096;
            row_cap = row_keys;
        }
        const size_t smem = dsa::cluster_smem_bytes(words_cap, cand_cap, row_cap);
        void* kern = ncta == 4
                         ? (forced ? (pre ? topk_cluster_fn<true, true, 4>() : topk_cluster_fn<true, false, 4>())
                                   : (pre ? topk_cluster_fn<false, true, 4>() : topk_cluster_fn<false, false, 4>()))
                         : (forced ? (pre ? topk_cluster_fn<true, true, 2>() : topk_cluster_fn<true, false, 2>())
                                   : (pre ? topk_cluster_fn<false, true, 2>() : topk_cluster_fn<false, false, 2>()));
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess)
            return DSA_ERR_CUDA;
        cudaLaunchAttribute cattr[2];
        cattr[0].id = cudaLaunchAttributeClusterDimension;
        cattr[0].val.clusterDim.x = static_cast<unsigned>(ncta);
        cattr[0].val.clusterDim.y = 1;
        cattr[0].val.clusterDim.z = 1;
        cattr[1] = attr[0];
        cfg.gridDim = dim3(static_cast<unsigned>(ncta), static_cast<unsigned>(rows), 1);
        cfg.attrs = cattr;
        cfg.numAttrs = 2;
        cfg.dynamicSmemBytes = smem;
        int a_B = B, a_rb = row_begin, a_k = k, a_ni = n_init, a_nl = n_local, a_sh = cmp_shift, a_wc = words_cap;
        void* args[] = {const_cast<float**>(&logits), &ld, const_cast<int32_t**>(&seq_lens), const_cast<int32_t**>(&cu_q),
                        &a_B, &a_rb, &a_k, &a_ni, &a_nl, &a_sh, &idx, &a_wc, const_cast<uint32_t**>(&hist_g),
                        &cand_cap, &row_cap};
        if (cudaLaunchKernelExC(&cfg, kern, args) != cudaSuccess) return DSA_ERR_CUDA;
    } else if (words <= dsa::kMaxBitmapWords) {
        int words_cap = words < 32 ? 32 : words;
        // with the histograms given: the row in shared memory as well when it fits
        int row_cap = 0;
        if (pre) {
            int smem_max = 0;
            if (cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
                return DSA_ERR_CUDA;
            const int wc4 = (words_cap + 3) & ~3;
            const int row_keys = (max_seq_len + 3) & ~3;
            if (dsa::bitmap_smem_bytes(wc4) + static_cast<size_t>(row_keys) * 4 <= static_cast<size_t>(smem_max)) {
                words_cap = wc4;
                row_cap = row_keys;
            }
        }
        const size_t smem = dsa::bitmap_smem_bytes(words_cap) + static_cast<size_t>(row_cap) * 4;
        void* kern = forced ? (pre ? topk_bitmap_fn<true, true>() : topk_bitmap_fn<true, false>())
                            : (pre ? topk_bitmap_fn<false, true>() : topk_bitmap_fn<false, false>());
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess)
            return DSA_ERR_CUDA;
        cfg.dynamicSmemBytes = smem;
        int a_B = B, a_rb = row_begin, a_k = k, a_ni = n_init, a_nl = n_local, a_sh = cmp_shift, a_wc = words_cap;
        void* args[] = {const_cast<float**>(&logits), &ld, const_cast<int32_t**>(&seq_lens), const_cast<int32_t**>(&cu_q),
                        &a_B, &a_rb, &a_k, &a_ni, &a_nl, &a_sh, &idx, &a_wc, const_cast<uint32_t**>(&hist_g),
                        &row_cap};
        if (cudaLaunchKernelExC(&cfg, kern, args) != cudaSuccess) return DSA_ERR_CUDA;
    } else {
        cfg.dynamicSmemBytes = 0;
        auto kern = forced ? dsa::topk_kernel<true> : dsa::topk_kernel<false>;
        if (cudaLaunchKernelEx(&cfg, kern, logits, ld, seq_lens, cu_q, static_cast<int>(B),
                               static_cast<int>(row_begin), static_cast<int>(k), n_init, n_local,
                               static_cast<int>(cmp_shift), idx) !=
                                   cudaSuccess)
            return DSA_ERR_CUDA;
    }
    return dsa::launch_status();
}

}  // namespace dsa

extern "C" dsa_status dsa_topk_forced(const float* logits, int64_t ld, const int32_t* seq_lens, const int32_t* cu_q,
                                      int32_t B, int32_t max_seq_len, int32_t row_begin, int32_t row_end, int32_t k,
                                      int32_t n_init, int32_t n_local, int32_t* idx, void* workspace,
                                      size_t workspace_bytes, void* stream) {
    (void)workspace; (void)workspace_bytes;
    return dsa::topk_launch(logits, ld, seq_lens, cu_q, B, max_seq_len, row_begin, row_end, k, n_init, n_local, idx,
                            stream, nullptr, 0);
}

extern "C" dsa_status dsa_topk(const float* logits, int64_t ld, const int32_t* seq_lens, const int32_t* cu_q,
                               int32_t B, int32_t max_seq_len, int32_t row_begin, int32_t row_end, int32_t k,
                               int32_t* idx, void* workspace, size_t workspace_bytes, void* stream) {
    return dsa_topk_forced(logits, ld, seq_lens, cu_q, B, max_seq_len, row_begin, row_end, k, 0, 0, idx, workspace,
                           workspace_bytes, stream);
}
