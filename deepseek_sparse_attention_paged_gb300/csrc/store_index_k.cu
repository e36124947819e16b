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
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "dsa_common.cuh"
#include "sm100_ptx.cuh"

namespace dsa {
namespace {

// fp32 value nearest to 1/sqrt(128) = 2^-3.5.
constexpr float kInvSqrt128 = 0x1.6a09e6p-4f;

// Quantise and store one key held by a warp (lane l: elements 4l .. 4l+3, exact fp32 values of
// bf16 numbers) at row `row` of page `pg`.
// ue8m0: the scale is the smallest power of two not below the fp32 scale.
__device__ __forceinline__ void quant_store(const float (&y)[4], int lane, uint8_t* __restrict__ pg, int row,
                                            bool ue8m0) {
    float amax = fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3])));
    amax = warp_max(amax);
    float scale = __fdiv_rn(fmaxf(amax, 1e-4f), 448.0f);
    if (ue8m0) {
        const uint32_t u = __float_as_uint(scale);
        if (u & 0x007fffffu) scale = __uint_as_float((u & 0x7f800000u) + 0x00800000u);
    }

    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(__fdiv_rn(y[e], scale), __NV_SATFINITE, __NV_E4M3);
        packed |= static_cast<uint32_t>(c) << (8 * e);
    }
    reinterpret_cast<uint32_t*>(pg + row * kIndexDim)[lane] = packed;
    if (lane == 0) reinterpret_cast<float*>(pg + kIndexScaleOffset)[row] = scale;
}

// Rotate, quantise and store one key held by a warp (layout as above).
__device__ __forceinline__ void rotate_quant_store(float (&x)[4], int lane, uint8_t* __restrict__ pg, int row,
                                                   bool ue8m0 = false) {
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
    quant_store(y, lane, pg, row, ue8m0);
}

__global__ void __launch_bounds__(256)
store_index_k_kernel(const uint16_t* __restrict__ keys, const int64_t* __restrict__ slots, int64_t n,
                     uint8_t* __restrict__ pool, int64_t num_pages, int32_t* err) {
    // the next kernel on the stream may be scheduled (the indexer's query prologue waits on the device
    // for this grid before it reads or writes anything)
    ptx::griddep_launch_dependents();
    const int64_t token = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (token >= n) return;                      // warp-uniform
    // both loads in flight before the slot is examined
    const int64_t slot = __ldg(slots + token);
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(keys + token * kIndexDim) + lane);
    if (slot < 0) return;                        // padding token
    const int64_t page = slot >> 6;
    const int row = static_cast<int>(slot & 63);
    if (page >= num_pages) {
        if (lane == 0) raise_error(err, DSA_DEVERR_SLOT_RANGE);
        return;
    }
    float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
    rotate_quant_store(x, lane, pool + page * kIndexPageBytes, row);
}

// ---------------------------------------------------------------- key norm and rotary embedding

__device__ __forceinline__ float round_bf16(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// fp32 sum of the 128 values a warp holds (lane l: v[0..3] = elements 4l .. 4l+3): within each
// lane, then a butterfly over lanes (distance 1, 2, 4, 8, 16).  At each level a lane adds its
// partner's partial to its own; both lanes of a pair add the same two numbers, so every lane ends
// with the same bits.  (The norm's definition sums exactly; this fp32 evaluation is within a few
// fp32 units of it.)
__device__ __forceinline__ float warp_sum128_tree(const float (&v)[4]) {
    float s = __fadd_rn(__fadd_rn(v[0], v[1]), __fadd_rn(v[2], v[3]));
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, m));
    return s;
}

// In place: LayerNorm (rms = false: y = ((x - mean) * rstd) * w + b) or RMSNorm (rms = true:
// y = (x * rstd) * w) of the 128-vector a warp holds, every step an IEEE fp32 operation without
// fused multiply-add, rstd = 1 / sqrt(var + eps), the result rounded to bf16.
__device__ __forceinline__ void warp_norm128(float (&x)[4], const float4 wv, const float4 bv, float eps, bool rms) {
    const float wl[4] = {wv.x, wv.y, wv.z, wv.w};
    float t[4];
    if (rms) {
#pragma unroll
        for (int e = 0; e < 4; ++e) t[e] = __fmul_rn(x[e], x[e]);
        const float ms = __fmul_rn(warp_sum128_tree(t), 1.0f / kIndexDim);
        const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = round_bf16(__fmul_rn(__fmul_rn(x[e], rstd), wl[e]));
        return;
    }
    const float bl[4] = {bv.x, bv.y, bv.z, bv.w};
    const float mean = __fmul_rn(warp_sum128_tree(x), 1.0f / kIndexDim);
    float d[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        d[e] = __fsub_rn(x[e], mean);
        t[e] = __fmul_rn(d[e], d[e]);
    }
    const float var = __fmul_rn(warp_sum128_tree(t), 1.0f / kIndexDim);
    const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, eps)));
#pragma unroll
    for (int e = 0; e < 4; ++e) x[e] = round_bf16(__fadd_rn(__fmul_rn(__fmul_rn(d[e], rstd), wl[e]), bl[e]));
}

// Rotary embedding of dims 0 .. 63 of the 128-vector a warp holds (exact fp32 values of bf16
// numbers), from the position's cos/sin row (cos in [0, 32), sin in [32, 64)).  neox pairing
// (i, i + 32): lane l < 8 holds i = 4l + e and lane l + 8 holds i + 32, exchanged with one
// shuffle; interleaved pairing (2i, 2i + 1): both halves in one lane.  ya = a c - b s,
// yb = b c + a s in fp32 without fused multiply-add, rounded to bf16; dims 64 .. 127 (lanes
// 16 .. 31) pass through.
struct RopeCoef {
    float c[4], s[4];   // neox: c[e], s[e] of i = 4 (lane & 7) + e; interleaved: c[p], s[p] of i = 2 lane + p
};

// This lane's cos / sin values (lanes 16 .. 31 need none).
__device__ __forceinline__ RopeCoef load_rope(const float* __restrict__ cs, int lane, bool neox) {
    RopeCoef r = {};
    if (lane >= 16) return r;
    if (neox) {
        const int i0 = 4 * (lane & 7);
        const float4 c = __ldg(reinterpret_cast<const float4*>(cs + i0));
        const float4 s = __ldg(reinterpret_cast<const float4*>(cs + 32 + i0));
        r.c[0] = c.x; r.c[1] = c.y; r.c[2] = c.z; r.c[3] = c.w;
        r.s[0] = s.x; r.s[1] = s.y; r.s[2] = s.z; r.s[3] = s.w;
    } else {
        const float2 c = __ldg(reinterpret_cast<const float2*>(cs + 2 * lane));
        const float2 s = __ldg(reinterpret_cast<const float2*>(cs + 32 + 2 * lane));
        r.c[0] = c.x; r.c[1] = c.y;
        r.s[0] = s.x; r.s[1] = s.y;
    }
    return r;
}

__device__ __forceinline__ void warp_rope64(float (&x)[4], int lane, const RopeCoef& k, bool neox) {
    if (neox) {
        float other[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) other[e] = __shfl_xor_sync(0xffffffffu, x[e], 8);
        if (lane >= 16) return;
        if (lane < 8) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                x[e] = round_bf16(__fsub_rn(__fmul_rn(x[e], k.c[e]), __fmul_rn(other[e], k.s[e])));
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                x[e] = round_bf16(__fadd_rn(__fmul_rn(x[e], k.c[e]), __fmul_rn(other[e], k.s[e])));
        }
        return;
    }
    if (lane >= 16) return;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const float a = x[2 * p], bb = x[2 * p + 1];
        x[2 * p] = round_bf16(__fsub_rn(__fmul_rn(a, k.c[p]), __fmul_rn(bb, k.s[p])));
        x[2 * p + 1] = round_bf16(__fadd_rn(__fmul_rn(bb, k.c[p]), __fmul_rn(a, k.s[p])));
    }
}

__global__ void __launch_bounds__(256)
store_index_k_prologue_kernel(const uint16_t* __restrict__ keys, const float* __restrict__ norm_w,
                              const float* __restrict__ norm_b, float eps, const float* __restrict__ cos_sin,
                              int64_t max_position, const int64_t* __restrict__ positions,
                              const int64_t* __restrict__ slots, int64_t n, uint8_t* __restrict__ pool,
                              int64_t num_pages, uint32_t flags, int32_t* err) {
    const int64_t token = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (token >= n) return;                      // warp-uniform
    const bool rms = (flags & DSA_NORM_RMS) != 0;
    const bool neox = (flags & DSA_ROPE_INTERLEAVED) == 0;
    // every load that does not depend on another is in flight before anything is examined
    const int64_t slot = __ldg(slots + token);
    const int64_t pos = __ldg(positions + token);
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(keys + token * kIndexDim) + lane);
    const float4 wv = __ldg(reinterpret_cast<const float4*>(norm_w) + lane);
    const float4 bv = __ldg(reinterpret_cast<const float4*>(norm_b) + lane);   // unused with RMSNorm
    if (slot < 0) return;                        // padding token
    if (pos < 0 || pos >= max_position) {
        if (lane == 0) raise_error(err, DSA_DEVERR_POSITION);
        return;
    }
    const RopeCoef rc = load_rope(cos_sin + pos * 64, lane, neox);   // in flight during the norm
    const int64_t page = slot >> 6;
    const int row = static_cast<int>(slot & 63);
    if (page >= num_pages) {
        if (lane == 0) raise_error(err, DSA_DEVERR_SLOT_RANGE);
        return;
    }
    float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
    warp_norm128(x, wv, bv, eps, rms);
    warp_rope64(x, lane, rc, neox);
    const bool ue8m0 = (flags & DSA_SCALE_UE8M0) != 0;
    if (flags & DSA_K_NO_ROTATE) quant_store(x, lane, pool + page * kIndexPageBytes, row, ue8m0);
    else rotate_quant_store(x, lane, pool + page * kIndexPageBytes, row, ue8m0);
}

// One warp per (row, group of HPW heads) of the indexer query: the row's cos/sin values are loaded
// once, the group's head vectors are read up to 8 at a time (independent 256-byte loads in flight
// per warp), rotated and written as bf16; a row whose position is out of range is copied
// unchanged.  HPW = 16 for many rows (fewer cos/sin loads, more bytes in flight per warp), 1 for
// few rows (more warps).
template <int HPW>
__global__ void __launch_bounds__(256)
indexer_rope_q_kernel(const uint16_t* q, const float* __restrict__ cos_sin, int64_t max_position,
                      const int64_t* __restrict__ positions, int64_t T, uint32_t flags, uint16_t* out,
                      int32_t* err) {
    constexpr int kGroups = kIndexHeads / HPW;
    constexpr int kBatch = HPW < 8 ? HPW : 8;
    const int64_t wg = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t t = wg / kGroups;
    if (t >= T) return;                          // warp-uniform
    const int64_t v0 = t * kIndexHeads + (wg % kGroups) * HPW;
    const int64_t pos = __ldg(positions + t);
    const bool ok = pos >= 0 && pos < max_position;
    if (!ok && lane == 0 && v0 % kIndexHeads == 0) raise_error(err, DSA_DEVERR_POSITION);
    const bool neox = (flags & DSA_ROPE_INTERLEAVED) == 0;
    RopeCoef rc = {};
    if (ok) rc = load_rope(cos_sin + pos * 64, lane, neox);
#pragma unroll 1
    for (int h0 = 0; h0 < HPW; h0 += kBatch) {
        // q and out may be the same array: each lane reads its 8 bytes before it writes them
        uint2 raw[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) raw[j] = reinterpret_cast<const uint2*>(q + (v0 + h0 + j) * kIndexDim)[lane];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            uint2 y = raw[j];
            if (ok) {
                float x[4] = {bf16_lo(raw[j].x), bf16_hi(raw[j].x), bf16_lo(raw[j].y), bf16_hi(raw[j].y)};
                warp_rope64(x, lane, rc, neox);
                // every value is an exact bf16 number: its bits are the top half of the fp32 word
                y = make_uint2((__float_as_uint(x[0]) >> 16) | (__float_as_uint(x[1]) & 0xffff0000u),
                               (__float_as_uint(x[2]) >> 16) | (__float_as_uint(x[3]) & 0xffff0000u));
            }
            reinterpret_cast<uint2*>(out + (v0 + h0 + j) * kIndexDim)[lane] = y;
        }
    }
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


extern "C" dsa_status dsa_store_index_k_prologue(const void* k_raw_bf16, const float* norm_weight,
                                                 const float* norm_bias, float eps, const float* cos_sin_cache,
                                                 int64_t max_position, const int64_t* positions,
                                                 const int64_t* slot_mapping, int64_t n, uint8_t* index_k_pool,
                                                 int64_t num_pages, int32_t page_size, uint32_t flags,
                                                 int32_t* dev_err, void* stream) {
    if (n < 0 || num_pages < 0 || max_position < 0) return DSA_ERR_INVALID_ARG;
    if (page_size != dsa::kPage) return DSA_ERR_UNSUPPORTED;
    if (flags & ~static_cast<uint32_t>(DSA_NORM_RMS | DSA_ROPE_INTERLEAVED | DSA_K_NO_ROTATE | DSA_SCALE_UE8M0))
        return DSA_ERR_INVALID_ARG;
    if (n == 0) return DSA_OK;
    const bool rms = (flags & DSA_NORM_RMS) != 0;
    if (!k_raw_bf16 || !norm_weight || (!rms && !norm_bias) || !cos_sin_cache || !positions || !slot_mapping ||
        !index_k_pool)
        return DSA_ERR_INVALID_ARG;
    if (!dsa::aligned16(k_raw_bf16) || !dsa::aligned16(index_k_pool) || !dsa::aligned16(norm_weight) ||
        (!rms && !dsa::aligned16(norm_bias)) || !dsa::aligned16(cos_sin_cache))
        return DSA_ERR_INVALID_ARG;
    const int64_t blocks = (n + 7) / 8;
    if (blocks > 0x7fffffffLL) return DSA_ERR_INVALID_ARG;
    dsa::store_index_k_prologue_kernel<<<static_cast<unsigned>(blocks), 256, 0,
                                         static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(k_raw_bf16), norm_weight, rms ? norm_weight : norm_bias, eps, cos_sin_cache,
        max_position, positions, slot_mapping, n, index_k_pool, num_pages, flags, dev_err);
    return dsa::launch_status();
}

extern "C" dsa_status dsa_indexer_rope_q(const void* q_raw_bf16, const float* cos_sin_cache, int64_t max_position,
                                         const int64_t* positions, int64_t T, uint32_t flags, void* q_out_bf16,
                                         int32_t* dev_err, void* stream) {
    if (T < 0 || max_position < 0) return DSA_ERR_INVALID_ARG;
    if (flags & ~static_cast<uint32_t>(DSA_ROPE_INTERLEAVED)) return DSA_ERR_INVALID_ARG;
    if (T == 0) return DSA_OK;
    if (!q_raw_bf16 || !cos_sin_cache || !positions || !q_out_bf16) return DSA_ERR_INVALID_ARG;
    if (!dsa::aligned16(q_raw_bf16) || !dsa::aligned16(q_out_bf16) || !dsa::aligned16(cos_sin_cache))
        return DSA_ERR_INVALID_ARG;
    // 16 heads per warp once that still gives about 32 warps per SM, else one
    const bool wide = T * (dsa::kIndexHeads / 16) >= static_cast<int64_t>(dsa::device_sm_count()) * 32;
    const int64_t warps = T * (wide ? dsa::kIndexHeads / 16 : dsa::kIndexHeads);
    const int64_t blocks = (warps + 7) / 8;
    if (blocks > 0x7fffffffLL) return DSA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint16_t* qi = static_cast<const uint16_t*>(q_raw_bf16);
    uint16_t* qo = static_cast<uint16_t*>(q_out_bf16);
    if (wide)
        dsa::indexer_rope_q_kernel<16><<<static_cast<unsigned>(blocks), 256, 0, s>>>(qi, cos_sin_cache, max_position,
                                                                                     positions, T, flags, qo, dev_err);
    else
        dsa::indexer_rope_q_kernel<1><<<static_cast<unsigned>(blocks), 256, 0, s>>>(qi, cos_sin_cache, max_position,
                                                                                    positions, T, flags, qo, dev_err);
    return dsa::launch_status();
}

// ---------------------------------------------------------------- FP8 latent cache store

namespace dsa {
namespace {

// One warp per token: the 576 bf16 latent + rope values (lane l: the pairs 2 (l + 32 i), i < 9) to
// E4M3FN codes of x / k_scale (one IEEE fp32 division, round to nearest even, saturating), written
// to row slot & 63 of page slot >> 6 of the FP8 cache.  Follows vllm mla/common.py,
// MLACommonImpl.forward: concat_and_cache_mla(k_c_normed, k_pe, kv_cache, slot_mapping,
// kv_cache_dtype = "fp8", scale = layer._k_scale).
__global__ void __launch_bounds__(256)
store_latent_fp8_kernel(const uint32_t* __restrict__ latent, const int64_t* __restrict__ slots, int64_t n,
                        float k_scale, uint16_t* __restrict__ pool, int64_t num_pages, int32_t* err) {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= n) return;
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) return;
    if ((slot >> 6) >= num_pages) {
        if (lane == 0) raise_error(err, DSA_DEVERR_SLOT_RANGE);
        return;
    }
    const uint32_t* src = latent + t * (kLatentDim / 2);
    uint16_t* dst = pool + slot * (kLatentDim / 2);
#pragma unroll
    for (int i = 0; i < kLatentDim / 64; ++i) {
        const uint32_t two = __ldg(src + lane + 32 * i);
        const __nv_fp8_storage_t c0 = __nv_cvt_float_to_fp8(__fdiv_rn(bf16_lo(two), k_scale), __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8_storage_t c1 = __nv_cvt_float_to_fp8(__fdiv_rn(bf16_hi(two), k_scale), __NV_SATFINITE, __NV_E4M3);
        dst[lane + 32 * i] = static_cast<uint16_t>(c0) | (static_cast<uint16_t>(c1) << 8);
    }
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_store_latent_fp8(const void* latent_bf16, const int64_t* slot_mapping, int64_t n,
                                           float k_scale, uint8_t* kv_pool_fp8, int64_t num_pages, int32_t* dev_err,
                                           void* stream) {
    if (n < 0 || num_pages < 0) return DSA_ERR_INVALID_ARG;
    if (!(k_scale > 0.0f) || !(k_scale < INFINITY)) return DSA_ERR_INVALID_ARG;
    if (n == 0) return DSA_OK;
    if (!latent_bf16 || !slot_mapping || !kv_pool_fp8) return DSA_ERR_INVALID_ARG;
    if (!dsa::aligned16(latent_bf16) || !dsa::aligned16(kv_pool_fp8)) return DSA_ERR_INVALID_ARG;
    const int64_t blocks = (n + 7) / 8;
    if (blocks > 0x7fffffffLL) return DSA_ERR_INVALID_ARG;
    dsa::store_latent_fp8_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint32_t*>(latent_bf16), slot_mapping, n, k_scale, reinterpret_cast<uint16_t*>(kv_pool_fp8),
        num_pages, dev_err);
    return dsa::launch_status();
}

// ---------------------------------------------------------------- int8 ("c8") index cache

namespace dsa {
namespace {

// One warp per token: rotate with the bf16 Hadamard / sqrt(128), quantise to int8 with one scale
// (c8_rotate_quant), write the 128 codes to row slot & 63 of page slot >> 6 and the scale, rounded
// to fp16, to the page's scale area.  Follows vllm-ascend sfa_v1.py, indexer_select_pre_process with
// use_sparse_c8_indexer (k_li @ qk_hadamard, npu_dynamic_quant, scale .to(float16)) and the
// npu_scatter_nd_update_ of codes and scales by slot_mapping.
__global__ void __launch_bounds__(256)
store_index_k_c8_kernel(const uint16_t* __restrict__ keys, const int64_t* __restrict__ slots, int64_t n,
                        uint8_t* __restrict__ pool, int64_t num_pages, int32_t* err) {
    const int64_t token = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (token >= n) return;                      // warp-uniform
    const int64_t slot = __ldg(slots + token);
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(keys + token * kIndexDim) + lane);
    if (slot < 0) return;                        // padding token
    const int64_t page = slot >> 6;
    const int row = static_cast<int>(slot & 63);
    if (page >= num_pages) {
        if (lane == 0) raise_error(err, DSA_DEVERR_SLOT_RANGE);
        return;
    }
    const float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
    float scale;
    const uint32_t packed = c8_rotate_quant(x, lane, &scale);
    uint8_t* pg = pool + page * kC8PageBytes;
    reinterpret_cast<uint32_t*>(pg + row * kIndexDim)[lane] = packed;
    if (lane == 0) reinterpret_cast<__half*>(pg + kC8ScaleOffset)[row] = __float2half_rn(scale);
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_store_index_k_c8(const void* k_bf16, const int64_t* slot_mapping, int64_t n,
                                           uint8_t* index_k_pool_c8, int64_t num_pages, int32_t page_size,
                                           int32_t* dev_err, void* stream) {
    if (n < 0 || num_pages < 0) return DSA_ERR_INVALID_ARG;
    if (page_size != dsa::kPage) return DSA_ERR_UNSUPPORTED;
    if (n == 0) return DSA_OK;
    if (!k_bf16 || !slot_mapping || !index_k_pool_c8) return DSA_ERR_INVALID_ARG;
    if (!dsa::aligned16(k_bf16) || !dsa::aligned16(index_k_pool_c8)) return DSA_ERR_INVALID_ARG;
    const int64_t blocks = (n + 7) / 8;
    if (blocks > 0x7fffffffLL) return DSA_ERR_INVALID_ARG;
    dsa::store_index_k_c8_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(k_bf16), slot_mapping, n, index_k_pool_c8, num_pages, dev_err);
    return dsa::launch_status();
}
