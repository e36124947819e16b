/*
 * dsa_oracle.c -- plain CPU oracle for the DeepSeek Sparse Attention (DSA) decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark may load this library.  The product path (the CUDA library) never calls it, and the
 * two share no code, header, table or constant.
 *
 * Every function is the plain definition written out: loops in the order the method states them,
 * double accumulation, no blocking, no fusion.  It is deliberately slow.
 *
 * Sources (web pages; each function names the passage it follows):
 *   [sfa]    vllm_ascend/attention/sfa_v1.py         (vLLM-Ascend SFA backend, DeepSeek-V3.2)
 *   [dsa]    vllm_ascend/attention/dsa_v1.py         (vLLM-Ascend DSA backend)
 *   [idx]    sglang/srt/layers/attention/dsa/dsa_indexer.py  (sglang Indexer)
 *   [mla]    vllm/v1/attention/backends/mla/common.py        (vLLM MLACommonImpl)
 *
 * Readings of points the pages leave open are stated at each function; they are the same
 * readings the CUDA path implements (stated independently there).
 *
 * Parity pins: every function here is pinned by tests under tests/ (closed forms, library
 * routines, brute force, invariants).  No function is "parity unpinned".
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fopenmp -fPIC -shared (no fast-math: the
 * quantisation steps must follow IEEE single precision exactly).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define PAGE 64          /* page size: [idx] Indexer._get_topk_paged asserts page size 64 */
#define DI 128           /* indexer head dim ([sfa] AscendSFAImpl: head_dim = 128) */
#define HI 64            /* indexer heads ([sfa] AscendSFAImpl: n_head = 64) */
#define ROW_BYTES 132    /* 128 FP8 codes + one fp32 scale ([idx] head_dim_with_sf = 132) */
#define PAGE_BYTES (PAGE * ROW_BYTES)
#define DQK 576          /* absorbed MLA query/key width: 512 latent + 64 rope ([mla] head size 576) */
#define DV 512           /* latent value width */
#define C8_PAGE_BYTES (PAGE * DI + PAGE * 2)   /* int8 cache page: 64 x 128 codes + 64 fp16 scales */

/* ---------------------------------------------------------------- number formats */

/* bf16 -> fp32 is exact: the bf16 bits are the upper half of the fp32 bits. */
static float bf16_bits_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even (the IEEE default rounding).  Written from the
 * definition: keep the upper 16 bits, look at the discarded lower 16 bits, and round up when
 * they exceed half an ulp, or equal half an ulp and the kept part is odd.  A carry out of the
 * mantissa correctly bumps the exponent (and overflows to infinity). */
uint16_t dsa_oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays a (quiet) NaN */
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xffffu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

float dsa_oracle_bf16_to_f32(uint16_t h) { return bf16_bits_to_f32(h); }

/* Round a double to the nearest bf16 (ties to even) with a single rounding: the double is first
 * narrowed to fp32 rounding toward zero with a sticky last bit ("round to odd"; fp32 keeps 16 more
 * bits than bf16, so the second rounding cannot be misled), then rounded to bf16 as above. */
uint16_t dsa_oracle_f64_to_bf16(double x) {
    if (isnan(x)) return 0x7fc0u;
    float f = (float)x;                     /* nearest fp32 */
    if ((double)f != x && !isinf(f)) {
        if (fabs((double)f) > fabs(x)) f = nextafterf(f, 0.0f);   /* truncate toward zero */
        uint32_t u;
        memcpy(&u, &f, 4);
        u |= 1u;                            /* inexact: sticky bit */
        memcpy(&f, &u, 4);
    }
    return dsa_oracle_f32_to_bf16(f);
}

void dsa_oracle_f64_to_bf16_array(const double* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = dsa_oracle_f64_to_bf16(x[i]);
}

/* OCP 8-bit floating point, E4M3 "fn" variant (the torch.float8_e4m3fn type the [idx] page uses
 * for the index-K cache; not the fnuz variant).  1 sign bit, 4 exponent bits with bias 7, 3
 * mantissa bits; exponent field 0 encodes subnormals m/8 * 2^-6; there is no infinity; the only
 * NaN patterns are S.1111.111.  Largest finite magnitude: 1.75 * 2^8 = 448. */
double dsa_oracle_e4m3_decode(uint8_t c) {
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 15;
    int m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Values of the 127 non-negative finite codes 0x00 .. 0x7e, in increasing order (the E4M3FN
 * encoding is monotonic for non-negative values), filled from the decoder when the library loads. */
static double e4m3_pos_values[127];

__attribute__((constructor)) static void e4m3_table_init(void) {
    for (int c = 0; c <= 0x7e; ++c) e4m3_pos_values[c] = dsa_oracle_e4m3_decode((uint8_t)c);
}

/* fp32 -> E4M3FN, round to nearest with ties to even code, saturating to +-448 (no value maps to
 * NaN except NaN).  Find the two codes whose values bracket |x| (binary search in the increasing
 * table of non-negative code values) and take the nearer one; on an exact tie take the one whose
 * code is even (an even code has an even mantissa LSB).  The sign bit is kept, so -0 and negative
 * values that round to zero give code 0x80. */
uint8_t dsa_oracle_e4m3_encode(float x) {
    if (isnan(x)) return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7e);
    /* lo = largest code with value <= a (exists: code 0 has value 0 <= a) */
    int lo = 0, hi = 0x7e;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (e4m3_pos_values[mid] <= a) lo = mid; else hi = mid - 1;
    }
    double vlo = e4m3_pos_values[lo];
    double vhi = e4m3_pos_values[lo + 1];
    double dlo = a - vlo, dhi = vhi - a;
    int c;
    if (dlo < dhi) c = lo;
    else if (dhi < dlo) c = lo + 1;
    else c = (lo & 1) ? lo + 1 : lo;
    return (uint8_t)(sign | c);
}

/* ---------------------------------------------------------------- Hadamard rotation */

/* Unnormalised fast Walsh-Hadamard transform of a 128-vector in fp32, Sylvester (natural)
 * order: for h = 1, 2, 4, ..., 64, every pair (j, j+h) inside each block of 2h becomes
 * (a+b, a-b).  This equals multiplication by the Sylvester matrix H_128, the matrix
 * scipy.linalg.hadamard(128) builds ([sfa] qk_hadamard; [dsa] hadamard_transform_ref multiplies
 * by that matrix).  The butterfly order is part of the definition here: it fixes the fp32
 * rounding of every intermediate. */
void dsa_oracle_fwht128(float* x) {
    for (int h = 1; h < DI; h <<= 1) {
        for (int i = 0; i < DI; i += 2 * h) {
            for (int j = i; j < i + h; ++j) {
                float a = x[j];
                float b = x[j + h];
                x[j] = a + b;
                x[j + h] = a - b;
            }
        }
    }
}

/* Rotation of one bf16 128-vector ([idx] rotate_activation: hadamard_transform(x, scale =
 * 128^-0.5); [dsa] rotate_activation = hadamard_transform_ref(x, H, 128^-0.5)): fp32 butterflies,
 * one multiply by the fp32 value of 1/sqrt(128), round to bf16 (the pages keep the rotated
 * activation in the input dtype, bf16).  Output: the rotated values as bf16 bits. */
void dsa_oracle_rotate128(const uint16_t* in_bf16, uint16_t* out_bf16) {
    const float inv_sqrt_n = (float)(1.0 / sqrt((double)DI));
    float x[DI];
    for (int d = 0; d < DI; ++d) x[d] = bf16_bits_to_f32(in_bf16[d]);
    dsa_oracle_fwht128(x);
    for (int d = 0; d < DI; ++d) out_bf16[d] = dsa_oracle_f32_to_bf16(x[d] * inv_sqrt_n);
}

/* ---------------------------------------------------------------- FP8 quantisation */

/* Per-128-vector FP8 quantisation ([idx] act_quant(x, block_size=128): one scale per block of
 * 128 values, which for a 128-wide key or query head is one scale per token / per head).
 * Reading of the unprinted formula: amax = max |y|; scale = max(amax, 1e-4) / 448 in fp32 with
 * IEEE division; code = E4M3FN(y / scale) with IEEE fp32 division then round-to-nearest-even and
 * saturation.  The scale is plain fp32 (no power-of-two rounding). */
/* Quantisation with the scale format of act_quant's scale_fmt ([idx] Indexer(scale_fmt=...),
 * act_quant(x, block_size, scale_fmt); the rule itself is not printed).  Reading: plain format:
 * the fp32 scale above; "ue8m0" (an unsigned 8-bit exponent, no mantissa): the smallest power of
 * two >= that fp32 scale, so that every |y / scale| <= 448 still holds. */
static float pow2_at_least(float s) {
    int e;
    const float m = frexpf(s, &e); /* s = m * 2^e, m in [0.5, 1) */
    return m == 0.5f ? s : ldexpf(1.0f, e);
}

void dsa_oracle_quant128_fmt(const float* y, uint8_t* codes, float* scale, int ue8m0) {
    float amax = 0.0f;
    for (int d = 0; d < DI; ++d) {
        float a = fabsf(y[d]);
        if (a > amax) amax = a;
    }
    float s = fmaxf(amax, 1e-4f) / 448.0f;
    if (ue8m0) s = pow2_at_least(s);
    for (int d = 0; d < DI; ++d) {
        float t = y[d] / s;
        codes[d] = dsa_oracle_e4m3_encode(t);
    }
    *scale = s;
}

void dsa_oracle_quant128(const float* y, uint8_t* codes, float* scale) { dsa_oracle_quant128_fmt(y, codes, scale, 0); }

/* ---------------------------------------------------------------- index-K store */

/* Store new indexer keys into the paged FP8 cache ([idx] Indexer._store_index_k_cache:
 * fused_store_index_k_cache(key, buf, out_cache_loc, page_size), or act_quant followed by
 * set_index_k_scale_buffer; [sfa] scatter of the quantised key by slot_mapping).
 * Steps per token: rotate (Hadamard, bf16), quantise (per token), scatter to slot.
 * slot < 0 is a padding slot and is skipped ([sfa] pads slot_mapping with -1).
 * Page layout (reading: the pages fix 132 bytes per token and 64 tokens per page but not the
 * order inside a page): page-blocked, bytes [0, 8192) hold the 64 x 128 codes row by row,
 * bytes [8192, 8448) hold the 64 fp32 scales.
 * Returns the number of tokens whose slot pointed past the pool (those are skipped). */
/* Quantise one bf16 key (rotated first when `rotate`) into its slot; returns 1 when the slot is
 * past the pool (nothing written), else 0. */
static int store_one(const uint16_t* key, int rotate, int ue8m0, int64_t slot, uint8_t* pool, int64_t num_pages) {
    int64_t page = slot / PAGE, row = slot % PAGE;
    if (page >= num_pages) return 1;
    uint16_t rot[DI];
    float y[DI];
    uint8_t codes[DI];
    float s;
    if (rotate) dsa_oracle_rotate128(key, rot);
    else memcpy(rot, key, sizeof(rot));
    for (int d = 0; d < DI; ++d) y[d] = bf16_bits_to_f32(rot[d]);
    dsa_oracle_quant128_fmt(y, codes, &s, ue8m0);
    uint8_t* pg = pool + page * PAGE_BYTES;
    memcpy(pg + row * DI, codes, DI);
    memcpy(pg + PAGE * DI + row * 4, &s, 4);
    return 0;
}

int64_t dsa_oracle_store_index_k(const uint16_t* k_bf16, const int64_t* slot_mapping, int64_t n,
                                 uint8_t* pool, int64_t num_pages) {
    int64_t bad = 0;
    for (int64_t t = 0; t < n; ++t) {
        if (slot_mapping[t] < 0) continue;
        bad += store_one(k_bf16 + t * DI, 1, 0, slot_mapping[t], pool, num_pages);
    }
    return bad;
}

/* ---------------------------------------------------------------- indexer key / query prologues */

/* Norm of one bf16 128-vector ([idx] Indexer.k_norm: LayerNorm(head_dim) with weight and bias,
 * eps = k_norm.variance_epsilon, or RMSNorm(head_dim) when the config's index_k_norm_type is
 * "rms"; [sfa] indexer_select_pre_process: k_li = k_norm(wk(x))).
 * LayerNorm: mean = sum(x) / 128; d = x - mean; var = sum(d * d) / 128; rstd = 1 / sqrt(var + eps);
 * y = (d * rstd) * w + b.  RMSNorm: ms = sum(x * x) / 128; rstd = 1 / sqrt(ms + eps);
 * y = (x * rstd) * w.  Reading: the pages do not print the norm kernel, so the definition is the
 * exact one: every step in float64 (standing in for exact arithmetic; the sums run in index
 * order), and the result rounded once to bf16, the dtype of the k_norm output the pages pass on. */
void dsa_oracle_k_norm128(const uint16_t* in_bf16, const float* w, const float* b, float eps, int rms,
                          uint16_t* out_bf16) {
    double x[DI];
    for (int d = 0; d < DI; ++d) x[d] = (double)bf16_bits_to_f32(in_bf16[d]);
    if (rms) {
        double ss = 0.0;
        for (int d = 0; d < DI; ++d) ss += x[d] * x[d];
        const double rstd = 1.0 / sqrt(ss / DI + (double)eps);
        for (int d = 0; d < DI; ++d) out_bf16[d] = dsa_oracle_f64_to_bf16((x[d] * rstd) * (double)w[d]);
        return;
    }
    double sum = 0.0;
    for (int d = 0; d < DI; ++d) sum += x[d];
    const double mean = sum / DI;
    double sq = 0.0;
    for (int d = 0; d < DI; ++d) sq += (x[d] - mean) * (x[d] - mean);
    const double rstd = 1.0 / sqrt(sq / DI + (double)eps);
    for (int d = 0; d < DI; ++d)
        out_bf16[d] = dsa_oracle_f64_to_bf16(((x[d] - mean) * rstd) * (double)w[d] + (double)b[d]);
}

/* Rotary embedding of the first 64 dims of one bf16 128-vector ([idx] rotary_emb with rotary_dim
 * = rope_head_dim = 64 on the split [64 rope, 64 nope], fused_q_indexer_rope_first_quant;
 * [sfa] npu_rotary_mul / rope_forward_triton_siso).  cs = the position's row of cos_sin_cache,
 * cos in cs[0:32] and sin in cs[32:64] ([idx] NPU path: cos_sin_cache[positions].chunk(2)).
 * neox style (default): pairs (i, i + 32): y_i = x_i c_i - x_{i+32} s_i,
 * y_{i+32} = x_{i+32} c_i + x_i s_i; interleaved style ([sfa] GLM models): pairs (2i, 2i + 1).
 * Reading: fp32 products and sum without fused multiply-add, rounded to bf16; dims 64 .. 127 pass
 * through. */
void dsa_oracle_rope64(const uint16_t* in_bf16, const float* cs, int neox, uint16_t* out_bf16) {
    memcpy(out_bf16, in_bf16, DI * sizeof(uint16_t));
    for (int i = 0; i < 32; ++i) {
        const int ia = neox ? i : 2 * i, ib = neox ? i + 32 : 2 * i + 1;
        const float a = bf16_bits_to_f32(in_bf16[ia]), b = bf16_bits_to_f32(in_bf16[ib]);
        const float c = cs[i], sn = cs[32 + i];
        const float ya = a * c - b * sn;
        const float yb = b * c + a * sn;
        out_bf16[ia] = dsa_oracle_f32_to_bf16(ya);
        out_bf16[ib] = dsa_oracle_f32_to_bf16(yb);
    }
}

/* Key prologue and store.  With `rotate` ([idx] Indexer._get_k_bf16, the path without indexer
 * fusion: k_norm, rotary_emb on the rope dims, rotate_activation, then _store_index_k_cache):
 * norm, rotary embedding at the token's position, then the store above (rotate, quantise,
 * scatter).  Without it ([idx] Indexer._fused_k_prepare_and_store:
 * fused_k_indexer_norm_rope_store(key_raw, buffer, out_cache_loc, k_norm.weight, k_norm.bias,
 * eps, cos_sin_cache, positions, page_size); Indexer._maybe_rotate: the fused path drops the
 * Hadamard rotation, which is orthogonal and applied to both sides): norm, rotary embedding,
 * quantise, scatter.  A position outside [0, max_pos) skips the token.  Returns the number of
 * skipped tokens (slot past the pool or position out of range). */
int64_t dsa_oracle_store_index_k_prologue(const uint16_t* k_raw, const float* w, const float* b, float eps, int rms,
                                          const float* cos_sin, int64_t max_pos, const int64_t* positions,
                                          int neox, int rotate, int ue8m0, const int64_t* slot_mapping,
                                          int64_t n, uint8_t* pool, int64_t num_pages) {
    int64_t bad = 0;
    for (int64_t t = 0; t < n; ++t) {
        if (slot_mapping[t] < 0) continue;
        if (positions[t] < 0 || positions[t] >= max_pos) { ++bad; continue; }
        uint16_t nrm[DI], rop[DI];
        dsa_oracle_k_norm128(k_raw + t * DI, w, b, eps, rms, nrm);
        dsa_oracle_rope64(nrm, cos_sin + positions[t] * 64, neox, rop);
        bad += store_one(rop, rotate, ue8m0, slot_mapping[t], pool, num_pages);
    }
    return bad;
}

/* Query rotary embedding ([idx] fused_q_indexer_rope_first_quant(q, weights, gate, cos_sin_cache,
 * positions): the rope part; the Hadamard rotation and per-head quantisation that follow are the
 * logits call's query prologue): every head of row t at positions[t].  A row whose position is
 * outside [0, max_pos) is copied unchanged.  Returns the number of such rows. */
int64_t dsa_oracle_rope_q(const uint16_t* q_raw, const float* cos_sin, int64_t max_pos, const int64_t* positions,
                          int neox, int64_t T, uint16_t* out) {
    int64_t bad = 0;
    for (int64_t t = 0; t < T; ++t) {
        const int ok = positions[t] >= 0 && positions[t] < max_pos;
        if (!ok) ++bad;
        for (int h = 0; h < HI; ++h) {
            const uint16_t* src = q_raw + (t * HI + h) * DI;
            uint16_t* dst = out + (t * HI + h) * DI;
            if (ok) dsa_oracle_rope64(src, cos_sin + positions[t] * 64, neox, dst);
            else memcpy(dst, src, DI * sizeof(uint16_t));
        }
    }
    return bad;
}

/* ---------------------------------------------------------------- causal visibility */

/* Request of global query row r: the b with cu_q[b] <= r < cu_q[b+1]. */
static int row_request(const int32_t* cu_q, int32_t B, int64_t r) {
    for (int b = 0; b < B; ++b)
        if (r >= cu_q[b] && r < cu_q[b + 1]) return b;
    return -1;
}

/* Visible keys of query row r ([idx] ragged key ends ke = start + pos + 1; next_n query tokens of
 * a request are its last next_n positions; NPU sparse_mode=3 is causal).  Row j of request b
 * (q_len_b rows, seq_lens[b] cached tokens including this step's) sits at absolute position
 * p = seq_lens[b] - q_len_b + j and sees keys [0, p]. */
int32_t dsa_oracle_visible_len(const int32_t* seq_lens, const int32_t* cu_q, int32_t B, int64_t r) {
    int b = row_request(cu_q, B, r);
    if (b < 0) return 0;
    int32_t q_len = cu_q[b + 1] - cu_q[b];
    int64_t j = r - cu_q[b];
    int64_t v = (int64_t)seq_lens[b] - q_len + j + 1;
    if (v < 0) v = 0;
    return (int32_t)v;
}

/* Visible entries of a compressed cache ([dsa] AscendDSAImpl._forward_decode with compress_ratio
 * 4: npu_vllm_quant_lightning_indexer(..., actual_seq_lengths_key = seq_lens, sparse_mode = 3,
 * cmp_ratio = 4) and the attention's cmp_mask_mode = 3).  Reading: compressed entry e stands for
 * the tokens [ratio e, ratio e + ratio) and a row sees it once all of them are visible, i.e. the
 * row's visible length (above) divided by the ratio, rounded down. */
int32_t dsa_oracle_visible_len_cmp(const int32_t* seq_lens, const int32_t* cu_q, int32_t B, int64_t r,
                                   int32_t ratio) {
    return dsa_oracle_visible_len(seq_lens, cu_q, B, r) / ratio;
}

/* ---------------------------------------------------------------- indexer logits */

/* Lightning-indexer logits over the paged FP8 cache ([idx] Indexer._get_topk_paged: paged MQA
 * logits over block_table / seq_lens with the head gate from _get_logits_head_gate; [sfa]
 * npu_lightning_indexer):
 *     I[r,s] = sum_h w'[r,h] * ReLU(k_scale[s] * sum_d dec(cq[r,h,d]) * dec(ck[s,d]))
 * with w'[r,h] = w[r,h] * q_scale[r,h] (the query scale folded into the head gate, as
 * _get_logits_head_gate multiplies the gate by q_scale) and the query quantised per head by the
 * same per-128 rule as the keys.  The input w already carries n_heads^-0.5 * head_dim^-0.5.
 * q_mode bit 0 first rotates each query head (the pages rotate q before quantising it); bit 1
 * quantises the query with the ue8m0 scale format (see dsa_oracle_quant128_fmt).
 * Computed in double, rounded once to fp32.  Only s < v_r is written.
 * rows[i] lists the global rows to compute; output row i goes to logits[i*ld ...].
 * mag (nullable, double [n_rows, ld]) receives sum_h |w'| * ReLU(...), the magnitude of the
 * terms, which bounds the rounding error of any evaluation order.
 * Returns the number of (row, key) pairs skipped because the page id was out of range. */
/* With cmp_ratio > 1 the cache holds compressed entries and row r scores entries
 * s < dsa_oracle_visible_len_cmp(r) (the DSV4 indexer over the compressed index keys, [dsa]
 * indexer_select_qli / npu_vllm_quant_lightning_indexer(..., cmp_ratio = 4)). */
int64_t dsa_oracle_indexer_logits_cmp(const uint16_t* q_bf16, const float* w, const uint8_t* pool,
                                      int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                      const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                                      int32_t q_mode, int32_t cmp_ratio, const int64_t* rows, int64_t n_rows,
                                      float* logits, int64_t ld, double* mag) {
    int64_t bad = 0;
    for (int64_t i = 0; i < n_rows; ++i) {
        int64_t r = rows[i];
        int b = row_request(cu_q, B, r);
        if (b < 0) continue;
        int32_t v = dsa_oracle_visible_len_cmp(seq_lens, cu_q, B, r, cmp_ratio);
        /* query prologue: per head, optional rotation, then per-128 quantisation */
        uint8_t cq[HI][DI];
        double wq[HI];
        for (int h = 0; h < HI; ++h) {
            const uint16_t* src = q_bf16 + (r * HI + h) * DI;
            uint16_t rot[DI];
            float y[DI];
            float sq;
            if (q_mode & 1) {
                dsa_oracle_rotate128(src, rot);
                src = rot;
            }
            for (int d = 0; d < DI; ++d) y[d] = bf16_bits_to_f32(src[d]);
            dsa_oracle_quant128_fmt(y, cq[h], &sq, (q_mode >> 1) & 1);
            wq[h] = (double)w[r * HI + h] * (double)sq;
        }
        double dq[HI][DI];
        for (int h = 0; h < HI; ++h)
            for (int d = 0; d < DI; ++d) dq[h][d] = dsa_oracle_e4m3_decode(cq[h][d]);
        int64_t row_bad = 0;
#pragma omp parallel for schedule(static) reduction(+ : row_bad)
        for (int64_t s = 0; s < v; ++s) {
            int64_t lp = s / PAGE;
            int32_t page = (lp < max_pages) ? block_table[(int64_t)b * max_pages + lp] : -1;
            if (page < 0 || page >= num_pages) { ++row_bad; continue; }
            const uint8_t* pg = pool + (int64_t)page * PAGE_BYTES;
            const uint8_t* ck = pg + (s % PAGE) * DI;
            float ks;
            memcpy(&ks, pg + PAGE * DI + (s % PAGE) * 4, 4);
            double dk[DI];
            for (int d = 0; d < DI; ++d) dk[d] = dsa_oracle_e4m3_decode(ck[d]);
            double acc = 0.0, accm = 0.0;
            for (int h = 0; h < HI; ++h) {
                double dot = 0.0;
                for (int d = 0; d < DI; ++d) dot += dq[h][d] * dk[d];
                double relu = (double)ks * dot;
                if (relu < 0.0) relu = 0.0;
                acc += wq[h] * relu;
                accm += fabs(wq[h]) * relu;
            }
            logits[i * ld + s] = (float)acc;
            if (mag) mag[i * ld + s] = accm;
        }
        bad += row_bad;
    }
    return bad;
}

int64_t dsa_oracle_indexer_logits(const uint16_t* q_bf16, const float* w, const uint8_t* pool,
                                  int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                  const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                                  int32_t q_mode, const int64_t* rows, int64_t n_rows,
                                  float* logits, int64_t ld, double* mag) {
    return dsa_oracle_indexer_logits_cmp(q_bf16, w, pool, num_pages, block_table, max_pages, seq_lens, cu_q, B,
                                         q_mode, 1, rows, n_rows, logits, ld, mag);
}

/* ---------------------------------------------------------------- int8 ("c8") index-K cache */

/* IEEE binary16 (torch.float16): 1 sign bit, 5 exponent bits with bias 15, 10 mantissa bits;
 * exponent field 0 encodes subnormals m * 2^-24; field 31 encodes infinity (m = 0) and NaN. */
double dsa_oracle_f16_decode(uint16_t h) {
    int e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(1024 + m), e - 25);
    return (h & 0x8000) ? -v : v;
}

/* fp32 -> fp16, round to nearest with ties to even, overflow to infinity (the IEEE default that
 * torch's .to(float16) follows).  From the definition: the fp16 grid spacing in the binade of |x|
 * is 2^(e-10) for exponents e >= -14 and 2^-24 below (subnormals); divide by it (exact, a power of
 * two), round to an integer with ties to even, multiply back, and encode that value (a carry into
 * the next binade is encoded there; anything from 65520 up has become infinity). */
uint16_t dsa_oracle_f32_to_f16(float x) {
    const uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return 0x7e00;
    if (isinf(x)) return sign | 0x7c00;
    const double a = fabs((double)x);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                    /* a in [2^(e-1), 2^e) */
    int ue = e - 1;
    if (ue < -14) ue = -14;
    const double ulp = ldexp(1.0, ue - 10);
    const double v = nearbyint(a / ulp) * ulp;   /* default rounding mode: nearest, ties to even */
    if (v < ldexp(1.0, -14)) return sign | (uint16_t)(v / ldexp(1.0, -24));
    frexp(v, &e);
    ue = e - 1;
    if (ue > 15) return sign | 0x7c00;
    const int m = (int)(v / ldexp(1.0, ue - 10)) - 1024;
    return sign | (uint16_t)(((ue + 15) << 10) | m);
}

/* The c8 rotation ([sfa] AscendSFAImpl: qk_hadamard = torch.tensor(scipy.linalg.hadamard(128),
 * dtype=bf16) / 128**0.5, so every entry is +-c with c = bf16(128^-0.5) = 181 * 2^-11; the c8 path
 * multiplies k_li and every query head q_li by it in bf16):
 *     y_j = bf16( sum_i x_i * H[i][j] ),   H[i][j] = c * (-1)^popcount(i & j)  (Sylvester order).
 * Reading: the bf16 matmul is the exact dot product rounded once to bf16 (float64 stands in for the
 * exact sum, in index order). */
void dsa_oracle_c8_rotate128(const uint16_t* in_bf16, uint16_t* out_bf16) {
    const double c = (double)bf16_bits_to_f32(dsa_oracle_f64_to_bf16(1.0 / sqrt(128.0)));
    double x[DI];
    for (int i = 0; i < DI; ++i) x[i] = (double)bf16_bits_to_f32(in_bf16[i]);
    for (int j = 0; j < DI; ++j) {
        double acc = 0.0;
        for (int i = 0; i < DI; ++i) {
            int par = 0;
            for (int t = i & j; t; t >>= 1) par ^= t & 1;
            acc += (par ? -c : c) * x[i];
        }
        out_bf16[j] = dsa_oracle_f64_to_bf16(acc);
    }
}

/* Dynamic symmetric int8 quantisation of one vector ([sfa] torch_npu.npu_dynamic_quant(x.view(-1,
 * 128), dst_type=int8): one scale per row, i.e. per key token and per (query token, head); the
 * scale comes back in fp32 and is cast to fp16 for the cache and the logits call).  The formula is
 * not printed; reading: amax = max |y|; scale = amax / 127 (fp32, IEEE division); code =
 * round-to-nearest-even(y / scale) (fp32 IEEE division), so |code| <= 127; a vector of zeros has
 * scale 0 and codes 0.  The codes use the fp32 scale; only the stored scale is rounded to fp16. */
void dsa_oracle_quant_int8(const float* y, int n, int8_t* codes, float* scale) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(y[i]);
        if (a > amax) amax = a;
    }
    const float s = amax / 127.0f;
    *scale = s;
    for (int i = 0; i < n; ++i) {
        if (s == 0.0f) {
            codes[i] = 0;
            continue;
        }
        const float q = rintf(y[i] / s);
        codes[i] = (int8_t)(q > 127.0f ? 127.0f : (q < -127.0f ? -127.0f : q));
    }
}

/* Store new indexer keys into the paged int8 cache ([sfa] indexer_select_pre_process with
 * use_sparse_c8_indexer: k_li @ qk_hadamard, npu_dynamic_quant per token, scale to fp16; then
 * npu_scatter_nd_update_ of the codes into kv_cache[2] and of the scales into kv_cache[3] by
 * slot_mapping).  slot < 0 is padding and is skipped.  Page layout (reading: the pages keep codes
 * [pages, 64, 1, 128] int8 and scales [pages, 64, 1, 1] fp16 as two tensors; here one page-blocked
 * pool like the FP8 cache): bytes [0, 8192) hold the 64 x 128 codes row by row, bytes
 * [8192, 8320) the 64 fp16 scales.  Returns the number of tokens whose slot pointed past the pool. */
int64_t dsa_oracle_store_index_k_c8(const uint16_t* k_bf16, const int64_t* slot_mapping, int64_t n,
                                    uint8_t* pool, int64_t num_pages) {
    /* every token's codes and scale (independent per token), then the scatter in token order */
    int8_t* codes = (int8_t*)malloc((size_t)(n > 0 ? n : 1) * DI);
    uint16_t* sc16 = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(n > 0 ? n : 1));
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        if (slot_mapping[t] < 0 || slot_mapping[t] / PAGE >= num_pages) continue;
        uint16_t rot[DI];
        float y[DI], sc;
        dsa_oracle_c8_rotate128(k_bf16 + t * DI, rot);
        for (int d = 0; d < DI; ++d) y[d] = bf16_bits_to_f32(rot[d]);
        dsa_oracle_quant_int8(y, DI, codes + t * DI, &sc);
        sc16[t] = dsa_oracle_f32_to_f16(sc);
    }
    int64_t bad = 0;
    for (int64_t t = 0; t < n; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        const int64_t page = slot / PAGE;
        if (page >= num_pages) {
            ++bad;
            continue;
        }
        uint8_t* pg = pool + page * C8_PAGE_BYTES;
        memcpy(pg + (slot % PAGE) * DI, codes + t * DI, DI);
        pg[PAGE * DI + (slot % PAGE) * 2] = (uint8_t)(sc16[t] & 0xff);
        pg[PAGE * DI + (slot % PAGE) * 2 + 1] = (uint8_t)(sc16[t] >> 8);
    }
    free(codes);
    free(sc16);
    return bad;
}

/* Lightning-indexer logits over the int8 cache ([sfa] indexer_select_post_process with
 * use_sparse_c8_indexer: the query heads rotated by qk_hadamard and quantised per (token, head) by
 * npu_dynamic_quant, the weights cast to fp16, then npu_lightning_indexer_quant(query, key, weights,
 * query_dequant_scale, key_dequant_scale, ..., query_quant_mode=0, key_quant_mode=0)).  Reading: the
 * lightning-indexer score on the dequantised query and key,
 *     I[r,s] = sum_h w16[r,h] * ReLU( qs16[r,h] * ks16[s] * sum_d cq[r,h,d] * ck[s,d] ),
 * with w16, qs16, ks16 the fp16 weight and scales.  Computed in double (the integer dot product is
 * exact), rounded once to fp32; only s < v_r is written.  mag as in dsa_oracle_indexer_logits.
 * Returns the number of (row, key) pairs skipped because the page id was out of range. */
int64_t dsa_oracle_indexer_logits_c8(const uint16_t* q_bf16, const float* w, const uint8_t* pool,
                                     int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                     const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                                     const int64_t* rows, int64_t n_rows, float* logits, int64_t ld,
                                     double* mag) {
    int64_t bad = 0;
    for (int64_t i = 0; i < n_rows; ++i) {
        const int64_t r = rows[i];
        const int b = row_request(cu_q, B, r);
        if (b < 0) continue;
        const int32_t v = dsa_oracle_visible_len(seq_lens, cu_q, B, r);
        int8_t cq[HI][DI];
        double wq[HI], qs[HI];
        for (int h = 0; h < HI; ++h) {
            uint16_t rot[DI];
            float y[DI], sc;
            dsa_oracle_c8_rotate128(q_bf16 + (r * HI + h) * DI, rot);
            for (int d = 0; d < DI; ++d) y[d] = bf16_bits_to_f32(rot[d]);
            dsa_oracle_quant_int8(y, DI, cq[h], &sc);
            qs[h] = dsa_oracle_f16_decode(dsa_oracle_f32_to_f16(sc));
            wq[h] = dsa_oracle_f16_decode(dsa_oracle_f32_to_f16(w[r * HI + h]));
        }
        int64_t row_bad = 0;
#pragma omp parallel for schedule(static) reduction(+ : row_bad)
        for (int64_t s = 0; s < v; ++s) {
            const int64_t lp = s / PAGE;
            const int32_t page = (lp < max_pages) ? block_table[(int64_t)b * max_pages + lp] : -1;
            if (page < 0 || page >= num_pages) {
                ++row_bad;
                continue;
            }
            const uint8_t* pg = pool + (int64_t)page * C8_PAGE_BYTES;
            const int8_t* ck = (const int8_t*)(pg + (s % PAGE) * DI);
            const uint16_t kh = (uint16_t)(pg[PAGE * DI + (s % PAGE) * 2] | (pg[PAGE * DI + (s % PAGE) * 2 + 1] << 8));
            const double ks = dsa_oracle_f16_decode(kh);
            double acc = 0.0, accm = 0.0;
            for (int h = 0; h < HI; ++h) {
                int64_t dot = 0;
                for (int d = 0; d < DI; ++d) dot += (int64_t)cq[h][d] * (int64_t)ck[d];
                double relu = qs[h] * ks * (double)dot;
                if (relu < 0.0) relu = 0.0;
                acc += wq[h] * relu;
                accm += fabs(wq[h]) * relu;
            }
            logits[i * ld + s] = (float)acc;
            if (mag) mag[i * ld + s] = accm;
        }
        bad += row_bad;
    }
    return bad;
}

/* ---------------------------------------------------------------- top-k */

typedef struct {
    float v;
    int32_t s;
} keyed_t;

/* Total order used by the selection: larger value first; -0 equals +0; NaN after every number;
 * equal values keep the lower index first (a stable descending sort). */
static int cmp_desc_stable(const void* pa, const void* pb) {
    const keyed_t* a = (const keyed_t*)pa;
    const keyed_t* b = (const keyed_t*)pb;
    int na = isnan(a->v), nb = isnan(b->v);
    if (na != nb) return na ? 1 : -1;
    if (!na) {
        if (a->v > b->v) return -1;
        if (a->v < b->v) return 1;
    }
    return (a->s < b->s) ? -1 : (a->s > b->s) ? 1 : 0;
}

static int cmp_i32(const void* pa, const void* pb) {
    int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    return (a < b) ? -1 : (a > b) ? 1 : 0;
}

/* Per-row top-k ([idx] forward_indexer: logits.topk(min(topk, seq_len)) then pad with -1 to the
 * top-k width; _get_topk_paged pads rows it did not score with -1).  Readings: the kept set is
 * the first min(k, v) entries of a stable descending sort of I[r, 0:v) (lower index wins ties),
 * returned in ascending index order, padded with -1 to k.  rows[i] gives the global row (for its
 * visible length); logits row i is logits[i*ld ...]. */
/* With cmp_ratio > 1 the row's visible length is that of the compressed entries. */
void dsa_oracle_topk_cmp(const float* logits, int64_t ld, const int32_t* seq_lens, const int32_t* cu_q,
                         int32_t B, const int64_t* rows, int64_t n_rows, int32_t k, int32_t cmp_ratio, int32_t* idx) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n_rows; ++i) {
        int32_t v = dsa_oracle_visible_len_cmp(seq_lens, cu_q, B, rows[i], cmp_ratio);
        int32_t* out = idx + i * (int64_t)k;
        keyed_t* keys = (keyed_t*)malloc(sizeof(keyed_t) * (size_t)(v > 0 ? v : 1));
        for (int32_t s = 0; s < v; ++s) {
            keys[s].v = logits[i * ld + s];
            keys[s].s = s;
        }
        qsort(keys, (size_t)v, sizeof(keyed_t), cmp_desc_stable);
        int32_t n = v < k ? v : k;
        for (int32_t j = 0; j < n; ++j) out[j] = keys[j].s;
        qsort(out, (size_t)n, sizeof(int32_t), cmp_i32);
        for (int32_t j = n; j < k; ++j) out[j] = -1;
        free(keys);
    }
}

void dsa_oracle_topk(const float* logits, int64_t ld, const int32_t* seq_lens, const int32_t* cu_q,
                     int32_t B, const int64_t* rows, int64_t n_rows, int32_t k, int32_t* idx) {
    dsa_oracle_topk_cmp(logits, ld, seq_lens, cu_q, B, rows, n_rows, k, 1, idx);
}

/* ---------------------------------------------------------------- sparse MLA */

/* Physical latent-cache row of logical position pos of request b, or -1 when the block table
 * does not map it (one block table, page size 64, serves both caches: [sfa] passes the same
 * block_table to the indexer and to the sparse attention). */
static int64_t latent_row(const int32_t* block_table, int32_t max_pages, int64_t num_pages, int b,
                          int64_t pos) {
    int64_t lp = pos / PAGE;
    if (lp >= max_pages) return -1;
    int32_t page = block_table[(int64_t)b * max_pages + lp];
    if (page < 0 || page >= num_pages) return -1;
    return (int64_t)page * PAGE + pos % PAGE;
}

/* Attention of one (row, head) over a list of latent rows (absorbed MLA, [mla]
 * MLACommonImpl.forward decode branch: q = [ql_nope (512), q_pe (64)] against the 576-wide
 * latent cache rows; key and value are the same latent vector, the value is its first 512 dims;
 * one shared KV head).  S_i = scale * <q, c_i>; P = softmax(S); o = sum_i P_i c_i[0:512];
 * lse = max S + log sum exp(S - max S).  No valid row: o = 0, lse = -inf (reading). */
static void attend_rows(const uint16_t* qh, const uint16_t* kv, const int64_t* g, int64_t n,
                        double scale, double* o, double* lse, double* ssum_out) {
    for (int d = 0; d < DV; ++d) o[d] = 0.0;
    if (n == 0) {
        *lse = -INFINITY;
        if (ssum_out) *ssum_out = 0.0;
        return;
    }
    double q[DQK];
    for (int d = 0; d < DQK; ++d) q[d] = (double)bf16_bits_to_f32(qh[d]);
    double* S = (double*)malloc(sizeof(double) * (size_t)n);
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        const uint16_t* c = kv + g[i] * DQK;
        double dot = 0.0;
        for (int d = 0; d < DQK; ++d) dot += q[d] * (double)bf16_bits_to_f32(c[d]);
        S[i] = scale * dot;
        if (S[i] > m) m = S[i];
    }
    double l = 0.0;
    for (int64_t i = 0; i < n; ++i) l += exp(S[i] - m);
    double psum = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double p = exp(S[i] - m) / l;
        psum += p;
        const uint16_t* c = kv + g[i] * DQK;
        for (int d = 0; d < DV; ++d) o[d] += p * (double)bf16_bits_to_f32(c[d]);
    }
    *lse = m + log(l);
    if (ssum_out) *ssum_out = psum;
    free(S);
}

/* Sparse MLA decode over the selected positions ([sfa] npu_sparse_flash_attention with
 * sparse_indices = top-k, sparse_block_size = 1, block_table; [mla] decode returns (out, lse)).
 * idx[r, :] holds logical positions within the request; -1 entries are padding; an entry outside
 * [0, v_r) or on an unmapped page is skipped (counted in the return value).
 * q: [T, H, 576] bf16; kv: [num_pages, 64, 576] bf16; out: double [n_rows, H, 512];
 * lse: double [n_rows, H]; psum (nullable): double [n_rows, H], the sum of the softmax weights. */
int64_t dsa_oracle_sparse_mla(const uint16_t* q_bf16, const uint16_t* kv, int64_t num_pages,
                              const int32_t* block_table, int32_t max_pages, const int32_t* seq_lens,
                              const int32_t* cu_q, int32_t B, const int32_t* idx, int32_t k,
                              int32_t H, double scale, const int64_t* rows, int64_t n_rows,
                              double* out, double* lse, double* psum) {
    int64_t bad_total = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad_total)
    for (int64_t i = 0; i < n_rows * H; ++i) {
        int64_t ri = i / H;
        int h = (int)(i % H);
        int64_t r = rows[ri];
        int b = row_request(cu_q, B, r);
        int32_t v = dsa_oracle_visible_len(seq_lens, cu_q, B, r);
        int64_t* g = (int64_t*)malloc(sizeof(int64_t) * (size_t)k);
        int64_t n = 0, bad = 0;
        for (int32_t j = 0; j < k; ++j) {
            int32_t pos = idx[r * (int64_t)k + j];
            if (pos < 0) continue;
            int64_t gr = (b >= 0 && pos < v) ? latent_row(block_table, max_pages, num_pages, b, pos) : -1;
            if (gr < 0) { ++bad; continue; }
            g[n++] = gr;
        }
        attend_rows(q_bf16 + (r * H + h) * DQK, kv, g, n, scale, out + (ri * H + h) * DV,
                    lse + ri * H + h, psum ? psum + ri * H + h : NULL);
        free(g);
        if (h == 0) bad_total += bad;
    }
    return bad_total;
}

/* ---------------------------------------------------------------- DSV4: window + compressed entries + sinks */

/* Decode attention of the compressed-KV variant with compress ratio 4 ([dsa]
 * AscendDSAImpl._forward_decode: attn_op(q, ori_kv = swa_kv_cache, cmp_kv = compress_kv_cache,
 * cmp_sparse_indices = compress_topk_idxs, ori_block_table, cmp_block_table, seqused_kv = seq_lens,
 * sinks = attn_sink, softmax_scale, cmp_ratio = 4, ori_mask_mode = 4 (sliding window),
 * cmp_mask_mode = 3, ori_win_left = window_size - 1, ori_win_right = 0)).  For row r at absolute
 * position p (visible length v = p + 1) and head h, the keys are
 *   - the window: original-cache positions max(0, p - window + 1) .. p (through swa_block_table);
 *   - the selected compressed entries: cmp_idx[r, j] >= 0 with cmp_idx < v / ratio (through
 *     cmp_block_table; other entries are skipped and counted);
 * one softmax over all of them with the head's sink logit in the denominator:
 *   S_i = scale * <q, c_i>;  D = sum_i exp(S_i) + exp(sink_h);  o = sum_i exp(S_i) / D * c_i[0:512];
 *   lse = log D.
 * Readings (the op's source is not printed): the rows are 576-wide latent rows like the MLA cache
 * (score over all 576 dims, value = the first 512); an entry present in both sets counts twice
 * (they are different vectors); with no key at all o = 0 and lse = sink_h.
 * out: double [n_rows, H, 512], lse: double [n_rows, H].  Returns the skipped entries. */
int64_t dsa_oracle_dsv4_attention(const uint16_t* q_bf16, const uint16_t* swa_kv, int64_t swa_pages,
                                  const int32_t* swa_block_table, int32_t swa_max_pages, const uint16_t* cmp_kv,
                                  int64_t cmp_pages, const int32_t* cmp_block_table, int32_t cmp_max_pages,
                                  const int32_t* seq_lens, const int32_t* cu_q, int32_t B, const int32_t* cmp_idx,
                                  int32_t k, int32_t window, int32_t ratio, const float* sinks, int32_t H,
                                  double scale, const int64_t* rows, int64_t n_rows, double* out, double* lse) {
    int64_t bad_total = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad_total)
    for (int64_t i = 0; i < n_rows * H; ++i) {
        const int64_t ri = i / H;
        const int h = (int)(i % H);
        const int64_t r = rows[ri];
        const int b = row_request(cu_q, B, r);
        const int32_t v = dsa_oracle_visible_len(seq_lens, cu_q, B, r);
        const int32_t vc = v / ratio;
        const int64_t nmax = (int64_t)window + k;
        const uint16_t** rowp = (const uint16_t**)malloc(sizeof(uint16_t*) * (size_t)(nmax > 0 ? nmax : 1));
        int64_t n = 0, bad = 0;
        for (int32_t pos = v - window > 0 ? v - window : 0; b >= 0 && pos < v; ++pos) {
            const int64_t g = latent_row(swa_block_table, swa_max_pages, swa_pages, b, pos);
            if (g < 0) { ++bad; continue; }
            rowp[n++] = swa_kv + g * DQK;
        }
        for (int32_t j = 0; b >= 0 && j < k; ++j) {
            const int32_t e = cmp_idx[r * (int64_t)k + j];
            if (e < 0) continue;
            const int64_t g = e < vc ? latent_row(cmp_block_table, cmp_max_pages, cmp_pages, b, e) : -1;
            if (g < 0) { ++bad; continue; }
            rowp[n++] = cmp_kv + g * DQK;
        }
        double q[DQK];
        for (int d = 0; d < DQK; ++d) q[d] = (double)bf16_bits_to_f32(q_bf16[(r * H + h) * DQK + d]);
        double* S = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        const double sink = (double)sinks[h];
        double m = sink;
        for (int64_t t = 0; t < n; ++t) {
            double dot = 0.0;
            for (int d = 0; d < DQK; ++d) dot += q[d] * (double)bf16_bits_to_f32(rowp[t][d]);
            S[t] = scale * dot;
            if (S[t] > m) m = S[t];
        }
        double D = exp(sink - m);
        for (int64_t t = 0; t < n; ++t) D += exp(S[t] - m);
        double* o = out + (ri * H + h) * DV;
        for (int d = 0; d < DV; ++d) o[d] = 0.0;
        for (int64_t t = 0; t < n; ++t) {
            const double pw = exp(S[t] - m) / D;
            for (int d = 0; d < DV; ++d) o[d] += pw * (double)bf16_bits_to_f32(rowp[t][d]);
        }
        lse[ri * H + h] = m + log(D);
        free(S);
        free(rowp);
        if (h == 0) bad_total += bad;
    }
    return bad_total;
}

/* ---------------------------------------------------------------- FP8 latent cache */

/* Per-tensor FP8 quantisation ([mla] MLACommonImpl.forward with kv_cache_dtype "fp8": the latent
 * cache is written by concat_and_cache_mla(k_c_normed, k_pe, kv_cache, slot_mapping, kv_cache_dtype,
 * scale = layer._k_scale) and the decode query by ops.scaled_fp8_quant(decode_ql_nope /
 * decode_q_pe, layer._q_scale); the cache is then viewed as the fp8 dtype).  Reading: code =
 * E4M3FN(x / scale) with x the bf16 value, the division one IEEE fp32 operation, round to nearest
 * even with saturation to +-448 (the encoder above); one fp32 scale for the whole tensor. */
void dsa_oracle_quant_fp8_tensor(const uint16_t* x_bf16, int64_t n, float scale, uint8_t* codes) {
    for (int64_t i = 0; i < n; ++i) codes[i] = dsa_oracle_e4m3_encode(bf16_bits_to_f32(x_bf16[i]) / scale);
}

/* Latent rows (512 latent + 64 rope dims, bf16) into the FP8 cache [num_pages, 64, 576] by slot
 * ([mla] concat_and_cache_mla with the fp8 cache): row slot & 63 of page slot >> 6 gets the 576
 * codes.  A negative slot is padding (skipped); a slot past the pool is skipped and counted. */
int64_t dsa_oracle_store_latent_fp8(const uint16_t* latent_bf16, const int64_t* slot_mapping, int64_t n, float k_scale,
                                    uint8_t* pool, int64_t num_pages) {
    int64_t bad = 0;
    for (int64_t t = 0; t < n; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot / PAGE >= num_pages) { ++bad; continue; }
        dsa_oracle_quant_fp8_tensor(latent_bf16 + t * DQK, DQK, k_scale, pool + slot * DQK);
    }
    return bad;
}

/* Attention of one (row, head) over FP8 latent rows: the query quantised per tensor with q_scale,
 * keys and values the cached codes times k_scale ([mla] _forward_decode on the fp8 query and cache):
 * S_i = scale * sum_d (dec(qc_d) q_scale)(dec(kc_id) k_scale); P = softmax(S);
 * o = sum_i P_i dec(kc_i[0:512]) k_scale; the same steps as attend_rows on the dequantised values. */
static void attend_rows_fp8(const uint16_t* qh, float q_scale, const uint8_t* kv, float k_scale, const int64_t* g,
                            int64_t n, double scale, double* o, double* lse) {
    for (int d = 0; d < DV; ++d) o[d] = 0.0;
    if (n == 0) {
        *lse = -INFINITY;
        return;
    }
    double q[DQK];
    for (int d = 0; d < DQK; ++d)
        q[d] = dsa_oracle_e4m3_decode(dsa_oracle_e4m3_encode(bf16_bits_to_f32(qh[d]) / q_scale)) * (double)q_scale;
    double* S = (double*)malloc(sizeof(double) * (size_t)n);
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        const uint8_t* c = kv + g[i] * DQK;
        double dot = 0.0;
        for (int d = 0; d < DQK; ++d) dot += q[d] * (dsa_oracle_e4m3_decode(c[d]) * (double)k_scale);
        S[i] = scale * dot;
        if (S[i] > m) m = S[i];
    }
    double l = 0.0;
    for (int64_t i = 0; i < n; ++i) l += exp(S[i] - m);
    for (int64_t i = 0; i < n; ++i) {
        const double p = exp(S[i] - m) / l;
        const uint8_t* c = kv + g[i] * DQK;
        for (int d = 0; d < DV; ++d) o[d] += p * (dsa_oracle_e4m3_decode(c[d]) * (double)k_scale);
    }
    *lse = m + log(l);
    free(S);
}

/* Sparse MLA decode over the FP8 latent cache: dsa_oracle_sparse_mla with the query quantised by
 * q_scale and the cache rows as FP8 codes with k_scale (kv: uint8 [num_pages, 64, 576]). */
int64_t dsa_oracle_sparse_mla_fp8(const uint16_t* q_bf16, float q_scale, const uint8_t* kv, float k_scale,
                                  int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                  const int32_t* seq_lens, const int32_t* cu_q, int32_t B, const int32_t* idx, int32_t k,
                                  int32_t H, double scale, const int64_t* rows, int64_t n_rows, double* out,
                                  double* lse) {
    int64_t bad_total = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad_total)
    for (int64_t i = 0; i < n_rows * H; ++i) {
        int64_t ri = i / H;
        int h = (int)(i % H);
        int64_t r = rows[ri];
        int b = row_request(cu_q, B, r);
        int32_t v = dsa_oracle_visible_len(seq_lens, cu_q, B, r);
        int64_t* g = (int64_t*)malloc(sizeof(int64_t) * (size_t)k);
        int64_t n = 0, bad = 0;
        for (int32_t j = 0; j < k; ++j) {
            int32_t pos = idx[r * (int64_t)k + j];
            if (pos < 0) continue;
            int64_t gr = (b >= 0 && pos < v) ? latent_row(block_table, max_pages, num_pages, b, pos) : -1;
            if (gr < 0) { ++bad; continue; }
            g[n++] = gr;
        }
        attend_rows_fp8(q_bf16 + (r * H + h) * DQK, q_scale, kv, k_scale, g, n, scale, out + (ri * H + h) * DV,
                        lse + ri * H + h);
        free(g);
        if (h == 0) bad_total += bad;
    }
    return bad_total;
}

/* Dense MLA decode over every visible position [0, v_r) of the request, the same attention with
 * no selection ([mla] _forward_decode over the whole paged latent cache).  Used to pin the sparse
 * form: with k >= v_r the selection keeps every position and the two must agree. */
void dsa_oracle_dense_mla(const uint16_t* q_bf16, const uint16_t* kv, int64_t num_pages,
                          const int32_t* block_table, int32_t max_pages, const int32_t* seq_lens,
                          const int32_t* cu_q, int32_t B, int32_t H, double scale,
                          const int64_t* rows, int64_t n_rows, double* out, double* lse) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n_rows * H; ++i) {
        int64_t ri = i / H;
        int h = (int)(i % H);
        int64_t r = rows[ri];
        int b = row_request(cu_q, B, r);
        int32_t v = dsa_oracle_visible_len(seq_lens, cu_q, B, r);
        int64_t* g = (int64_t*)malloc(sizeof(int64_t) * (size_t)(v > 0 ? v : 1));
        int64_t n = 0;
        for (int32_t pos = 0; pos < v; ++pos) {
            int64_t gr = latent_row(block_table, max_pages, num_pages, b, pos);
            if (gr >= 0) g[n++] = gr;
        }
        attend_rows(q_bf16 + (r * H + h) * DQK, kv, g, n, scale, out + (ri * H + h) * DV,
                    lse + ri * H + h, NULL);
        free(g);
    }
}

/* Merge of two partial attention results by their log-sum-exp ([mla] merge_attn_states(output,
 * output_lse, prefix_output, prefix_lse, suffix_output, suffix_lse) in the chunked-context loop):
 * lse = log(e^lse1 + e^lse2); o = e^(lse1 - lse) o1 + e^(lse2 - lse) o2.  Both -inf gives o = 0,
 * lse = -inf.  n vectors of width dv. */
void dsa_oracle_lse_merge(const double* o1, const double* lse1, const double* o2, const double* lse2,
                          int64_t n, int32_t dv, double* o, double* lse) {
    for (int64_t i = 0; i < n; ++i) {
        double a = lse1[i], b = lse2[i];
        double m = a > b ? a : b;
        if (m == -INFINITY) {
            lse[i] = -INFINITY;
            for (int d = 0; d < dv; ++d) o[i * dv + d] = 0.0;
            continue;
        }
        double l = exp(a - m) + exp(b - m);
        double L = m + log(l);
        double wa = exp(a - L), wb = exp(b - L);
        for (int d = 0; d < dv; ++d) o[i * dv + d] = wa * o1[i * dv + d] + wb * o2[i * dv + d];
        lse[i] = L;
    }
}

int dsa_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void dsa_oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
