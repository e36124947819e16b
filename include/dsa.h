/*
 * dsa.h -- C ABI of the GB300 (sm_103a) DeepSeek Sparse Attention decode path.
 *
 * Three stages run on one GPU, each a hand-written CUDA kernel:
 *   1. lightning indexer: I[r,s] = sum_h w[r,h] * ReLU(q_I[r,h] . k_I[s]) over a paged FP8-E4M3
 *      index-K cache with one fp32 scale per token (64 heads x 128 dims, page size 64);
 *   2. per-row top-k over the logits (causal and length-masked, lower index wins ties);
 *   3. absorbed-form sparse MLA over the selected rows of a paged 576-wide bf16 latent cache
 *      (512 latent + 64 rope, one shared KV head, 512-wide latent output).
 * A fourth call writes new keys into the index-K cache (Hadamard rotation, per-token FP8
 * quantisation, paged scatter by slot); two prologue calls add the key norm and rotary embedding
 * in front of that store and the rotary embedding of the indexer query; two more compute the
 * per-head projections around the absorbed attention (absorbed query, value up-projection).
 * Variants: the top-k with forced initial / local tokens, power-of-two (ue8m0) quantisation
 * scales, a one-call indexer that returns top-k indices, and a sparse MLA call that needs no
 * workspace.
 *
 * Conventions shared by every call
 * --------------------------------
 * Pointers.  Every array argument is a DEVICE pointer unless stated otherwise; scalars are passed
 *   by value.  bf16 arrays are passed as `const void*` holding IEEE bfloat16 bit patterns.
 * Ownership.  The caller owns every buffer.  The library never allocates or frees device memory
 *   and keeps no state between calls; scratch space is passed in as `workspace` with its size
 *   queried from the matching *_workspace_size() call.  The one exception is
 *   dsa_sparse_mla_decode_noalloc, whose scratch is a fixed array inside the library.
 * Streams.  `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls enqueue work on
 *   it and return without synchronising; results are ready when the stream reaches them.
 * Requests and rows.  B requests; request b has seq_lens[b] cached tokens (this step's tokens
 *   included) and q_len_b = cu_q[b+1] - cu_q[b] query tokens; global query row r = cu_q[b] + j,
 *   0 <= j < q_len_b, sits at absolute position p = seq_lens[b] - q_len_b + j and sees keys
 *   [0, p], i.e. v_r = p + 1 keys (causal rule of the ragged key ends `ke = start + pos + 1` in
 *   sglang dsa_indexer.py, Indexer._get_topk_ragged / forward, and sparse_mode=3 in vllm_ascend
 *   sfa_v1.py).  T = cu_q[B] rows in total.
 * Paging.  Page size is 64 tokens for both caches (sglang dsa_indexer.py,
 *   Indexer._get_topk_paged: "only support page size 64").  One int32 block table
 *   [B, max_pages] maps logical page i of request b to a physical page id; entries that are not
 *   used may hold -1.  The same table serves the index-K cache and the latent cache (vllm_ascend
 *   sfa_v1.py passes one block_table to the indexer and to the sparse attention).
 * Index-K cache layout.  uint8 [num_pages, 64 * 132]: 132 bytes per token (sglang
 *   Indexer._get_topk_paged: head_dim_with_sf = 132).  Inside a page: bytes [0, 8192) hold the
 *   64 tokens' 128 FP8-E4M3FN codes row by row, bytes [8192, 8448) hold their 64 fp32 scales
 *   (page-blocked; the pages fix the byte count, not the order inside a page).  The dequantised
 *   key is code * scale.
 * Latent cache layout.  bf16 [num_pages, 64, 576]: per token 512 latent dims then 64 rope dims
 *   (vllm mla/common.py, MLACommonBackend: head size 576, one KV head).
 * Errors.  Argument checks on the host return DSA_ERR_INVALID_ARG or DSA_ERR_UNSUPPORTED before
 *   anything is enqueued.  A failed kernel launch returns DSA_ERR_CUDA.  Data-dependent problems
 *   found on the device (a slot, page id or top-k index out of range) never fault: the access is
 *   skipped and a bit is OR-ed into the optional device word `dev_err` (int32, caller-zeroed);
 *   read it with dsa_read_device_error().
 */
#ifndef DSA_GB300_DSA_H
#define DSA_GB300_DSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, inconsistent arguments */
    DSA_ERR_UNSUPPORTED = 2,   /* valid in principle, not implemented (page size != 64, ...) */
    DSA_ERR_CUDA = 3,          /* a CUDA launch or runtime call failed */
    DSA_ERR_DEVICE_BOUNDS = 4, /* the device error word reports skipped out-of-range accesses */
    DSA_ERR_TIMEOUT = 5        /* the device error word reports a bounded wait that gave up */
} dsa_status;

/* Bits of the device error word. */
#define DSA_DEVERR_SLOT_RANGE 0x1  /* store: slot past the pool (token skipped) */
#define DSA_DEVERR_PAGE_RANGE 0x2  /* a block-table entry outside [0, num_pages) was needed */
#define DSA_DEVERR_INDEX_RANGE 0x4 /* a top-k index outside [0, v_r) (entry skipped) */
#define DSA_DEVERR_TIMEOUT 0x8     /* a bounded spin-wait gave up */
#define DSA_DEVERR_POSITION 0x10   /* a rotary position outside [0, max_position) */

/* Flags of dsa_indexer_logits. */
#define DSA_Q_ROTATE 0x1u          /* Hadamard-rotate each query head before quantising it */

/* Flags of dsa_store_index_k_prologue and dsa_indexer_rope_q. */
#define DSA_NORM_RMS 0x2u          /* key norm is RMSNorm (default: LayerNorm with bias) */
#define DSA_ROPE_INTERLEAVED 0x4u  /* rotary pairs (2i, 2i+1) (default: neox pairs (i, i+32)) */
#define DSA_K_NO_ROTATE 0x8u       /* key prologue: quantise without the Hadamard rotation */

/* Flag of dsa_store_index_k_prologue and dsa_indexer_logits: the "ue8m0" scale format -- every
 * quantisation scale is the smallest power of two not below the fp32 scale max(amax, 1e-4) / 448
 * (sglang dsa_indexer.py, Indexer(scale_fmt) handed to act_quant). */
#define DSA_SCALE_UE8M0 0x10u
/* Flag of dsa_indexer_logits / dsa_lightning_indexer: the cache holds compressed keys, one entry per
 * 4 tokens (DSV4 compress ratio 4: vllm_ascend dsa_v1.py, npu_vllm_quant_lightning_indexer(...,
 * cmp_ratio = 4)).  Row r then sees the entries s < v_r / 4 (entry s stands for tokens
 * [4s, 4s + 4), visible once all four are); seq_lens stay the token counts, and max_seq_len bounds
 * the entries (>= every v_r / 4).  The top-k of dsa_lightning_indexer uses the same rule. */
#define DSA_KEYS_CMP4 0x20u

/* Fixed shape constants of the path. */
#define DSA_PAGE_SIZE 64
#define DSA_INDEX_HEADS 64
#define DSA_INDEX_DIM 128
#define DSA_INDEX_ROW_BYTES 132
#define DSA_INDEX_PAGE_BYTES (64 * 132)
#define DSA_LATENT_DIM 576
#define DSA_VALUE_DIM 512
#define DSA_MAX_TOPK 2048

/* Human-readable name of a status code (static string). */
const char* dsa_status_str(dsa_status s);

/*
 * dsa_store_index_k -- write n new indexer keys into the paged FP8 index-K cache.
 * Source: sglang dsa_indexer.py, Indexer._store_index_k_cache (fused_store_index_k_cache(key,
 * buf, out_cache_loc, page_size), or act_quant(key, 128) followed by set_index_k_scale_buffer)
 * and rotate_activation (Hadamard transform with scale 128^-0.5); vllm_ascend sfa_v1.py,
 * indexer_select_pre_process (k @ hadamard) and the slot_mapping scatter.
 * Per token t:
 *   x = k_bf16[t, 0:128] (bf16 -> fp32, exact);
 *   Walsh-Hadamard butterflies in fp32, Sylvester order (h = 1, 2, ..., 64: (a, b) -> (a+b, a-b));
 *   y = bf16_rn(x * fp32(1/sqrt(128)));
 *   scale = max(max_d |y_d|, 1e-4) / 448 (fp32, IEEE division);
 *   code_d = E4M3FN round-to-nearest-even with saturation of (y_d / scale) (IEEE division);
 *   page = slot >> 6, row = slot & 63: codes to bytes [row*128, row*128+128) of the page,
 *   scale to bytes [8192 + row*4, +4).
 * Arguments:
 *   k_bf16        [n, 128] bf16, row-major (16-byte aligned).
 *   slot_mapping  [n] int64; slot < 0 marks a padding token and is skipped.
 *   n             number of tokens (0 is allowed and enqueues nothing).
 *   index_k_pool  uint8 [num_pages, 8448] (16-byte aligned), written in place.
 *   page_size     must be 64 (DSA_ERR_UNSUPPORTED otherwise).
 *   dev_err       nullable; DSA_DEVERR_SLOT_RANGE when slot >= num_pages * 64 (token skipped).
 * Results are bit-exact with the CPU definition above.
 */
dsa_status dsa_store_index_k(const void* k_bf16, const int64_t* slot_mapping, int64_t n,
                             uint8_t* index_k_pool, int64_t num_pages, int32_t page_size,
                             int32_t* dev_err, void* stream);

/*
 * dsa_store_index_k_prologue -- key norm, rotary embedding, then dsa_store_index_k, in one kernel.
 * Source: sglang dsa_indexer.py, Indexer._get_k_bf16 (k_norm, rotary_emb on the first 64 (rope)
 * dims of the 64 rope + 64 nope split, rotate_activation) followed by _store_index_k_cache;
 * Indexer._fused_k_prepare_and_store (fused_k_indexer_norm_rope_store(key, buffer,
 * out_cache_loc, k_norm weight / bias / eps, cos_sin_cache, positions)), which drops the Hadamard
 * rotation (Indexer._maybe_rotate: the rotation is orthogonal and applied to both query and key)
 * -- flag DSA_K_NO_ROTATE; Indexer.k_norm (LayerNorm over the 128 dims, RMSNorm when the model
 * config asks for it); vllm_ascend sfa_v1.py, indexer_select_pre_process (k_norm, then rope on
 * k_pe, then the Hadamard rotation and the slot_mapping scatter).
 * Per token t with slot >= 0:
 *   x = k_raw_bf16[t, 0:128];
 *   LayerNorm: mean = S(x) / 128, d = x - mean, var = S(d * d) / 128, rstd = 1 / sqrt(var + eps),
 *     n = bf16_rn((d * rstd) * w + b);  RMSNorm (DSA_NORM_RMS): rstd = 1 / sqrt(S(x * x) / 128 + eps),
 *     n = bf16_rn((x * rstd) * w).  The definition is exact (the sums, square root and division
 *     exact, one rounding to bf16); the kernel evaluates it in fp32, so where the exact n lies within
 *     that fp32 error of a bf16 rounding boundary (about 2 outputs in 10^5) its n is one bf16 unit
 *     away and that token's codes may move by one E4M3 step.
 *   Rotary: c, s = cos_sin_cache[positions[t], 0:32], [32:64]; neox pairs (a, b) = (n_i, n_{i+32})
 *     (DSA_ROPE_INTERLEAVED: (n_{2i}, n_{2i+1})), i < 32: a' = bf16_rn(a c_i - b s_i),
 *     b' = bf16_rn(b c_i + a s_i); dims 64 .. 127 unchanged.
 *   Then the steps of dsa_store_index_k on the result; with DSA_K_NO_ROTATE the rotation is
 *   skipped and the rotary output itself is quantised and stored.
 *   The rotary embedding and everything after it are IEEE fp32 operations without fused
 *   multiply-add, as the definition states them.
 * Arguments:
 *   k_raw_bf16     [n, 128] bf16 (16-byte aligned): the key projection before the norm.
 *   norm_weight    fp32 [128] (16-byte aligned).  norm_bias: fp32 [128] (16-byte aligned) for
 *                  LayerNorm; ignored (may be NULL) with DSA_NORM_RMS.
 *   eps            the norm's epsilon.
 *   cos_sin_cache  fp32 [max_position, 64] (16-byte aligned): cos in [0, 32), sin in [32, 64).
 *   positions      int64 [n].  slot_mapping int64 [n] (slot < 0: padding, skipped).
 *   index_k_pool, num_pages, page_size  as for dsa_store_index_k.
 *   flags          0 or a combination of DSA_NORM_RMS, DSA_ROPE_INTERLEAVED, DSA_K_NO_ROTATE and
 *                  DSA_SCALE_UE8M0 (power-of-two key scales).
 *   dev_err        nullable; DSA_DEVERR_POSITION for a position outside [0, max_position),
 *                  DSA_DEVERR_SLOT_RANGE for a slot past the pool (the token is skipped either way).
 */
dsa_status dsa_store_index_k_prologue(const void* k_raw_bf16, const float* norm_weight,
                                      const float* norm_bias, float eps, const float* cos_sin_cache,
                                      int64_t max_position, const int64_t* positions,
                                      const int64_t* slot_mapping, int64_t n, uint8_t* index_k_pool,
                                      int64_t num_pages, int32_t page_size, uint32_t flags,
                                      int32_t* dev_err, void* stream);

/*
 * dsa_indexer_rope_q -- rotary embedding of the indexer query (the rope step that precedes the
 * query prologue of dsa_indexer_logits).
 * Source: sglang dsa_indexer.py, Indexer.forward_cuda / fused_q_indexer_rope_first_quant (rope on
 * the first 64 dims of every head, then the Hadamard rotation and FP8 quantisation, which
 * dsa_indexer_logits does with DSA_Q_ROTATE); vllm_ascend sfa_v1.py, indexer_select_pre_process
 * (q_pe rope before the indexer).
 *   Every head h of row t: the rotary step of dsa_store_index_k_prologue at positions[t].
 *   A row whose position is outside [0, max_position) is copied unchanged and
 *   DSA_DEVERR_POSITION is set.
 * Arguments:
 *   q_raw_bf16     [T, 64, 128] bf16 (16-byte aligned).  q_out_bf16: same shape (may equal
 *                  q_raw_bf16: each vector is read before it is written by the same warp).
 *   cos_sin_cache, max_position  as above.  positions int64 [T].
 *   flags          0 or DSA_ROPE_INTERLEAVED.
 * Bit-exact with the CPU definition.
 */
dsa_status dsa_indexer_rope_q(const void* q_raw_bf16, const float* cos_sin_cache, int64_t max_position,
                              const int64_t* positions, int64_t T, uint32_t flags, void* q_out_bf16,
                              int32_t* dev_err, void* stream);

/*
 * dsa_indexer_logits -- lightning-indexer logits over the paged index-K cache.
 * Source: sglang dsa_indexer.py, Indexer._get_topk_paged (paged MQA logits over block_tables /
 * seqlens, kv cache viewed as [pages, 64, 1, 132]) with the head gate of _get_logits_head_gate
 * (weights * q_scale); Indexer.forward_cuda (act_quant of the query per 128 dims);
 * vllm_ascend sfa_v1.py, npu_lightning_indexer.
 *   Query prologue, per row r and head h: optional Hadamard rotation (flag DSA_Q_ROTATE; same
 *   steps as the key rotation above), then per-128 FP8 quantisation with scale q_scale[r,h]
 *   (same rule as the keys); w'[r,h] = weights[r,h] * q_scale[r,h].
 *   I[r,s] = sum_h w'[r,h] * ReLU(k_scale[s] * sum_d q_code[r,h,d] * k_code[s,d]),  s < v_r,
 *   accumulated in fp32 (FP8 x FP8 products are exact in fp32).
 * Arguments:
 *   q_bf16       [T, 64, 128] bf16 (16-byte aligned).
 *   weights      [T, 64] fp32 head gates (already scaled by 64^-0.5 * 128^-0.5 by the caller).
 *   index_k_pool uint8 [num_pages, 8448] written by dsa_store_index_k (16-byte aligned).
 *   block_table  int32 [B, max_pages]; seq_lens int32 [B]; cu_q int32 [B + 1] (device).
 *   max_seq_len  host upper bound of seq_lens (sizes the launch; must be >= every seq_lens[b]).
 *   max_q_len    host upper bound of the per-request query counts.
 *   row_begin, row_end  host: the global rows [row_begin, row_end) to score (row tiling of a long
 *                prefill chunk; pass 0, T for all rows).
 *   logits       fp32 [row_end - row_begin, ld]; row r goes to logits[(r - row_begin) * ld].
 *                Entries s >= v_r are left untouched.  ld >= max_seq_len.
 *   flags        0 or a combination of DSA_Q_ROTATE and DSA_SCALE_UE8M0 (power-of-two query scales).
 *   workspace    device scratch of at least dsa_indexer_logits_workspace_size(row_end - row_begin)
 *                bytes, 16-byte aligned, owned by the caller.  It holds the quantised query rows
 *                (the prologue runs once per row instead of once per key tile); its contents need
 *                no initialisation and are dead after the call, but two calls in flight at the
 *                same time must not share it.
 *   dev_err      nullable; DSA_DEVERR_PAGE_RANGE when a needed page id is out of range (those
 *                keys' logits are not written).
 * Two kernels are enqueued on `stream`: the query prologue, then the logits kernel as its
 * programmatic dependent (it may start before the prologue ends and waits for it on the device).
 * The prologue is itself a programmatic dependent of whatever kernel precedes it on the stream: it
 * may be scheduled early but waits on the device for that kernel's completion before it reads or
 * writes anything.
 */
size_t dsa_indexer_logits_workspace_size(int32_t rows);
dsa_status dsa_indexer_logits(const void* q_bf16, const float* weights, const uint8_t* index_k_pool,
                              int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                              const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                              int32_t max_seq_len, int32_t max_q_len, int32_t row_begin,
                              int32_t row_end, float* logits, int64_t ld, uint32_t flags,
                              void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream);

/*
 * dsa_store_index_k_c8 -- write n new indexer keys into the paged int8 ("c8") index-K cache.
 * Source: vllm_ascend sfa_v1.py, AscendSFAImpl with enable_sparse_c8 (c8 k cache dtype int8, scale
 * cache dtype float16; qk_hadamard = bf16 tensor of scipy.linalg.hadamard(128) / 128**0.5) and
 * indexer_select_pre_process (k_li @ qk_hadamard; npu_dynamic_quant(k_li.view(-1, 128),
 * dst_type=int8); scale .to(float16)); the npu_scatter_nd_update_ of codes (kv_cache[2]) and scales
 * (kv_cache[3]) by slot_mapping.
 * Per token t (c = bf16(128^-0.5) = 181 * 2^-11, the value of every entry of the bf16 matrix):
 *   y_j = bf16_rn(c * sum_i (-1)^popcount(i & j) x_i)  (the exact sum rounded once: the correctly
 *         rounded bf16 matrix product; the kernel's fp64 butterflies are exact for 128 bf16 values);
 *   scale = max_j |y_j| / 127 (fp32, IEEE division);
 *   code_j = round-to-nearest-even(y_j / scale) (fp32 IEEE division), in [-127, 127]; all 0 when
 *            every y_j is 0;
 *   page = slot >> 6, row = slot & 63: the 128 int8 codes to bytes [row*128, +128) of the page, the
 *   scale rounded to fp16 (nearest even) to bytes [8192 + row*2, +2).
 * (npu_dynamic_quant is not printed on the pages: the fp32 scale amax / 127 with nearest-even codes
 * is the plain symmetric per-row quantisation.)
 * Arguments:
 *   k_bf16           [n, 128] bf16, row-major (16-byte aligned).
 *   slot_mapping     [n] int64; slot < 0 marks a padding token and is skipped.
 *   index_k_pool_c8  uint8 [num_pages, 8320] (16-byte aligned), written in place.
 *   page_size        must be 64 (DSA_ERR_UNSUPPORTED otherwise).
 *   dev_err          nullable; DSA_DEVERR_SLOT_RANGE when slot >= num_pages * 64 (token skipped).
 * Results are bit-exact with the CPU definition above.
 */
dsa_status dsa_store_index_k_c8(const void* k_bf16, const int64_t* slot_mapping, int64_t n,
                                uint8_t* index_k_pool_c8, int64_t num_pages, int32_t page_size,
                                int32_t* dev_err, void* stream);

/*
 * dsa_indexer_logits_c8 -- lightning-indexer logits over the int8 ("c8") index-K cache.
 * Source: vllm_ascend sfa_v1.py, indexer_select_post_process with use_sparse_c8_indexer: q_li @
 * qk_hadamard, npu_dynamic_quant per (token, head), weights.to(float16), then
 * npu_lightning_indexer_quant(query, key, weights, query_dequant_scale, key_dequant_scale,
 * query_quant_mode=0, key_quant_mode=0, ...).
 *   Query prologue, per row r and head h: the transform of dsa_store_index_k_c8 (rotation, int8
 *   codes cq[r,h,:], fp32 scale rounded to fp16 qs16[r,h]); g[r,h] = w16[r,h] * qs16[r,h] with
 *   w16 = fp16_rn(weights[r,h]) (exact in fp32).
 *   I[r,s] = ks16[s] * sum_h g[r,h] * ReLU(sum_d cq[r,h,d] * ck[s,d]),  s < v_r
 *   -- the lightning-indexer score on the dequantised query and keys.  The integer dot products are
 *   exact (the int8 values are widened to f16 and multiplied on the tensor cores with fp32
 *   accumulation, exact below 2^24); the head sum is fp32.
 * Arguments: as dsa_indexer_logits, without flags; index_k_pool_c8 is uint8 [num_pages, 8320]
 *   written by dsa_store_index_k_c8; workspace at least dsa_indexer_logits_c8_workspace_size(
 *   row_end - row_begin) bytes (16-byte aligned, caller-owned; it holds the rows' f16 query codes).
 * Two kernels are enqueued on `stream` (query prologue, then the logits kernel as its programmatic
 * dependent).  The top-k over these logits is dsa_topk.
 */
size_t dsa_indexer_logits_c8_workspace_size(int32_t rows);
dsa_status dsa_indexer_logits_c8(const void* q_bf16, const float* weights, const uint8_t* index_k_pool_c8,
                                 int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                 const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                                 int32_t max_seq_len, int32_t max_q_len, int32_t row_begin,
                                 int32_t row_end, float* logits, int64_t ld, void* workspace,
                                 size_t ws_bytes, int32_t* dev_err, void* stream);

/*
 * dsa_topk -- per-row top-k of the indexer logits.
 * Source: sglang dsa_indexer.py, forward_indexer (logits.topk(min(topk, seq_len)) then -1
 * padding to 2048), Indexer._get_topk_paged (topk_transform; rows not scored are -1).
 *   For row r the kept set is the min(k, v_r) largest I[r, 0:v_r) with ties broken toward the
 *   lower index (a stable descending order); -0 equals +0; NaN is never kept ahead of a number.
 *   idx[r] lists the kept indices in ASCENDING index order, then -1 up to k.  Logits at
 *   s >= v_r are never read.
 * Arguments:
 *   logits      fp32 rows as written by dsa_indexer_logits for [row_begin, row_end), stride ld.
 *   k           1 .. 2048.
 *   idx         int32 [row_end - row_begin, k].
 *   workspace   device scratch of dsa_topk_workspace_size(rows, k, max_seq_len) bytes (may be
 *               NULL when that size is 0).
 * Output is deterministic and bit-exact with the CPU definition.
 */
size_t dsa_topk_workspace_size(int32_t rows, int32_t k, int32_t max_seq_len);
dsa_status dsa_topk(const float* logits, int64_t ld, const int32_t* seq_lens, const int32_t* cu_q,
                    int32_t B, int32_t max_seq_len, int32_t row_begin, int32_t row_end, int32_t k,
                    int32_t* idx, void* workspace, size_t workspace_bytes, void* stream);

/*
 * dsa_topk_forced -- dsa_topk with forced initial and local tokens.
 * Source: sglang dsa_indexer.py, Indexer._mask_init_and_local_tokens (the logits of the first
 * index_init_tokens and of the last index_local_tokens positions of each row are set to +inf
 * before the top-k; the model config's index_init_tokens / index_local_tokens, 0 by default).
 *   For row r with v_r visible keys, positions [0, min(n_init, v_r)) and [max(0, v_r - n_local),
 *   v_r) count as +inf; then the rule of dsa_topk (ties, including a logit that is itself +inf,
 *   go to the lower index).  n_init = n_local = 0 is dsa_topk.
 *   n_init, n_local >= 0 (DSA_ERR_INVALID_ARG otherwise); other arguments as for dsa_topk.
 */
dsa_status dsa_topk_forced(const float* logits, int64_t ld, const int32_t* seq_lens, const int32_t* cu_q,
                           int32_t B, int32_t max_seq_len, int32_t row_begin, int32_t row_end, int32_t k,
                           int32_t n_init, int32_t n_local, int32_t* idx, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * dsa_lightning_indexer -- indexer logits and top-k in one call that returns the indices.
 * Source: vllm_ascend sfa_v1.py, the indexer's npu_lightning_indexer(query, key = paged index
 * cache, weights, actual_seq_lengths_query / _key, block_table, sparse_count, sparse_mode = 3)
 * returning topk_indices; sglang dsa_indexer.py, Indexer._get_topk_paged (logits, the
 * init / local token mask, then topk_transform).
 *   idx[r] = dsa_topk_forced(dsa_indexer_logits(...)[r]) for every row r < T.  The logits are
 *   kept in `workspace` (dsa_lightning_indexer_workspace_size(T, max_seq_len) bytes, 16-byte
 *   aligned); the stages are chained on the device.
 *   Fused (max_q_len < 4, i.e. row groups of 1 or 2 query rows, and max_seq_len <= 131072): the
 *   logits kernel also counts, per row, the top 12 bits of each logit's order key (the key the
 *   top-k selects on) and the top-k kernels take that histogram instead of a first read of the row.
 *   Selected indices are the same as unfused; a visible key whose page id is out of range gets the
 *   logit -inf (unfused: left unwritten).  Otherwise the two calls run as they are.
 *   Workspace layout, each part starting 256-byte aligned: T x 4096 uint32 histograms; the logits
 *   call's query scratch (dsa_indexer_logits_workspace_size(T) bytes); the fp32 logits, row r at
 *   row r * ld, ld = max_seq_len rounded up to a multiple of 4 (at least 4).  They stay there
 *   after the call.
 * Arguments: as for dsa_indexer_logits (all rows, 0 .. T) and dsa_topk_forced; flags: as for
 * dsa_indexer_logits.
 */
size_t dsa_lightning_indexer_workspace_size(int32_t T, int32_t max_seq_len);
dsa_status dsa_lightning_indexer(const void* q_bf16, const float* weights, const uint8_t* index_k_pool,
                                 int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                 const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                                 int32_t max_seq_len, int32_t max_q_len, int32_t T, int32_t k,
                                 int32_t n_init, int32_t n_local, uint32_t flags, int32_t* idx,
                                 void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream);

/*
 * dsa_sparse_mla_decode -- absorbed sparse MLA over the selected latent rows.
 * Source: vllm_ascend sfa_v1.py, _execute_sparse_flash_attention_process
 * (npu_sparse_flash_attention(query = ql_nope, key = value = latent cache, sparse_indices =
 * top-k, sparse_block_size = 1, block_table, query_rope = q_pe, key_rope)); vllm mla/common.py,
 * MLACommonImpl.forward decode branch (absorbed query [ql_nope 512, q_pe 64], _forward_decode
 * returns (out, lse); merge_attn_states combines partial results by log-sum-exp).
 *   For row r and head h, over every valid entry i of idx[r, 0:k) (valid: 0 <= i < v_r; -1 is
 *   padding): g(i) = block_table[b][i >> 6] * 64 + (i & 63);
 *   S_i = scale * <q[r,h,0:576], C[g(i),0:576]>; P = softmax(S);
 *   out[r,h,0:512] = bf16_rn(sum_i P_i * C[g(i),0:512]);  lse[r,h] = max S + ln sum exp(S - max S).
 *   A row with no valid entry gives out = 0 and lse = -inf.  Accumulation in fp32; the work is
 *   split over the selected entries and the partial results are merged by log-sum-exp.
 * Arguments:
 *   q_bf16      [T, H, 576] bf16 (16-byte aligned); H in {16, 32, 64, 128}.
 *   kv_pool     bf16 [num_pages, 64, 576] (16-byte aligned).
 *   idx         int32 [T, k] logical positions within the request (as dsa_topk writes them).
 *   k           1 .. 2048.  T: number of rows (= cu_q[B]).
 *   scale       softmax scale (1/sqrt(192) for the DeepSeek configuration).
 *   out_bf16    [T, H, 512] bf16.   lse: fp32 [T, H], nullable.
 *   workspace   device scratch of dsa_sparse_mla_workspace_size(T, H, k) bytes.
 *   dev_err     nullable; DSA_DEVERR_INDEX_RANGE for an index >= v_r, DSA_DEVERR_PAGE_RANGE for an
 *               unmapped page (the entry is skipped either way).
 */
size_t dsa_sparse_mla_workspace_size(int32_t T, int32_t H, int32_t k);
dsa_status dsa_sparse_mla_decode(const void* q_bf16, const void* kv_pool, int64_t num_pages,
                                 const int32_t* block_table, int32_t max_pages,
                                 const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                                 const int32_t* idx, int32_t k, int32_t T, int32_t H, float scale,
                                 void* out_bf16, float* lse, void* workspace,
                                 size_t workspace_bytes, int32_t* dev_err, void* stream);

/*
 * dsa_sparse_mla_decode_noalloc -- dsa_sparse_mla_decode for callers that cannot allocate.
 * The source pages have no counterpart of this call; it exists for callers that may not
 * allocate device memory while they run attention (an engine plugin whose per-step hook must
 * not allocate because the engine owns and budgets all device memory, a loop whose caching
 * allocator already holds the free memory).
 * Same arguments, semantics and kernels as dsa_sparse_mla_decode, minus the workspace: the
 * split-K scratch is a fixed 16 MiB array inside the library, which every GPU that loads the
 * library holds until the process exits.  The call itself calls no allocator.
 *   Limit: problems with dsa_sparse_mla_workspace_size(T, H, k) > 16 MiB are rejected with
 *   DSA_ERR_UNSUPPORTED before anything is enqueued.  That size is T * H * splits * 2052 bytes,
 *   the split count depending on T, k and the GPU's multiprocessor count (no scratch at all once
 *   one split per row fills the GPU: on a 152-SM GB300, at k >= 512, from 39 rows up); at
 *   H = 128, k = 2048 on that GPU it exceeds 16 MiB for 8-9, 16-19 and 32-38 rows.
 *   Set-up: the first call on each device looks up the array's device address with that device
 *   current.  With lazy module loading (CUDA's default) that lookup is also what loads the
 *   library's device code on that device and so makes the 16 MiB array resident there: it can
 *   fail with DSA_ERR_CUDA if the device has no free memory left.  Make that first call before the
 *   caller hands its free memory to its own allocator or fixes its memory budget, and before any
 *   stream capture.
 *   Sharing: every call uses the same array.  Calls whose kernels overlap on the GPU (different
 *   streams, or different host threads, without ordering between them) race on it: order them,
 *   e.g. on one stream.  Nothing in the array has to start at zero; a call never reads what an
 *   earlier call left there.
 */
dsa_status dsa_sparse_mla_decode_noalloc(const void* q_bf16, const void* kv_pool, int64_t num_pages,
                                         const int32_t* block_table, int32_t max_pages,
                                         const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                                         const int32_t* idx, int32_t k, int32_t T, int32_t H,
                                         float scale, void* out_bf16, float* lse, int32_t* dev_err,
                                         void* stream);

/*
 * dsa_store_latent_fp8 -- latent rows into an FP8 latent cache (the fp8 kv-cache variant).
 * Source: vllm mla/common.py, MLACommonImpl.forward: concat_and_cache_mla(k_c_normed, k_pe,
 * kv_cache, slot_mapping, kv_cache_dtype = "fp8", scale = layer._k_scale), then kv_cache viewed as
 * the fp8 dtype.
 *   For each token t with slot = slot_mapping[t] >= 0: row slot & 63 of page slot >> 6 of the
 *   cache gets code_d = E4M3FN(x_d / k_scale), d < 576 (x: the bf16 latent (512) + rope (64)
 *   values; one IEEE fp32 division; round to nearest even; saturating to +-448).  One k_scale for
 *   the whole cache (per-tensor, as the pages' layer._k_scale).
 * Arguments:
 *   latent_bf16   [n, 576] bf16 (16-byte aligned).   slot_mapping  int64 [n] (< 0: padding).
 *   k_scale       > 0, finite.   kv_pool_fp8  uint8 [num_pages, 64, 576] (16-byte aligned).
 *   dev_err       nullable; DSA_DEVERR_SLOT_RANGE for a slot past the pool (token skipped).
 */
dsa_status dsa_store_latent_fp8(const void* latent_bf16, const int64_t* slot_mapping, int64_t n, float k_scale,
                                uint8_t* kv_pool_fp8, int64_t num_pages, int32_t* dev_err, void* stream);

/*
 * dsa_sparse_mla_decode_fp8 -- dsa_sparse_mla_decode over an FP8 latent cache.
 * Source: vllm mla/common.py, MLACommonImpl.forward decode branch with fp8_attention:
 * ops.scaled_fp8_quant(decode_ql_nope, layer._q_scale) and (decode_q_pe, layer._q_scale), then
 * _forward_decode on the fp8 query and the fp8 cache.
 *   The query is quantised here: qc = E4M3FN(q / q_scale) (all 576 dims, as above).  With
 *   c = code * k_scale the cached rows and q^ = qc * q_scale the query, the result is that of
 *   dsa_sparse_mla_decode on (q^, c): S_i = scale * <q^, c_g(i)>, P = softmax(S),
 *   out = bf16_rn(sum_i P_i c_g(i)[0:512]), lse.  Score products are exact (E4M3 x E4M3 on the
 *   tensor cores, fp32 accumulation); P stays bf16 and multiplies the cached values widened to bf16
 *   (exact), so the rounding is that of the bf16 call.
 * Arguments: as dsa_sparse_mla_decode, plus q_scale and k_scale (> 0, finite); kv_pool_fp8 is
 * uint8 [num_pages, 64, 576] (16-byte aligned) written by dsa_store_latent_fp8.  The workspace is
 * the bf16 call's (dsa_sparse_mla_workspace_size).
 */
dsa_status dsa_sparse_mla_decode_fp8(const void* q_bf16, float q_scale, const uint8_t* kv_pool_fp8, float k_scale,
                                     int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                     const int32_t* seq_lens, const int32_t* cu_q, int32_t B, const int32_t* idx,
                                     int32_t k, int32_t T, int32_t H, float scale, void* out_bf16, float* lse,
                                     void* workspace, size_t workspace_bytes, int32_t* dev_err, void* stream);

/*
 * dsa_sparse_attn_swa_cmp -- decode attention of the compressed-KV (DSV4) variant: a sliding window
 * of the original cache plus the selected compressed entries, with per-head attention sinks.
 * Source: vllm_ascend dsa_v1.py, AscendDSAImpl._forward_decode with compress_ratio 4:
 * attn_op(q, ori_kv = swa_kv_cache, cmp_kv = compress_kv_cache, cmp_sparse_indices =
 * compress_topk_idxs, ori_block_table, cmp_block_table, seqused_kv = seq_lens, sinks = attn_sink,
 * softmax_scale, cmp_ratio, ori_mask_mode = 4 (sliding window), cmp_mask_mode = 3,
 * ori_win_left = window_size - 1, ori_win_right = 0).
 *   For row r with visible length v (absolute position v - 1) and head h the keys are the
 *   original-cache positions max(0, v - window) .. v - 1 and the compressed entries
 *   cmp_idx[r, j] with 0 <= cmp_idx < v / cmp_ratio (others: -1 padding, or skipped with
 *   DSA_DEVERR_INDEX_RANGE); S_i = scale * <q[r,h], c_i> over the 576 dims;
 *   D = sum_i e^{S_i} + e^{sinks[h]};  out[r,h] = bf16_rn(sum_i e^{S_i} / D * c_i[0:512]);
 *   lse[r,h] = log D.  The rows of both caches are 576-wide latent rows (512 value + 64 rope dims,
 *   as dsa_sparse_mla_decode's cache); an entry in both sets counts twice (different vectors).
 * (The op's source is not printed: the union under one softmax, the sink in the denominator only,
 * and the 576-wide rows are the reading taken.)
 * Arguments:
 *   q_bf16           [T, H, 576] bf16.   swa_kv / cmp_kv  bf16 [pages, 64, 576] (16-byte aligned).
 *   swa_block_table  int32 [B, swa_max_pages] over token positions; cmp_block_table int32
 *                    [B, cmp_max_pages] over compressed entries.   seq_lens / cu_q as elsewhere.
 *   cmp_idx          int32 [T, k] compressed entries (dsa_lightning_indexer with DSA_KEYS_CMP4).
 *   window           1 .. 2048.   cmp_ratio a power of two 1 .. 128 (4 for the pages' indexed layers).
 *   sinks            fp32 [H] per-head sink logits (-inf: none).   H in {16, 32, 64, 128}.
 *   out_bf16 [T, H, 512]; lse fp32 [T, H] (nullable).
 *   workspace        >= dsa_sparse_attn_swa_cmp_workspace_size(T, H, window, k) bytes, 16-byte
 *                    aligned (split-K partials for small batches; 0 bytes, nullable, when each row
 *                    is one split).
 * One pass of the sparse-attention kernel over both key sets (the window positions computed in
 * the kernel, the compressed entries through their own cache, page table and visibility), the sink
 * folded into the softmax denominator of its epilogue; for small batches split over the entries,
 * with the sink added by the split-K combine.
 */
size_t dsa_sparse_attn_swa_cmp_workspace_size(int32_t T, int32_t H, int32_t window, int32_t k);
dsa_status dsa_sparse_attn_swa_cmp(const void* q_bf16, const void* swa_kv, int64_t swa_num_pages,
                                   const int32_t* swa_block_table, int32_t swa_max_pages, const void* cmp_kv,
                                   int64_t cmp_num_pages, const int32_t* cmp_block_table, int32_t cmp_max_pages,
                                   const int32_t* seq_lens, const int32_t* cu_q, int32_t B, const int32_t* cmp_idx,
                                   int32_t k, int32_t window, int32_t cmp_ratio, const float* sinks, int32_t T,
                                   int32_t H, float scale, void* out_bf16, float* lse, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_err, void* stream);

/*
 * dsa_mla_absorb_q -- absorbed latent query: ql[t, n, 0:512] = q_nope[t, n, 0:128] W_UK_T[n].
 * Source: vllm mla/common.py, MLACommonImpl.forward decode branch and _q_proj_and_k_up_proj
 * (torch.bmm(q_nope as (N, B, P), W_UK_T (N, P, L)); W_UK_T = W_UK.permute(1, 2, 0) where W_UK is
 * the qk_nope part of kv_b_proj's weight viewed (L, N, P)).
 *   ql[t, n, l] = bf16_rn(sum_{p < 128} q_nope[t, n, p] * W_UK_T[n, p, l]), bf16 operands,
 *   fp32 accumulation on the tensor cores.
 * Arguments:
 *   q_nope_bf16     element (t, n, p) at q_nope_bf16[t * q_row_stride + n * q_head_stride + p];
 *                   16-byte aligned; both strides multiples of 8 elements (e.g. the q_nope part of
 *                   a [T, H, 192] projection output: strides H * 192 and 192).
 *   w_uk_t_bf16     [H, 128, 512] bf16, contiguous, 16-byte aligned.
 *   ql_bf16         element (t, n, l) at ql_bf16[t * out_row_stride + n * out_head_stride + l];
 *                   e.g. the first 512 columns of the [T, H, 576] attention query (strides H * 576
 *                   and 576).  Distinct (t, n) outputs must not overlap.
 *   dev_err         nullable; DSA_DEVERR_TIMEOUT if a bounded wait gave up.
 */
dsa_status dsa_mla_absorb_q(const void* q_nope_bf16, int64_t q_row_stride, int64_t q_head_stride,
                            const void* w_uk_t_bf16, int32_t T, int32_t H, void* ql_bf16,
                            int64_t out_row_stride, int64_t out_head_stride, int32_t* dev_err,
                            void* stream);

/*
 * dsa_mla_v_up -- value up-projection of the latent attention output:
 * out[t, n, 0:128] = o_lat[t, n, 0:512] W_UV[n].
 * Source: vllm mla/common.py, MLACommonImpl._v_up_proj (torch.bmm(o_lat as (N, B, L), W_UV
 * (N, L, V)); W_UV = the v part of kv_b_proj's weight viewed (L, N, V), transposed to (N, L, V)).
 *   out[t, n, v] = bf16_rn(sum_{l < 512} o_lat[t, n, l] * W_UV[n, l, v]), fp32 accumulation.
 * Arguments:
 *   o_lat_bf16      element (t, n, l) at o_lat_bf16[t * o_row_stride + n * o_head_stride + l]
 *                   (dsa_sparse_mla_decode's output: strides H * 512 and 512); 16-byte aligned,
 *                   strides multiples of 8 elements.
 *   w_uv_bf16       [H, 512, 128] bf16, contiguous, 16-byte aligned.
 *   out_bf16        element (t, n, v) at out_bf16[t * out_row_stride + n * out_head_stride + v]
 *                   (e.g. [T, H * 128]: strides H * 128 and 128).
 *   dev_err         nullable; DSA_DEVERR_TIMEOUT if a bounded wait gave up.
 */
dsa_status dsa_mla_v_up(const void* o_lat_bf16, int64_t o_row_stride, int64_t o_head_stride,
                        const void* w_uv_bf16, int32_t T, int32_t H, void* out_bf16,
                        int64_t out_row_stride, int64_t out_head_stride, int32_t* dev_err, void* stream);

/*
 * dsa_read_device_error -- synchronise `stream`, copy the device error word to the host
 * (*host_word, nullable) and map it: 0 -> DSA_OK, a timeout bit -> DSA_ERR_TIMEOUT, any range
 * bit -> DSA_ERR_DEVICE_BOUNDS.  Does not clear the word.
 */
dsa_status dsa_read_device_error(const int32_t* dev_err, int32_t* host_word, void* stream);

/*
 * dsa_selftest_wait_timeout -- failure-detection self-test of the bounded waits.
 * The pipelined kernels (indexer logits, sparse MLA) synchronise their warps through mbarriers
 * and never wait without a limit: a wait that has not completed after its cycle budget gives up,
 * sets DSA_DEVERR_TIMEOUT in the error word and lets the kernel return.  This call runs one such
 * wait on a barrier that nothing ever arrives on, with a budget of `cycles` SM clock cycles
 * (1 .. 4e9), so that a test can check the timeout path end to end: afterwards *dev_err has
 * DSA_DEVERR_TIMEOUT set and the CUDA context is still usable.  No fault, trap or hang is involved.
 */
dsa_status dsa_selftest_wait_timeout(int32_t* dev_err, uint64_t cycles, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_GB300_DSA_H */
