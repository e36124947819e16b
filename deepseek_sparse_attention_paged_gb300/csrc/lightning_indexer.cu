// lightning_indexer.cu -- the indexer and the top-k behind one call that returns indices.
//
// Follows vllm_ascend sfa_v1.py, the indexer's npu_lightning_indexer call (query, paged key
// cache, weights, per-request query and key lengths, block table, sparse_count, sparse_mode = 3
// causal) that returns the top-k indices directly.
//
// Fused: the logits kernel also builds, per row, the histogram of the top 12 bits of its logits'
// order keys (in shared memory while it writes them, added into a zeroed per-row histogram in the
// workspace at the end of each row group); the top-k kernels start from that histogram instead of
// a first read of the row, so the row is read once less and the first digit's scan happens with
// no pass over the row.  The logits live only in the caller's workspace.  For row groups of more
// than 2 query rows (the histograms would not fit beside the key stages) or rows longer than
// 131072 keys the two calls run unfused.
//
// Workspace layout (offsets 256-byte aligned): the per-row histograms (T x 4096 uint32), the logits
// call's query scratch, then the logits (T rows, row stride max_seq_len rounded up to 4 floats).
#include "dsa_common.cuh"

namespace {

int64_t lightning_logits_ld(int32_t max_seq_len) { return max_seq_len < 4 ? 4 : (int64_t(max_seq_len) + 3) / 4 * 4; }

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

size_t hist_bytes(int32_t T) { return align256(static_cast<size_t>(T) * dsa::kHistBins * 4); }

// row groups of 1 or 2 rows (max_q_len < 4) and rows the one-pass top-k kernels take
bool fused_ok(int32_t max_seq_len, int32_t max_q_len) { return max_q_len < 4 && max_seq_len <= 131072; }

}  // namespace

extern "C" size_t dsa_lightning_indexer_workspace_size(int32_t T, int32_t max_seq_len) {
    if (T <= 0 || max_seq_len < 0) return 0;
    return hist_bytes(T) + align256(dsa_indexer_logits_workspace_size(T)) +
           static_cast<size_t>(T) * static_cast<size_t>(lightning_logits_ld(max_seq_len)) * 4;
}

extern "C" dsa_status dsa_lightning_indexer(const void* q_bf16, const float* weights, const uint8_t* index_k_pool,
                                            int64_t num_pages, const int32_t* block_table, int32_t max_pages,
                                            const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                                            int32_t max_seq_len, int32_t max_q_len, int32_t T, int32_t k,
                                            int32_t n_init, int32_t n_local, uint32_t flags, int32_t* idx,
                                            void* workspace, size_t ws_bytes, int32_t* dev_err, void* stream) {
    if (T < 0 || k < 1 || k > DSA_MAX_TOPK || n_init < 0 || n_local < 0) return DSA_ERR_INVALID_ARG;
    if (T == 0) return DSA_OK;
    if (!workspace || !idx || ws_bytes < dsa_lightning_indexer_workspace_size(T, max_seq_len))
        return DSA_ERR_INVALID_ARG;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    uint32_t* hist = reinterpret_cast<uint32_t*>(ws);
    const size_t idx_ws = align256(dsa_indexer_logits_workspace_size(T));
    void* logits_ws = ws + hist_bytes(T);
    float* logits = reinterpret_cast<float*>(ws + hist_bytes(T) + idx_ws);
    const int64_t ld = lightning_logits_ld(max_seq_len);
    const bool fused = fused_ok(max_seq_len, max_q_len);
    dsa_status st = dsa::indexer_logits_launch(q_bf16, weights, index_k_pool, num_pages, block_table, max_pages,
                                               seq_lens, cu_q, B, max_seq_len, max_q_len, 0, T, logits, ld, flags,
                                               logits_ws, idx_ws, dev_err, stream, fused ? hist : nullptr);
    if (st != DSA_OK) return st;
    return dsa::topk_launch(logits, ld, seq_lens, cu_q, B, max_seq_len, 0, T, k, n_init, n_local, idx, stream,
                            fused ? hist : nullptr, (flags & DSA_KEYS_CMP4) != 0u ? 2 : 0);
}
