// lightning_indexer.cu -- the indexer and the top-k behind one call that returns indices.
//
// Follows vllm_ascend sfa_v1.py, the indexer's npu_lightning_indexer call (query, paged key
// cache, weights, per-request query and key lengths, block table, sparse_count, sparse_mode = 3
// causal) that returns the top-k indices directly.  The two stages run as the kernels of
// dsa_indexer_logits and dsa_topk_forced, chained on the device by programmatic dependent launch;
// the logits live only in the caller's workspace.
#include "dsa_common.cuh"

namespace {

int64_t lightning_logits_ld(int32_t max_seq_len) { return max_seq_len < 4 ? 4 : (int64_t(max_seq_len) + 3) / 4 * 4; }

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

}  // namespace

extern "C" size_t dsa_lightning_indexer_workspace_size(int32_t T, int32_t max_seq_len) {
    if (T <= 0 || max_seq_len < 0) return 0;
    return align256(dsa_indexer_logits_workspace_size(T)) +
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
    const size_t idx_ws = align256(dsa_indexer_logits_workspace_size(T));
    float* logits = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + idx_ws);
    const int64_t ld = lightning_logits_ld(max_seq_len);
    dsa_status st = dsa_indexer_logits(q_bf16, weights, index_k_pool, num_pages, block_table, max_pages, seq_lens,
                                       cu_q, B, max_seq_len, max_q_len, 0, T, logits, ld, flags, workspace, idx_ws,
                                       dev_err, stream);
    if (st != DSA_OK) return st;
    return dsa_topk_forced(logits, ld, seq_lens, cu_q, B, max_seq_len, 0, T, k, n_init, n_local, idx, nullptr, 0,
                           stream);
}
