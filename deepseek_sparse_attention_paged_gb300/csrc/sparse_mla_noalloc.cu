// sparse_mla_noalloc.cu -- sparse MLA decode for callers that may not allocate device memory.
//
// Some callers of this library cannot call cudaMalloc (or any allocator) when they run the
// attention: an inference-engine plugin whose per-step "enqueue" hook is forbidden to allocate
// because the host engine owns every byte of device memory and budgets it up front; a serving
// loop that has given all free memory to its own caching allocator.  They still own the inputs and
// outputs, but have nowhere to get the split-K scratch that dsa_sparse_mla_decode() takes as
// `workspace`.
//
// dsa_sparse_mla_decode_noalloc() serves them: it runs exactly the same kernels as
// dsa_sparse_mla_decode(), with the scratch taken from the fixed array below, which the CUDA
// module holds on every GPU that loads the library until the process exits.
#include <atomic>

#include "dsa_common.cuh"

namespace dsa {
namespace {

// 16 MiB of split-K scratch (partial outputs and their log-sum-exps).
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_mla_scratch[kNoAllocScratchBytes];

// Device address of g_mla_scratch, per device ordinal.  In host code the name g_mla_scratch is a
// host-side stand-in, not a device address, so it is never passed to a kernel; the address comes
// from cudaGetSymbolAddress, taken once per device with that device current.  Under lazy module
// loading that first lookup also loads this library's device code on the device, which is when
// the array is placed in device memory (and can fail for lack of it).  Concurrent first calls on
// one device may both look it up; they store the same value.
std::atomic<void*> g_scratch_addr[kMaxDevices];

dsa_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSA_ERR_CUDA;
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        if (cudaGetSymbolAddress(&p, g_mla_scratch) != cudaSuccess || p == nullptr) return DSA_ERR_CUDA;
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return DSA_OK;
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_sparse_mla_decode_noalloc(const void* q_bf16, const void* kv_pool, int64_t num_pages,
                                                    const int32_t* block_table, int32_t max_pages,
                                                    const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                                                    const int32_t* idx, int32_t k, int32_t T, int32_t H,
                                                    float scale, void* out_bf16, float* lse, int32_t* dev_err,
                                                    void* stream) {
    if (k < 1 || k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
    if (H != 16 && H != 32 && H != 64 && H != 128) return DSA_ERR_UNSUPPORTED;
    if (T < 0) return DSA_ERR_INVALID_ARG;
    if (T == 0) return DSA_OK;
    // the problem must fit the fixed scratch: reject it rather than overrun the array
    if (dsa_sparse_mla_workspace_size(T, H, k) > dsa::kNoAllocScratchBytes) return DSA_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const dsa_status st = dsa::scratch_address(&scratch);
    if (st != DSA_OK) return st;
    // The split kernel writes every partial output and log-sum-exp it later reads, so nothing in
    // the scratch has to start at zero and the previous call's contents are never read.
    return dsa_sparse_mla_decode(q_bf16, kv_pool, num_pages, block_table, max_pages, seq_lens, cu_q, B, idx, k, T,
                                 H, scale, out_bf16, lse, scratch, dsa::kNoAllocScratchBytes, dev_err, stream);
}
