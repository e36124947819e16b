// dsa_api.cu -- status strings and the device error word reader of the C ABI.
#include "dsa_common.cuh"

extern "C" const char* dsa_status_str(dsa_status s) {
    switch (s) {
        case DSA_OK: return "ok";
        case DSA_ERR_INVALID_ARG: return "invalid argument";
        case DSA_ERR_UNSUPPORTED: return "unsupported configuration";
        case DSA_ERR_CUDA: return "CUDA error";
        case DSA_ERR_DEVICE_BOUNDS: return "device reported out-of-range accesses (skipped)";
        case DSA_ERR_TIMEOUT: return "device reported a bounded wait that gave up";
        default: return "unknown status";
    }
}

extern "C" dsa_status dsa_read_device_error(const int32_t* dev_err, int32_t* host_word, void* stream) {
    if (dev_err == nullptr) return DSA_ERR_INVALID_ARG;
    int32_t word = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&word, dev_err, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess) return DSA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DSA_ERR_CUDA;
    if (host_word != nullptr) *host_word = word;
    if (word & DSA_DEVERR_TIMEOUT) return DSA_ERR_TIMEOUT;
    if (word != 0) return DSA_ERR_DEVICE_BOUNDS;
    return DSA_OK;
}
