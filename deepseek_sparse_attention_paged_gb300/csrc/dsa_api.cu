// dsa_api.cu -- status strings, the device error word reader and the bounded-wait self-test of the
// C ABI.
#include "dsa_common.cuh"
#include "sm100_ptx.cuh"

namespace dsa {
namespace {

// Waits on an mbarrier that nothing ever arrives on, with the same bounded wait the pipelined
// kernels use; the wait must give up after `cycles` SM clock cycles and report the timeout in the
// error word instead of hanging.
__global__ void selftest_wait_kernel(int32_t* err, unsigned long long cycles) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::fence_barrier_init();
    }
    __syncthreads();
    const uint64_t deadline = ptx::wait_deadline(cycles);
    if (!ptx::mbar_wait(&bar, 0, deadline) && threadIdx.x == 0) raise_error(err, DSA_DEVERR_TIMEOUT);
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status dsa_selftest_wait_timeout(int32_t* dev_err, uint64_t cycles, void* stream) {
    if (dev_err == nullptr || cycles == 0 || cycles > 4000000000ull) return DSA_ERR_INVALID_ARG;
    dsa::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_err, cycles);
    return dsa::launch_status();
}

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
