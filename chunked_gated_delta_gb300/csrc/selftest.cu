// selftest.cu -- a check of the kernels' bounded pipeline wait: one CTA waits
// on an mbarrier that nothing arrives on, with a short limit, and records the
// timeout exactly as the intra / scan kernels do.  No trap, no fault: the wait
// ends by itself and the context stays usable.
#include "../../include/kda.h"
#include "common.cuh"
#include "ptx.cuh"

namespace kda {
namespace {

__global__ void kda_wait_timeout_kernel(int32_t* status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    bool ok = true;
    if (threadIdx.x == 0) ok = ptx::mbar_wait(&bar, 0, limit_ns);  // phase 0 never completes
    if (!ok) atomicOr(status, kStatusTimeout);
}

}  // namespace
}  // namespace kda

extern "C" kda_status kda_selftest_wait_timeout(void* status_word, unsigned long long limit_ns,
                                                void* stream) {
    if (!status_word || (reinterpret_cast<uintptr_t>(status_word) & 3) != 0) return KDA_ERR_INVALID_ARG;
    if (limit_ns == 0 || limit_ns > kda::kWaitLimitNs) return KDA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t* st = static_cast<int32_t*>(status_word);
    if (cudaMemsetAsync(st, 0, sizeof(int32_t), s) != cudaSuccess) return KDA_ERR_CUDA;
    kda::kda_wait_timeout_kernel<<<1, 32, 0, s>>>(st, limit_ns);
    if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
    return kda_fwd_status(status_word, stream);
}
