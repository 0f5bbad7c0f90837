// Diagnostics: make one bounded device wait run out on purpose and report it.
//
// Every wait in the step's kernels (mbarrier phases fed by TMA copies and tensor-core
// commits) gives up after a time limit, sets KVP_ERRBIT_TIMEOUT and lets the kernel
// finish, instead of spinning forever.  This entry point exercises that path without
// faulting or hanging the GPU: one thread waits on an mbarrier that nothing arrives at,
// with a short limit, and the host reads whether the wait gave up.
#include <cuda_runtime.h>

#include "kvpaged.h"
#include "kvp_device.cuh"

namespace {

__global__ void bounded_wait_kernel(int* gave_up, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    kvp::mbar_init(&bar, 1);
    kvp::fence_barrier_init();
    const uint32_t a = kvp::smem_u32(&bar);
    const uint64_t t0 = kvp::global_ns();
    int result = 1;
    while (kvp::global_ns() - t0 <= limit_ns) {
        if (kvp::mbar_try_wait(a, 0)) {   // phase 0 never completes: no thread arrives
            result = 0;
            break;
        }
    }
    *gave_up = result;
}

}  // namespace

extern "C" KVP_API kvp_status kvp_selftest_bounded_wait(long long limit_ns, kvp_stream stream) {
    if (limit_ns <= 0 || limit_ns > 2000000000ll) return KVP_E_INVALID_ARG;
    int* d = nullptr;
    int h = -1;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMalloc(&d, sizeof(int)) != cudaSuccess) return KVP_E_CUDA;
    bounded_wait_kernel<<<1, 32, 0, s>>>(d, (unsigned long long)limit_ns);
    const bool ok = cudaGetLastError() == cudaSuccess &&
                    cudaMemcpyAsync(&h, d, sizeof(int), cudaMemcpyDeviceToHost, s) == cudaSuccess &&
                    cudaStreamSynchronize(s) == cudaSuccess;
    cudaFree(d);
    if (!ok) return KVP_E_CUDA;
    return h == 1 ? KVP_E_TIMEOUT : KVP_OK;
}
