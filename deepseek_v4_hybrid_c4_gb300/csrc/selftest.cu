// Failure-detection self-test: a wait that nothing can satisfy.  The mbarrier's first phase
// never completes, so the bounded wait (the one every kernel of the library uses) runs out,
// records CSA_ERR_TIMEOUT in the device status word and the kernel returns: no trap, no fault,
// and the context stays usable.
#include "common.cuh"
#include "internal.h"

namespace csa {

__global__ void bounded_wait_selftest_kernel(int32_t* status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncthreads();
    // the library's own bound is about 8 s; the self-test waits about a second
    if (!mbar_wait(smem_u32(&bar), 0u, 1u << 18) && threadIdx.x == 0) raise_status(status, CSA_ERR_TIMEOUT);
}

}  // namespace csa

extern "C" csa_status csa_selftest_bounded_wait(void* stream) {
    int32_t* st = csa::device_status_ptr();
    if (!st) return CSA_ERR_CUDA;
    csa::bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(st);
    return cudaGetLastError() == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}
