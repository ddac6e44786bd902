// Batched copy: up to CSA_COPY_MAX copies in one kernel launch, each between device memory and/or
// page-locked host memory that the device can address (a pinned allocation; with unified virtual
// addressing its host pointer is its device pointer, and the kernel reaches host memory over
// NVLink-C2C).  A decode step's per-step uploads (the new token's inputs, its raw rows, its index
// row) and its download (the outputs) are a few small copies; as separate copy-engine operations
// each costs a copy's fixed latency, one after another in the stream, while one kernel moves them
// all with every 16-byte chunk's load in flight together.
#include "common.cuh"
#include "internal.h"

namespace csa {

struct CopyArgs {
    csa_copy c[CSA_COPY_MAX];
    int n;
};

// Thread t of the grid takes 16-byte chunks t, t + stride, ... of the copies laid end to end;
// four loads go out before their stores.
__global__ void __launch_bounds__(256) copy_batch_kernel(CopyArgs a) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t t0 = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint64_t base = 0;
    for (int i = 0; i < a.n; ++i) {
        const uint64_t n16 = a.c[i].bytes / 16;
        const uint4* src = static_cast<const uint4*>(a.c[i].src);
        uint4* dst = static_cast<uint4*>(a.c[i].dst);
        // this thread's first chunk of copy i
        uint64_t j = t0 >= base ? t0 - base : (stride - (base - t0) % stride) % stride;
        for (; j + 3 * stride < n16; j += 4 * stride) {
            const uint4 v0 = src[j], v1 = src[j + stride], v2 = src[j + 2 * stride], v3 = src[j + 3 * stride];
            dst[j] = v0;
            dst[j + stride] = v1;
            dst[j + 2 * stride] = v2;
            dst[j + 3 * stride] = v3;
        }
        for (; j < n16; j += stride) dst[j] = src[j];
        base += n16;
    }
}

}  // namespace csa

extern "C" csa_status csa_copy_batch(int32_t n, const csa_copy* copies, void* stream) {
    using namespace csa;
    if (n < 1 || n > CSA_COPY_MAX || !copies) return CSA_ERR_INVALID_ARG;
    CopyArgs a;
    a.n = n;
    uint64_t total = 0;
    for (int i = 0; i < n; ++i) {
        const csa_copy& c = copies[i];
        if (!c.src || !c.dst || (reinterpret_cast<uintptr_t>(c.src) & 15u) || (reinterpret_cast<uintptr_t>(c.dst) & 15u) ||
            (c.bytes & 15u))
            return CSA_ERR_INVALID_ARG;
        a.c[i] = c;
        total += c.bytes / 16;
    }
    if (total == 0) return CSA_OK;
    const int sms = device_sm_count();
    if (!sms) return CSA_ERR_CUDA;
    uint64_t blocks = (total + 4 * 256 - 1) / (4 * 256);  // about four chunks per thread
    if (blocks > (uint64_t)sms * 8) blocks = (uint64_t)sms * 8;
    if (blocks < 1) blocks = 1;
    copy_batch_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
    return cudaGetLastError() == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}
