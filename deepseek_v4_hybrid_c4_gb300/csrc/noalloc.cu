// csa_decode_noalloc: the fused decode step for callers that cannot allocate
// device memory themselves (code running inside an allocator or memory-pool
// callback, a host that hands the library only its input and output buffers,
// an embedding that forbids cudaMalloc after start-up).  The step's scratch
// (index scores, the radix histogram, the selection when the caller passes none,
// the attention split partials) lives in one fixed array in this library's
// device memory instead of a caller-provided workspace.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "csa.h"

namespace csa {

// Largest workspace a call may need, in bytes.  Every device that loads the
// library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
static void* g_noalloc_ptr[kNoAllocMaxDevices];
static std::mutex g_noalloc_mu;

// Device address of the scratch array for the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once per
// device (with that device current) and cached.
static void* noalloc_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_noalloc_ptr[dev] = p;
    }
    return g_noalloc_ptr[dev];
}

}  // namespace csa

extern "C" csa_status csa_decode_noalloc(const csa_decode_params* p, void* stream) {
    const size_t need = csa_decode_workspace_size(p);
    if (need == 0) return csa_decode(p, nullptr, 0, stream);  // rejected parameters: csa_decode reports why
    if (need > csa::kNoAllocScratchBytes) return CSA_ERR_WORKSPACE;
    void* scratch = csa::noalloc_scratch();
    if (!scratch) return CSA_ERR_CUDA;
    return csa_decode(p, scratch, csa::kNoAllocScratchBytes, stream);
}
