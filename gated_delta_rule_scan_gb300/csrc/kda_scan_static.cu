// kda_scan_static.cu -- the fixed device scratch behind kda_scan_varlen_static: one file-scope
// array per device, sized for modest chunked scans, so that the entry point allocates nothing.
// The array sits in a translation unit of its own, so its memory is claimed only by programs that
// use this entry point (the module holding it loads on first use).
#include <cuda_runtime.h>

#include "kda_internal.h"

namespace kda {

static __device__ __align__(256) unsigned char g_kda_static_scratch[kStaticScratchBytes];

cudaError_t static_scratch(void** ptr) {
    static PerDevice<void*> ptrs;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void* p = ptrs[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        // one-time setup on this device (the caller has made it current and checked that the
        // stream belongs to it)
        e = cudaGetSymbolAddress(&p, g_kda_static_scratch);
        if (e != cudaSuccess) return e;
        ptrs[dev].store(p, std::memory_order_release);
    }
    *ptr = p;
    return cudaSuccess;
}

}  // namespace kda
