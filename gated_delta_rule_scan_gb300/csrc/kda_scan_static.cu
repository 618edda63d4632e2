// kda_scan_static.cu -- the fixed device scratch behind kda_scan_varlen_static: one file-scope
// array per device, sized for modest chunked scans, so that the entry point allocates nothing.
// The array sits in a translation unit of its own, so its memory is claimed only by programs that
// use this entry point (the module holding it loads on first use).
#include <cuda_runtime.h>

#include "kda_internal.h"

namespace kda {

static __device__ __align__(256) unsigned char g_kda_static_scratch[kStaticScratchBytes];

cudaError_t static_scratch(void** ptr) {
    static void* ptrs[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (ptrs[dev] == nullptr) {
        // one-time setup on this device (the caller has made it current)
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_kda_static_scratch);
        if (e != cudaSuccess) return e;
        ptrs[dev] = p;
    }
    *ptr = ptrs[dev];
    return cudaSuccess;
}

}  // namespace kda
