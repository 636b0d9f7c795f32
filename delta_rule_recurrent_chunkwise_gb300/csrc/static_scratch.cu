// static_scratch.cu -- the library-owned device buffer behind
// la_prefill_delta_static, alone in its translation unit.
//
// Without relocatable device code every .cu file is its own CUDA module.
// Keeping this buffer apart from the kernels and the device error word means
// that, under lazy module loading (the CUDA runtime's default), only a
// process that calls la_prefill_delta_static loads this module and so
// reserves the buffer (LA_STATIC_SCRATCH_BYTES on each device it calls it
// on, held until the process exits).  Under eager loading
// (CUDA_MODULE_LOADING=EAGER) every device the process initialises
// reserves it at context creation.

#include <atomic>

#include "launch.h"

namespace la {

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

void *static_scratch() {
    // Device address per device, looked up with that device current.  Two
    // host threads making their first call at once both store the same
    // address; a failed lookup is retried on the next call.
    static std::atomic<void *> addr[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    void *p = addr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return nullptr;
        addr[dev].store(p, std::memory_order_release);
    }
    return p;
}

}  // namespace la
