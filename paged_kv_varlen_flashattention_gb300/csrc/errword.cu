// The library's device error word.  Kernels record the first PA_ERR_DEVICE_* code they
// meet here (bounded-wait timeouts, out-of-range metadata); pa_device_status() reads
// and clears it.  One copy per device that loads the library.
#include <mutex>

#include "pa_internal.h"

namespace pa {

static __device__ unsigned int g_error_word;

int error_word(unsigned int** ptr) {
    static std::mutex mu;
    static unsigned int* cached[256] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= 256) return (int)cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_error_word);
        if (e != cudaSuccess) return (int)e;
        cached[dev] = static_cast<unsigned int*>(p);
    }
    *ptr = cached[dev];
    return (int)cudaSuccess;
}

}  // namespace pa
