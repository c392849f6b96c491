// pa_varlen_fwd_noalloc: the forward call for callers that must not allocate device
// memory.  The split-KV path needs scratch for per-split partial results; instead of
// the library's cudaMalloc'd workspace, this entry point uses one fixed array that is
// part of the library's device image, so every device that loads the library holds it
// (PA_NOALLOC_SCRATCH_BYTES) until the process exits.  It creates no stream or event
// either: a batch with prefill-class sequences runs its prefill kernel and its split-KV
// pass one after the other on the caller's stream.
#include <cstdio>
#include <mutex>

#include "pa_internal.h"

#define PA_NOALLOC_SCRATCH_BYTES (32u << 20)  // 32 MiB

namespace pa {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device.  The host-side symbol
// g_noalloc_scratch is only a stand-in and must never be handed to a kernel; the first
// call on each device looks the real address up (cudaGetSymbolAddress allocates
// nothing) and caches it.
int scratch_address(void** ptr, char* msg, size_t msg_len) {
    static std::mutex mu;
    static void* cached[256] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "cudaGetDevice: %s", cudaGetErrorString(e));
        return PA_ERR_CUDA;
    }
    if (dev < 0 || dev >= 256) {
        snprintf(msg, msg_len, "device ordinal %d out of range", dev);
        return PA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            snprintf(msg, msg_len, "cudaGetSymbolAddress(no-allocation scratch): %s", cudaGetErrorString(e));
            return PA_ERR_CUDA;
        }
        cached[dev] = p;
    }
    *ptr = cached[dev];
    return PA_OK;
}

int static_scratch(void*, cudaStream_t, size_t bytes, void** ptr, char* msg, size_t msg_len) {
    if (bytes > PA_NOALLOC_SCRATCH_BYTES) {
        snprintf(msg, msg_len,
                 "this call needs %zu bytes of scratch; pa_varlen_fwd_noalloc has %u bytes (use "
                 "pa_varlen_fwd, fewer sequences per call, or a shorter max_seqlen_k)",
                 bytes, (unsigned)PA_NOALLOC_SCRATCH_BYTES);
        return PA_ERR_WORKSPACE;
    }
    // Every slot the combine reads is written by the split kernel of the same call, so
    // the scratch needs no clearing between calls.
    return scratch_address(ptr, msg, msg_len);
}

}  // namespace
}  // namespace pa

extern "C" int pa_varlen_fwd_noalloc(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                                     const pa_tensor* cu_seqlens_q, const pa_tensor* cu_seqlens_k,
                                     const pa_tensor* block_table, int32_t max_seqlen_q, int32_t max_seqlen_k,
                                     int32_t num_heads, int32_t num_heads_k, int32_t head_dim,
                                     int32_t page_block_size, float softmax_scale, int32_t window_left,
                                     int32_t window_right, const pa_tensor* out, const pa_tensor* softmax_lse,
                                     void* stream) {
    return pa::forward_impl(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_table, max_seqlen_q,
                            max_seqlen_k, num_heads, num_heads_k, head_dim, page_block_size, softmax_scale,
                            window_left, window_right, nullptr, out, softmax_lse, stream, pa::static_scratch,
                            nullptr, false);
}
