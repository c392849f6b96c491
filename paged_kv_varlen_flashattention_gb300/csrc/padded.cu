// Small helper kernels of the host-side plan, launched on the call's stream right before
// the kernels that read their output:
//  * uniform cumulative sequence lengths for the padded (non-varlen) entry point: every
//    sequence of the batch has sq queries and sk keys, so cu_q[b] = b sq, cu_k[b] = b sk;
//  * the longest-first order of a batch's sequences for the decode kernel.
#include <cstdio>

#include "pa_internal.h"

namespace pa {
namespace {

__global__ void uniform_cu_kernel(int32_t* cu_q, int32_t* cu_k, int batch, int sq, int sk) {
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b <= batch; b += gridDim.x * blockDim.x) {
        cu_q[b] = b * sq;
        cu_k[b] = b * sk;
    }
}

// order[r] = the sequence of rank r when sequences are sorted by key count, longest first
// (ties by index).  One CTA; each thread ranks its sequences by counting the batch, so the
// result is a permutation whatever cu_k holds.
constexpr int kOrderThreads = 1024;

__global__ void __launch_bounds__(kOrderThreads) longest_first_kernel(const int32_t* cu_k, int batch, int* order) {
    __shared__ int len[kMaxOrderBatch];
    for (int i = threadIdx.x; i < batch; i += kOrderThreads) len[i] = cu_k[i + 1] - cu_k[i];
    __syncthreads();
    for (int s = threadIdx.x; s < batch; s += kOrderThreads) {
        const int ls = len[s];
        int rank = 0;
        for (int t = 0; t < batch; ++t) {
            const int lt = len[t];
            rank += (lt > ls) || (lt == ls && t < s);
        }
        order[rank] = s;
    }
}

}  // namespace

int launch_longest_first(const int32_t* cu_k, int batch, int* order, cudaStream_t stream, char* msg, size_t msg_len) {
    if (batch < 1 || batch > kMaxOrderBatch) {
        snprintf(msg, msg_len, "longest-first order: batch %d outside [1, %d]", batch, kMaxOrderBatch);
        return PA_ERR_UNSUPPORTED;
    }
    NvtxRange nv("pa::longest_first_kernel");
    longest_first_kernel<<<1, kOrderThreads, 0, stream>>>(cu_k, batch, order);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "longest-first order launch: %s", cudaGetErrorString(e));
        return PA_ERR_CUDA;
    }
    count_launches(1);
    return PA_OK;
}

int launch_uniform_cu(int32_t* cu_q, int32_t* cu_k, int batch, int sq, int sk, cudaStream_t stream, char* msg,
                      size_t msg_len) {
    const int threads = 256, blocks = (batch + 1 + threads - 1) / threads;
    NvtxRange nv("pa::uniform_cu_kernel");
    uniform_cu_kernel<<<blocks, threads, 0, stream>>>(cu_q, cu_k, batch, sq, sk);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "uniform cu_seqlens launch: %s", cudaGetErrorString(e));
        return PA_ERR_CUDA;
    }
    count_launches(1);
    return PA_OK;
}

}  // namespace pa
