// Uniform cumulative sequence lengths for the padded (non-varlen) entry point: every
// sequence of the batch has sq queries and sk keys, so cu_q[b] = b sq and cu_k[b] = b sk.
// Written on the call's stream right before the attention kernels read them.
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

}  // namespace

int launch_uniform_cu(int32_t* cu_q, int32_t* cu_k, int batch, int sq, int sk, cudaStream_t stream, char* msg,
                      size_t msg_len) {
    const int threads = 256, blocks = (batch + 1 + threads - 1) / threads;
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
