// KV append: writes new key/value tokens into their pages (the step before the attention
// call in a serving loop).  Sequence b owns sk_b keys after the append, the last n_b of
// which are its new tokens, so new token t sits at logical key sk_b - n_b + t -- the same
// bottom-right alignment as the attention mask -- at slot (pos mod P) of block
// block_table[b, pos / P] (the block-table mapping of "flash-attn-varlen paged expects k/v
// tensors of rank 4", What it means).
//
// HBM-bound byte copy: each warp takes a contiguous run of tokens, finds the first one's
// sequence by a warp-wide search over cu_seqlens_new and walks on from there; the token's
// Hkv * D elements are moved in 16-byte units, consecutive lanes on consecutive units of
// the same (token, head) row, for K and then V.  Streaming loads and stores keep the copy
// out of L1.
#include <algorithm>
#include <cstdio>

#include "device_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kAppendThreads = 256;  // 8 warps
constexpr int kAppendCtasPerSm = 8;

__global__ void __launch_bounds__(kAppendThreads) kv_append_kernel(const AppendArgs a, unsigned int* err) {
    const int lane = threadIdx.x & 31;
    const int64_t warp_id = (int64_t)blockIdx.x * (kAppendThreads / 32) + (threadIdx.x >> 5);
    const int64_t n_warps = (int64_t)gridDim.x * (kAppendThreads / 32);
    const int64_t per_warp = (a.total_new + n_warps - 1) / n_warps;
    const int64_t t0 = warp_id * per_warp, t1 = min64(a.total_new, t0 + per_warp);
    if (t0 >= t1) return;
    // the sequence of token t0, the last b < batch with cu_new[b] <= t0: a 32-way search,
    // one probe per lane and round, so a batch of B sequences costs log32(B) dependent loads
    int lo = 0, span = a.batch;  // the answer is in [lo, lo + span)
    while (span > 1) {
        const int step = (span + 31) / 32;
        const int idx = lo + lane * step;
        const bool le = idx < lo + span && a.cu_new[idx] <= t0;
        const unsigned ok = __ballot_sync(0xffffffffu, le);
        const int last = ok ? 31 - __clz((int)ok) : 0;  // cu_new[lo] <= t0 always holds
        lo += last * step;
        span = min(step, span - last * step);
    }
    int b = lo;
    const int units = a.Hkv * (a.D / 8);  // 16-byte units per token
    const int upr = a.D / 8;              // units per (token, head) row
    int nb_end = a.cu_new[b + 1];
    for (int64_t t = t0; t < t1; ++t) {
        while (t >= nb_end && b + 1 < a.batch) {  // next sequence with tokens
            ++b;
            nb_end = a.cu_new[b + 1];
        }
        const int n_b = nb_end - a.cu_new[b];
        const int sk_b = a.cu_k[b + 1] - a.cu_k[b];
        const int64_t t_loc = t - a.cu_new[b];  // index among the sequence's new tokens
        const int64_t pos = (int64_t)sk_b - n_b + t_loc;
        const int64_t page = pos >= 0 ? pos / a.P : -1;
        int blk = -1;
        if (t_loc >= 0 && t_loc < n_b && n_b <= sk_b && pos >= 0 && page < a.bt_cols)
            blk = a.bt[(int64_t)b * a.bt_s0 + page];
        if (blk < 0 || blk >= a.num_blocks) {
            if (lane == 0) flag_error(err, PA_ERR_DEVICE_BOUNDS);
            continue;
        }
        const int64_t slot = pos - page * a.P;
        const int64_t dst_row = (int64_t)blk * a.c_s0 + slot * a.c_s1;
        // up to 4 units per lane in flight: every load of the batch before its stores
        for (int base = 0; base < units; base += 4 * 32) {
            int4 kr[4], vr[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int u = base + i * 32 + lane;
                if (u < units) {
                    const int h = u / upr, c = u - h * upr;
                    kr[i] = __ldcs(reinterpret_cast<const int4*>(static_cast<const uint16_t*>(a.k_new) + t * a.kn_s0 +
                                                                 (int64_t)h * a.kn_s1 + c * 8));
                    vr[i] = __ldcs(reinterpret_cast<const int4*>(static_cast<const uint16_t*>(a.v_new) + t * a.vn_s0 +
                                                                 (int64_t)h * a.vn_s1 + c * 8));
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int u = base + i * 32 + lane;
                if (u < units) {
                    const int h = u / upr, c = u - h * upr;
                    const int64_t dst = dst_row + (int64_t)h * a.c_s2 + c * 8;
                    __stcs(reinterpret_cast<int4*>(static_cast<uint16_t*>(a.k_cache) + dst), kr[i]);
                    __stcs(reinterpret_cast<int4*>(static_cast<uint16_t*>(a.v_cache) + dst), vr[i]);
                }
            }
        }
    }
}

}  // namespace

int launch_kv_append(const AppendArgs& a, unsigned int* err, char* msg, size_t msg_len) {
    if (a.total_new == 0 || a.batch == 0) return PA_OK;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "kv append: %s", cudaGetErrorString(e));
        return PA_ERR_CUDA;
    }
    // one token per warp while that fits in one wave of resident CTAs (each token's
    // metadata is a chain of dependent loads), else the wave with several tokens per warp
    const int64_t want = (a.total_new + kAppendThreads / 32 - 1) / (kAppendThreads / 32);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sms * kAppendCtasPerSm));
    NvtxRange nv("pa::kv_append_kernel");
    timer_begin(PA_KC_APPEND, a.stream);
    kv_append_kernel<<<grid, kAppendThreads, 0, a.stream>>>(a, err);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "kv append launch: %s", cudaGetErrorString(e));
        return PA_ERR_CUDA;
    }
    timer_end(PA_KC_APPEND, a.stream);
    count_launches(1);
    return PA_OK;
}

}  // namespace pa
