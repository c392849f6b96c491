// Internal interface between the C-ABI front end (api.cpp) and the kernel
// translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "pa_varlen.h"

#ifndef PA_WAIT_LIMIT_NS
#define PA_WAIT_LIMIT_NS 2000000000ull  // a bounded wait gives up after 2 s of wall time
#endif

namespace pa {

// Validated, flattened arguments of one pa_varlen_fwd call (element strides).
struct Args {
    int dtype;  // PA_F16 or PA_BF16
    const void* q;
    int64_t q_s0, q_s1;
    const void* k;
    const void* v;
    // paged: strides of (block, slot, head); non-paged: (token, unused, head)
    int64_t kv_s0, kv_s1, kv_s2;
    bool paged;
    int64_t num_blocks;  // paged: k_cache.shape[0]; non-paged: total_k
    int page;            // page_block_size (0 when non-paged)
    const int32_t* cu_q;
    const int32_t* cu_k;
    int batch;
    const int32_t* block_table;
    int64_t bt_s0;
    int bt_cols;
    int max_sq, max_sk;
    int H, Hkv, D;
    float scale;
    int wl, wr;
    void* out;
    int64_t o_s0, o_s1;
    float* lse;
    int64_t lse_s0;
    int64_t lse_sb;  // per-sequence lse offset: 0 for (H, total_q); H Sq - Sq for (B, H, Sq)
    int64_t total_q;
    cudaStream_t stream;
    uint64_t wait_ns;    // bound on every in-kernel wait
    int withhold_loads;  // test hook: producers issue no loads
    const float* alibi;  // per-query-head slopes of the linear position bias, or nullptr
};

// Scratch the split-KV path needs for a call (bytes), and where to put it.
struct Workspace {
    void* ptr;
    size_t bytes;
};

// Launch plan of the split-KV kernel (host-chosen; device recomputes the per-tile view).
struct SplitPlan {
    int dp;           // padded head dim: 64, 128, 256, 512
    int mt;           // 16-row groups per CTA (1 or 2)
    int nt;           // keys per tile (64 or 32)
    int row_tiles;    // row tiles per (sequence, kv head)
    int rows_cap;     // sequences with sq*G above this belong to the tensor-core prefill kernel
    int tile_rows;    // most rows a row tile can hold: min(16 * mt, max_seqlen_q * G)
    int split_tiles;  // key tiles per split
    int max_splits;   // grid.x
    size_t ws_bytes;     // scratch needed: the longest-first order or the work list, then the partial results
    size_t order_bytes;  // bytes of the order at the start of the scratch (0: none)
    size_t work_bytes;   // bytes of the persistent decode work list after it (0: not persistent)
    int slots;           // resident CTAs of the split-KV kernel on the device (persistent grid)
    int rank_in_cta;     // decode kernel CTAs rank the batch themselves (small batches)
    int tc;              // decode class on the tensor-core decode kernel (128-key tiles)
    int work;            // decode class on the persistent warp-sliced kernel (device work list)
};

// The decode kernel launches sequences longest first: batches of at most kRankInCta
// sequences are ranked inside every CTA, larger ones up to kMaxOrderBatch by a one-CTA pass.
constexpr int kRankInCta = 160;
constexpr int kMaxOrderBatch = 1024;
// Most keys one split-KV CTA of the decode class takes (the plan's cap for skewed batches).
constexpr int64_t kMaxSplitKeys = 8192;
// Persistent decode mode (a device-built work list taken by one CTA per resident slot) for
// batches of at least kWorkMinBatch sequences whose plan splits some sequence.
constexpr int kWorkMinBatch = 16;
int launch_longest_first(const int32_t* cu_k, int batch, int* order, cudaStream_t stream, char* msg,
                         size_t msg_len);

// Dense-prefill (tcgen05) launch availability for these arguments.
bool prefill_supported(const Args& a);
int prefill_rows_threshold();  // sequences with sq*G > this go to the prefill kernel
// The prefill kernels are persistent (one CTA per SM over a device counter of work items):
// each call takes kPrefillCounterBytes of scratch for the counter, which launch_prefill
// zeroes on a.stream before the kernel.
constexpr size_t kPrefillCounterBytes = 256;
int launch_prefill(const Args& a, int* counter, unsigned int* err, char* msg, size_t msg_len);
// Upper bound of the prefill kernel's work items (its grid is min(SMs, items)).
int64_t prefill_items_bound(const Args& a);

// `prefill_takes_long_rows`: rows of sequences with sq*G above the threshold belong to the
// prefill kernel; `prefill_sms`: SMs the prefill kernel's grid may hold while this pass
// runs (0 when the prefill kernel runs before it).
SplitPlan plan_splitkv(const Args& a, bool prefill_takes_long_rows, int prefill_sms, int num_sms);
int launch_splitkv(const Args& a, const SplitPlan& plan, void* workspace, unsigned int* err, char* msg,
                   size_t msg_len);
int launch_splitkv_bf16(const Args& a, const SplitPlan& plan, void* workspace, unsigned int* err, char* msg,
                        size_t msg_len);
// Resident CTAs per SM of the split-KV kernel `plan` dispatches to (dp, mt, row_tiles set).
int splitkv_occupancy_bf16(const SplitPlan& plan);
int splitkv_occupancy_f16(const SplitPlan& plan);
// Resident CTAs per SM of the tensor-core decode kernel (padded head dim dp, nr rows).
int decode_tc_occupancy(int dtype, int dp, int nr);
// Whether decode-class rows (one row tile of at most 32 rows) of padded head dim `dp` >= 128
// go to the tensor-core decode kernel: when the PA_DECODE_TC environment variable is 1 (a
// switch between two complete kernels; off by default, where the other kernels measured faster).
bool decode_tc_wanted(int dp);
int launch_splitkv_f16(const Args& a, const SplitPlan& plan, void* workspace, unsigned int* err, char* msg,
                       size_t msg_len);

// Device address (current device) of the library's error word, which kernels set
// with the first PA_ERR_DEVICE_* code they meet (bit 31 = set).  Returns a cudaError_t.
int error_word(unsigned int** ptr);

// Counts successful kernel launches (pa_kernel_launches).
void count_launches(int n);

// KV append (pa_kv_append): validated arguments, element strides.
struct AppendArgs {
    const void* k_new;
    const void* v_new;
    int64_t kn_s0, kn_s1, vn_s0, vn_s1;  // (token, head) strides of k_new / v_new
    void* k_cache;
    void* v_cache;
    int64_t c_s0, c_s1, c_s2;  // (block, slot, head) strides shared by both caches
    const int32_t* cu_new;
    const int32_t* cu_k;
    const int32_t* bt;
    int64_t bt_s0;
    int bt_cols;
    int batch;
    int64_t total_new;
    int64_t num_blocks;
    int P, Hkv, D;
    cudaStream_t stream;
};
int launch_kv_append(const AppendArgs& a, unsigned int* err, char* msg, size_t msg_len);

// Per-kernel timing (pa_kernel_timing): timer_begin before a launch of kernel class `cls`
// (PA_KC_*) into `stream`, timer_end after it launched successfully.  Both do nothing
// unless timing is on.
void timer_begin(int cls, cudaStream_t stream);
void timer_end(int cls, cudaStream_t stream);

// Supplier of the split-KV scratch for one call: sets *ptr to at least `bytes` bytes of
// device memory usable on `stream`, or returns a status with a message in msg.
using ScratchFn = int (*)(void* ctx, cudaStream_t stream, size_t bytes, void** ptr, char* msg, size_t msg_len);

// NVTX range around a scope (a call, a launch), visible to profilers that record NVTX;
// costs a function-pointer check when no tool is attached.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// Validation and dispatch shared by the C entry points (api.cpp).  `side_stream_ok`: a
// batch with prefill-class sequences may fork its prefill kernel onto a side stream of the
// caller's stream (created on first use); when false, both kernels run on `stream`, one
// after the other, and nothing is created.
int launch_forward(Args& a, void* stream, ScratchFn scratch, void* scratch_ctx, bool side_stream_ok);
int launch_uniform_cu(int32_t* cu_q, int32_t* cu_k, int batch, int sq, int sk, cudaStream_t stream, char* msg,
                      size_t msg_len);
int forward_impl(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                 const pa_tensor* cu_seqlens_q, const pa_tensor* cu_seqlens_k, const pa_tensor* block_table,
                 int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_heads, int32_t num_heads_k,
                 int32_t head_dim, int32_t page_block_size, float softmax_scale, int32_t window_left,
                 int32_t window_right, const pa_tensor* alibi_slopes, const pa_tensor* out,
                 const pa_tensor* softmax_lse, void* stream, ScratchFn scratch, void* scratch_ctx,
                 bool side_stream_ok);

// Tensor-map encoding through the driver entry point (no libcuda link needed).
// Rank-4 bf16/f16 map over (d0 fastest .. d3), strides in bytes for dims 1..3.
int encode_tmap_4d(void* map, int dtype, const void* base, const uint64_t dims[4], const uint64_t strides_bytes[3],
                   const uint32_t box[4], int swizzle128, char* msg, size_t msg_len);

}  // namespace pa
