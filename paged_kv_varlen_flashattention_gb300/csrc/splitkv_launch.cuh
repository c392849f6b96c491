// Host-side launch of the split-KV kernel and the combine kernel for one element
// type.  Included by one translation unit per type so the instantiations compile
// in parallel.
#pragma once

#include <cstdio>

#include <cstdlib>

#include "decode_kernel.cuh"
#include "decode_wide.cuh"

namespace pa {

template <int DP>
struct SplitShape;  // tile width, pipeline depth and warps per padded head dim
template <>
struct SplitShape<64> {
    static constexpr int NT = 64, STAGES = 4, NW = 4;
};
template <>
struct SplitShape<128> {
    static constexpr int NT = 64, STAGES = 3, NW = 4;
};
template <>
struct SplitShape<256> {
    static constexpr int NT = 64, STAGES = 3, NW = 4;
};
template <>
struct SplitShape<512> {
    // 3 stages would exceed 227 KB with a 32-row Q tile; 8 warps (253 registers a thread
    // with 4: the issue latency of the MMA chains, not the loads, bounded the kernel)
    static constexpr int NT = 32, STAGES = 2, NW = 8;
};

// The combine as a programmatic dependent launch of the split kernel before it on the
// stream: its launch and prologue overlap that kernel's tail (it waits in griddepcontrol
// before touching the partial results).
template <typename T, int M, int NT>
static cudaError_t launch_combine(dim3 grid, const SplitParams& sp, cudaStream_t stream) {
    NvtxRange nv("pa::combine_kernel");
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, combine_kernel<T, M, NT>, sp);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

template <typename T, int DP, int MT>
static int run_splitkv(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& sp, const SplitPlan& plan,
                       cudaStream_t stream, char* msg, size_t msg_len) {
    constexpr int NT = SplitShape<DP>::NT, STAGES = SplitShape<DP>::STAGES, NW = SplitShape<DP>::NW;
    using C = SplitCfg<DP, MT, NT, STAGES, NW>;
    auto kern = splitkv_kernel<T, DP, MT, NT, STAGES, NW>;
    static bool configured = false;  // attribute set once per process (per instantiation)
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "cudaFuncSetAttribute(split-KV, %d bytes): %s", C::SMEM, cudaGetErrorString(e));
            return PA_ERR_CUDA;
        }
        configured = true;
    }
    dim3 grid(plan.max_splits, sp.Hkv * plan.row_tiles, sp.batch);
    NvtxRange nv("pa::splitkv_kernel");
    timer_begin(PA_KC_SPLITKV, stream);
    kern<<<grid, C::NTHR, C::SMEM, stream>>>(tk, tv, sp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "split-KV launch: %s", cudaGetErrorString(e));
        return PA_ERR_CUDA;
    }
    timer_end(PA_KC_SPLITKV, stream);
    count_launches(1);
    if (plan.max_splits > 1) {
        dim3 g2(((plan.tile_rows + kCombineRows - 1) / kCombineRows) * ((sp.D + 63) / 64), sp.Hkv * plan.row_tiles,
                sp.batch);
        timer_begin(PA_KC_COMBINE, stream);
        e = launch_combine<T, C::M, NT>(g2, sp, stream);
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "split-KV combine launch: %s", cudaGetErrorString(e));
            return PA_ERR_CUDA;
        }
        timer_end(PA_KC_COMBINE, stream);
        count_launches(1);
    }
    return PA_OK;
}

template <int DP>
struct DecShape;  // pipeline depth of the warp-sliced decode kernel per padded head dim
template <>
struct DecShape<64> {
    static constexpr int STAGES = 4;
};
template <>
struct DecShape<128> {
    static constexpr int STAGES = 3;
};
template <>
struct DecShape<256> {
    static constexpr int STAGES = 3;
};

// Work list of the persistent decode mode, one CTA and one sequence per thread: work[0] =
// the take counter (zeroed here), work[1] = the number of (sequence, split) items, then
// the items, sequences longest first (by key tiles, ties by index) with each sequence's
// splits in order.  A sequence's split count comes from the tile view the kernels use; a
// sequence whose rows attend no key still gets one item (its rows are written as zeros),
// one the prefill kernel owns or with no queries gets none.
template <int M, int NT>
__global__ void __launch_bounds__(kMaxOrderBatch) work_list_kernel(const SplitParams p, int* work) {
    __shared__ int s_tiles[kMaxOrderBatch];
    __shared__ int s_splits[kMaxOrderBatch];
    __shared__ int s_at[kMaxOrderBatch];
    __shared__ int s_warp[kMaxOrderBatch / 32];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    int nt = 0, ns = 0;
    if (t < p.batch) {
        TileView tv;
        if (tile_view<M, NT>(p, t, 0, tv, true, true)) {
            nt = tv.ntiles;
            ns = max(tv.nsplit, 1);
        }
        s_tiles[t] = nt;
        s_splits[t] = ns;
    }
    __syncthreads();
    if (t < p.batch) {
        int rank = 0;
        for (int u = 0; u < p.batch; ++u) {
            const int lu = s_tiles[u];
            rank += (lu > nt) || (lu == nt && u < t);
        }
        s_at[rank] = t;
    }
    __syncthreads();
    const int seq = t < p.batch ? s_at[t] : 0;
    const int v = t < p.batch ? s_splits[seq] : 0;  // items of the sequence of rank t
    int x = v;                                      // inclusive scan over the ranks
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = s_warp[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += y;
        }
        s_warp[lane] = w;
    }
    __syncthreads();
    const int first = x - v + (warp > 0 ? s_warp[warp - 1] : 0);
    for (int k = 0; k < v; ++k) {
        work[2 + 2 * (first + k)] = seq;
        work[3 + 2 * (first + k)] = k;
    }
    if (t == 0) {
        work[0] = 0;
        work[1] = s_warp[kMaxOrderBatch / 32 - 1];
    }
}

template <typename T, int DP, int MG>
static int run_decode(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& sp, const SplitPlan& plan,
                      cudaStream_t stream, char* msg, size_t msg_len) {
    constexpr int NT = 64, STAGES = DecShape<DP>::STAGES;
    using C = DecCfg<DP, MG, NT, STAGES>;
    auto kern = decode_kernel<T, DP, MG, NT, STAGES>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "cudaFuncSetAttribute(decode, %d bytes): %s", C::SMEM, cudaGetErrorString(e));
            return PA_ERR_CUDA;
        }
        configured = true;
    }
    if (sp.order) {
        const int rc = launch_longest_first(sp.cu_k, sp.batch, const_cast<int*>(sp.order), stream, msg, msg_len);
        if (rc != PA_OK) return rc;
    }
    if (sp.work) {
        if (sp.batch < 1 || sp.batch > kMaxOrderBatch || plan.slots < 1) {
            snprintf(msg, msg_len, "decode work list: batch %d, %d CTAs", sp.batch, plan.slots);
            return PA_ERR_UNSUPPORTED;
        }
        NvtxRange nvw("pa::work_list_kernel");
        work_list_kernel<C::M, NT><<<1, kMaxOrderBatch, 0, stream>>>(sp, sp.work);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "decode work list launch: %s", cudaGetErrorString(e));
            return PA_ERR_CUDA;
        }
        count_launches(1);
    }
    // persistent mode: one CTA per resident slot; otherwise (split, kv head, sequence rank)
    const dim3 grid = sp.work ? dim3(plan.slots, 1, 1) : dim3(plan.max_splits, sp.Hkv, sp.batch);
    NvtxRange nv("pa::decode_kernel");
    timer_begin(PA_KC_SPLITKV, stream);
    kern<<<grid, kDecodeThreads, C::SMEM, stream>>>(tk, tv, sp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "decode launch: %s", cudaGetErrorString(e));
        return PA_ERR_CUDA;
    }
    timer_end(PA_KC_SPLITKV, stream);
    count_launches(1);
    if (plan.max_splits > 1) {
        dim3 g2(((plan.tile_rows + kCombineRows - 1) / kCombineRows) * ((sp.D + 63) / 64), sp.Hkv, sp.batch);
        timer_begin(PA_KC_COMBINE, stream);
        e = launch_combine<T, C::M, NT>(g2, sp, stream);
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "decode combine launch: %s", cudaGetErrorString(e));
            return PA_ERR_CUDA;
        }
        timer_end(PA_KC_COMBINE, stream);
        count_launches(1);
    }
    return PA_OK;
}

// Head dim 257..512, at most 32 rows: the quarter-column decode kernel (32-key tiles, one
// 32-row box per tile; pages are multiples of 32).
constexpr int kWideStages = 3;

template <typename T, int MG>
static int run_decode512(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& sp, const SplitPlan& plan,
                         cudaStream_t stream, char* msg, size_t msg_len) {
    using C = WideCfg<MG, kWideStages>;
    auto kern = decode512_kernel<T, MG, kWideStages>;
    if (sp.box_rows != C::NT || sp.boxes_per_tile != 1) {
        snprintf(msg, msg_len, "decode512: box of %d rows, %d a tile (expected one of %d)", sp.box_rows,
                 sp.boxes_per_tile, C::NT);
        return PA_ERR_UNSUPPORTED;
    }
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "cudaFuncSetAttribute(decode512, %d bytes): %s", C::SMEM, cudaGetErrorString(e));
            return PA_ERR_CUDA;
        }
        configured = true;
    }
    if (sp.order) {
        const int rc = launch_longest_first(sp.cu_k, sp.batch, const_cast<int*>(sp.order), stream, msg, msg_len);
        if (rc != PA_OK) return rc;
    }
    dim3 grid(plan.max_splits, sp.Hkv, sp.batch);
    NvtxRange nv("pa::decode512_kernel");
    timer_begin(PA_KC_SPLITKV, stream);
    kern<<<grid, C::THREADS, C::SMEM, stream>>>(tk, tv, sp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "decode512 launch: %s", cudaGetErrorString(e));
        return PA_ERR_CUDA;
    }
    timer_end(PA_KC_SPLITKV, stream);
    count_launches(1);
    if (plan.max_splits > 1) {
        dim3 g2(((plan.tile_rows + kCombineRows - 1) / kCombineRows) * ((sp.D + 63) / 64), sp.Hkv, sp.batch);
        timer_begin(PA_KC_COMBINE, stream);
        e = launch_combine<T, C::M, C::NT>(g2, sp, stream);
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "decode512 combine launch: %s", cudaGetErrorString(e));
            return PA_ERR_CUDA;
        }
        timer_end(PA_KC_COMBINE, stream);
        count_launches(1);
    }
    return PA_OK;
}

// Resident CTAs per SM of the kernel a plan dispatches to (occupancy API, once per
// instantiation), for sizing the split count to whole waves.
template <typename KernelT>
static int resident_ctas(KernelT kern, int threads, int smem) {
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 1;
    }
    return n > 0 ? n : 1;
}

static_assert(kRankInCta <= kDecodeThreads, "in-CTA ranking: one sequence per thread");

template <typename T, int DP, int MG>
static int decode_occupancy() {
    constexpr int NT = 64, STAGES = DecShape<DP>::STAGES;
    static const int n =
        resident_ctas(decode_kernel<T, DP, MG, NT, STAGES>, kDecodeThreads, DecCfg<DP, MG, NT, STAGES>::SMEM);
    return n;
}

template <typename T, int MG>
static int decode512_occupancy() {
    using C = WideCfg<MG, kWideStages>;
    static const int n = resident_ctas(decode512_kernel<T, MG, kWideStages>, C::THREADS, C::SMEM);
    return n;
}

template <typename T, int DP, int MT>
static int generic_occupancy() {
    constexpr int NT = SplitShape<DP>::NT, STAGES = SplitShape<DP>::STAGES, NW = SplitShape<DP>::NW;
    using C = SplitCfg<DP, MT, NT, STAGES, NW>;
    static const int n = resident_ctas(splitkv_kernel<T, DP, MT, NT, STAGES, NW>, C::NTHR, C::SMEM);
    return n;
}

template <typename T>
static int splitkv_occupancy_t(const SplitPlan& plan) {
    static const bool force_generic = std::getenv("PA_FORCE_GENERIC") != nullptr;
    if (plan.row_tiles == 1 && plan.dp == 512 && !force_generic)  // the same choice as launch_splitkv_t
        return plan.mt == 1 ? decode512_occupancy<T, 1>() : decode512_occupancy<T, 2>();
    if (plan.row_tiles == 1 && plan.dp <= 256 && !force_generic) {
        if (plan.dp == 64) return plan.mt == 1 ? decode_occupancy<T, 64, 1>() : decode_occupancy<T, 64, 2>();
        if (plan.dp == 128) return plan.mt == 1 ? decode_occupancy<T, 128, 1>() : decode_occupancy<T, 128, 2>();
        return plan.mt == 1 ? decode_occupancy<T, 256, 1>() : decode_occupancy<T, 256, 2>();
    }
    switch (plan.dp * 4 + plan.mt) {
        case 64 * 4 + 1: return generic_occupancy<T, 64, 1>();
        case 64 * 4 + 2: return generic_occupancy<T, 64, 2>();
        case 128 * 4 + 1: return generic_occupancy<T, 128, 1>();
        case 128 * 4 + 2: return generic_occupancy<T, 128, 2>();
        case 256 * 4 + 1: return generic_occupancy<T, 256, 1>();
        case 256 * 4 + 2: return generic_occupancy<T, 256, 2>();
        case 512 * 4 + 1: return generic_occupancy<T, 512, 1>();
        default: return generic_occupancy<T, 512, 2>();
    }
}

template <typename T>
static int launch_splitkv_t(const Args& a, const SplitPlan& plan, void* workspace, unsigned int* err, char* msg,
                            size_t msg_len) {
    const int NT = plan.nt;
    // Box rows: the largest of {NT, 64, 32} that divides the page, so that a box never
    // straddles two pages (page sizes are multiples of 32).
    int box_rows = NT;
    if (a.paged)
        box_rows = (a.page % NT) == 0 ? NT : (NT > 64 && a.page % 64 == 0) ? 64 : 32;
    CUtensorMap tk, tv;
    uint64_t dims[4];
    uint64_t strides[3];
    if (a.paged) {
        dims[0] = (uint64_t)a.D;
        dims[1] = (uint64_t)a.Hkv;
        dims[2] = (uint64_t)a.page;
        dims[3] = (uint64_t)a.num_blocks;
        strides[0] = (uint64_t)a.kv_s2 * 2;
        strides[1] = (uint64_t)a.kv_s1 * 2;
        strides[2] = (uint64_t)a.kv_s0 * 2;
    } else {
        dims[0] = (uint64_t)a.D;
        dims[1] = (uint64_t)a.Hkv;
        dims[2] = (uint64_t)(a.num_blocks > 0 ? a.num_blocks : 1);
        dims[3] = 1;
        strides[0] = (uint64_t)a.kv_s2 * 2;
        strides[1] = (uint64_t)a.kv_s0 * 2;
        strides[2] = (uint64_t)a.kv_s0 * 2 * dims[2];
    }
    const uint32_t box[4] = {64u, 1u, (uint32_t)box_rows, 1u};
    int rc = encode_tmap_4d(&tk, a.dtype, a.k, dims, strides, box, 1, msg, msg_len);
    if (rc != PA_OK) return rc;
    rc = encode_tmap_4d(&tv, a.dtype, a.v, dims, strides, box, 1, msg, msg_len);
    if (rc != PA_OK) return rc;

    SplitParams sp{};
    sp.q = a.q;
    sp.q_s0 = a.q_s0;
    sp.q_s1 = a.q_s1;
    sp.out = a.out;
    sp.o_s0 = a.o_s0;
    sp.o_s1 = a.o_s1;
    sp.lse = a.lse;
    sp.lse_s0 = a.lse_s0;
    sp.lse_sb = a.lse_sb;
    sp.cu_q = a.cu_q;
    sp.cu_k = a.cu_k;
    sp.bt = a.block_table;
    sp.bt_s0 = a.bt_s0;
    sp.bt_cols = a.bt_cols;
    sp.batch = a.batch;
    sp.H = a.H;
    sp.Hkv = a.Hkv;
    sp.G = a.H / a.Hkv;
    sp.D = a.D;
    sp.P = a.paged ? a.page : 1;
    sp.num_blocks = a.num_blocks;
    sp.total_q = a.total_q;
    sp.paged = a.paged ? 1 : 0;
    sp.box_rows = box_rows;
    sp.boxes_per_tile = NT / box_rows;
    sp.max_sq = a.max_sq;
    sp.max_sk = a.max_sk;
    sp.scale_log2 = a.scale * 1.4426950408889634f;
    sp.alibi = a.alibi;
    sp.wl = a.wl;
    sp.wr = a.wr;
    sp.rows_cap = plan.rows_cap;
    sp.row_tiles = plan.row_tiles;
    sp.split_tiles = plan.split_tiles;
    sp.max_splits = plan.max_splits;
    sp.part_stride = a.total_q * a.H;
    if (plan.order_bytes) sp.order = static_cast<const int*>(workspace);
    if (plan.work_bytes) sp.work = reinterpret_cast<int*>(static_cast<char*>(workspace) + plan.order_bytes);
    sp.rank_in_cta = plan.rank_in_cta;
    if (plan.max_splits > 1) {
        sp.part_o = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.order_bytes + plan.work_bytes);
        sp.part_lse = sp.part_o + (size_t)plan.max_splits * sp.part_stride * a.D;
    }
    sp.err = err;
    sp.wait_ns = a.wait_ns;
    sp.withhold = a.withhold_loads;

    if (plan.tc) {  // decode class on the tensor cores
        if (plan.max_splits > 1) {
            const int rc = launch_decode_tc(tk, tv, sp, plan, a.dtype, a.stream, msg, msg_len);
            if (rc != PA_OK) return rc;
            const int M = 16 * plan.mt;
            dim3 g2(((plan.tile_rows + kCombineRows - 1) / kCombineRows) * ((sp.D + 63) / 64), sp.Hkv, sp.batch);
            timer_begin(PA_KC_COMBINE, a.stream);
            const cudaError_t e = M == 16 ? launch_combine<T, 16, 128>(g2, sp, a.stream)
                                          : launch_combine<T, 32, 128>(g2, sp, a.stream);
            if (e != cudaSuccess) {
                snprintf(msg, msg_len, "decode_tc combine launch: %s", cudaGetErrorString(e));
                return PA_ERR_CUDA;
            }
            timer_end(PA_KC_COMBINE, a.stream);
            count_launches(1);
            return PA_OK;
        }
        return launch_decode_tc(tk, tv, sp, plan, a.dtype, a.stream, msg, msg_len);
    }
    // decode class (one row tile of at most 32 rows): warp-sliced kernel up to head dim 256,
    // quarter-column kernel above
    static const bool force_generic = std::getenv("PA_FORCE_GENERIC") != nullptr;
    if (plan.row_tiles == 1 && plan.dp == 512 && !force_generic)
        return plan.mt == 1 ? run_decode512<T, 1>(tk, tv, sp, plan, a.stream, msg, msg_len)
                            : run_decode512<T, 2>(tk, tv, sp, plan, a.stream, msg, msg_len);
    if (plan.row_tiles == 1 && plan.dp <= 256 && !force_generic) {
        if (plan.dp == 64) return plan.mt == 1 ? run_decode<T, 64, 1>(tk, tv, sp, plan, a.stream, msg, msg_len)
                                               : run_decode<T, 64, 2>(tk, tv, sp, plan, a.stream, msg, msg_len);
        if (plan.dp == 128) return plan.mt == 1 ? run_decode<T, 128, 1>(tk, tv, sp, plan, a.stream, msg, msg_len)
                                                : run_decode<T, 128, 2>(tk, tv, sp, plan, a.stream, msg, msg_len);
        return plan.mt == 1 ? run_decode<T, 256, 1>(tk, tv, sp, plan, a.stream, msg, msg_len)
                            : run_decode<T, 256, 2>(tk, tv, sp, plan, a.stream, msg, msg_len);
    }

#define PA_SPLIT_CASE(DPV, MTV)                                                        \
    if (plan.dp == DPV && plan.mt == MTV)                                              \
        return run_splitkv<T, DPV, MTV>(tk, tv, sp, plan, a.stream, msg, msg_len);
    PA_SPLIT_CASE(64, 1)
    PA_SPLIT_CASE(64, 2)
    PA_SPLIT_CASE(128, 1)
    PA_SPLIT_CASE(128, 2)
    PA_SPLIT_CASE(256, 1)
    PA_SPLIT_CASE(256, 2)
    PA_SPLIT_CASE(512, 1)
    PA_SPLIT_CASE(512, 2)
#undef PA_SPLIT_CASE
    snprintf(msg, msg_len, "no split-KV kernel for head_dim tile %d, row groups %d", plan.dp, plan.mt);
    return PA_ERR_UNSUPPORTED;
}

}  // namespace pa
