// Split-KV paged attention kernel (decode class: few query rows per kv head) and
// the log-sum-exp combine of its partial results.
//
// One CTA owns one (sequence b, kv head hk, row tile, key split).  The rows of a
// tile are the (query i, head g) pairs of the GQA group of hk, ordered i * G + g, so
// every K/V byte a CTA reads serves all G query heads that share it.  K and V pages
// are pulled into shared memory with TMA tiled loads addressed through the block
// table (the paged layout of "flash-attn-varlen paged expects k/v tensors of rank 4",
// What it means: (num_blocks, page_block_size, num_heads_k, head_dim), last dim
// contiguous), in a multi-stage mbarrier pipeline.  Q.K^T and P.V run on the tensor
// cores (mma.sync m16n8k16, fp32 accumulate); the online softmax runs in fp32.
//
// Masking is bottom-right aligned: query i of a sequence with sq queries and sk keys
// attends key j iff 0 <= j < sk, j >= i + sk - sq - window_left (window_left >= 0)
// and j <= i + sk - sq + window_right (window_right >= 0).
#pragma once

#include <math.h>

#include "device_common.cuh"

namespace pa {

struct SplitParams {
    const void* q;
    int64_t q_s0, q_s1;
    void* out;
    int64_t o_s0, o_s1;
    float* lse;
    int64_t lse_s0, lse_sb;  // lse of (head h, token t, sequence b) at h lse_s0 + t + b lse_sb
    const int32_t* cu_q;
    const int32_t* cu_k;
    const int32_t* bt;
    int64_t bt_s0;
    int bt_cols;
    int batch, H, Hkv, G, D, P;
    int64_t num_blocks;
    int64_t total_q;
    int paged;
    int boxes_per_tile, box_rows;
    int max_sq, max_sk;
    float scale_log2;
    int wl, wr;
    const float* alibi;  // per-query-head slopes of the linear position bias, or nullptr
    const int* order;    // decode kernel: sequence of grid z index (longest first), or nullptr
    int* work;           // decode kernel, persistent mode: [take counter, item count, (sequence, split)...]
    int rank_in_cta;     // decode kernel: each CTA ranks the (<= kDecodeThreads) sequences itself
    int rows_cap, row_tiles, split_tiles, max_splits;
    float* part_o;
    float* part_lse;
    int64_t part_stride;  // rows per split slab (total_q * H)
    unsigned int* err;
    uint64_t wait_ns;    // bound on every wait
    int withhold;        // test hook: issue no loads
};

// The work of one (sequence, kv head, row tile), computed identically by the split
// kernel and the combine kernel.
struct TileView {
    int q0, sq, sk;
    int row0, rows;   // first row (i * G + g) and row count of the tile
    int lo, hi;       // inclusive key interval touched by the tile's rows (hi < lo: none)
    int kt0;          // first key tile start (multiple of the tile width)
    int ntiles, nsplit;
};

// Metadata out of range is flagged in the error word when `report` holds, by thread 0 of
// the CTA or, with `any_thread`, by the calling thread.
template <int M, int NT>
__device__ __forceinline__ bool tile_view(const SplitParams& p, int b, int rt, TileView& v, bool report,
                                          bool any_thread = false) {
    const int q0 = p.cu_q[b], q1 = p.cu_q[b + 1];
    const int k0 = p.cu_k[b], k1 = p.cu_k[b + 1];
    const int sq = q1 - q0, sk = k1 - k0;
    const bool bad = sq < 0 || sk < 0 || sq > p.max_sq || sk > p.max_sk || q0 < 0 || q1 > p.total_q ||
                     (!p.paged && (k0 < 0 || k1 > p.num_blocks));
    if (bad) {
        if (report && (any_thread || threadIdx.x == 0)) flag_error(p.err, PA_ERR_DEVICE_BOUNDS);
        return false;
    }
    if (sq == 0) return false;
    const int64_t rows_total = (int64_t)sq * p.G;
    if (rows_total > p.rows_cap) return false;  // owned by the tensor-core prefill kernel
    v.row0 = rt * M;
    if (v.row0 >= rows_total) return false;
    v.rows = (int)min64(M, rows_total - v.row0);
    v.q0 = q0;
    v.sq = sq;
    v.sk = sk;
    const int64_t i_lo = v.row0 / p.G, i_hi = (v.row0 + v.rows - 1) / p.G;
    const int64_t c = (int64_t)sk - sq;
    const int64_t lo = p.wl >= 0 ? max64(0, i_lo + c - p.wl) : 0;
    const int64_t hi = p.wr >= 0 ? min64(sk - 1, i_hi + c + p.wr) : (int64_t)sk - 1;
    v.lo = (int)lo;
    v.hi = (int)max64(hi, -1);
    if (hi < lo) {
        v.kt0 = 0;
        v.ntiles = 0;
        v.nsplit = 0;
    } else {
        v.kt0 = v.lo & ~(NT - 1);
        v.ntiles = (v.hi - v.kt0) / NT + 1;
        v.nsplit = (v.ntiles + p.split_tiles - 1) / p.split_tiles;
    }
    if (v.nsplit > p.max_splits) {  // a sequence longer than max_seqlen_k promised
        if (report && (any_thread || threadIdx.x == 0)) flag_error(p.err, PA_ERR_DEVICE_BOUNDS);
        v.nsplit = p.max_splits;
        v.ntiles = min(v.ntiles, p.max_splits * p.split_tiles);
    }
    return true;
}

// At a CTA's entry, before its sequence's lengths are known: lane `lane` of a warp hints the
// `lane`-th 128-byte line of the block-table entries of split `split` into L2, taking the
// sequence's keys to start at tile 0 (no left window), so that the producer's lookups after
// tile_view find them there instead of in HBM.  Every address stays inside row b of the
// table whatever the lengths turn out to be.
template <int NT>
__device__ __forceinline__ void prefetch_split_pages(const SplitParams& p, int b, int split, int lane) {
    if (!p.paged || b < 0 || b >= p.batch || p.bt_cols <= 0) return;
    const int64_t first = (int64_t)split * p.split_tiles * NT / p.P;
    const int64_t last = min64(((int64_t)(split + 1) * p.split_tiles * NT - 1) / p.P, (int64_t)p.bt_cols - 1);
    const int64_t page = first + 32 * (int64_t)lane;
    if (page <= last) prefetch_l2(p.bt + (int64_t)b * p.bt_s0 + page);
}

// NW warps: 4, each taking a quarter of the tile's keys in Q.K^T over the whole head dim;
// or 8 for the widest heads, each taking every key of the tile over one eighth of the head
// dim (4 k-steps: eight independent accumulator chains of 4 MMAs instead of two chains of
// 16, measured latency-bound), the softmax summing the 8 partial scores.  In P.V each warp
// owns DP / NW output columns.
template <int DP, int MT, int NT, int STAGES, int NW = 4>
struct SplitCfg {
    static constexpr int NTHR = NW * 32;
    static constexpr int KSLICES = NW == 8 ? 1 : 4;  // key slices of Q.K^T
    static constexpr int KSPLIT = NW / KSLICES;      // head-dim parts of Q.K^T
    static constexpr int M = 16 * MT;               // query rows per CTA
    static constexpr int CH = DP / 64;              // 64-element (128-byte) column chunks of a row
    static constexpr int TILE_BYTES = CH * NT * 128;  // one K (or V) tile of NT keys
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int Q_BYTES = CH * M * 128;
    static constexpr int P_BYTES = M * 128;         // P rows padded to 128 bytes
    static constexpr int S_STRIDE = NT + 4;         // fp32 score row stride
    static constexpr int S_BYTES = KSPLIT * M * S_STRIDE * 4;  // one partial score buffer per part
    static constexpr int OFF_Q = STAGES * STAGE_BYTES;
    static constexpr int OFF_P = OFF_Q + Q_BYTES;
    static constexpr int OFF_S = OFF_P + P_BYTES;
    // row_lo[M], row_hi[M], alpha[M], m[M], l[M], row_dg[M], row_ab[M]
    static constexpr int OFF_ROW = OFF_S + S_BYTES;
    static constexpr int OFF_BAR = (OFF_ROW + 7 * M * 4 + 15) & ~15;
    static constexpr int SMEM = OFF_BAR + STAGES * 8 + 1024;  // + slack for 1024-byte alignment
    static constexpr int KW = NT / KSLICES;         // keys per warp in Q.K^T
    static constexpr int DW = DP / NW;              // output columns per warp in P.V
    static_assert(NW == 4 || NW == 8, "warps");
    static_assert(NT == 64 || NT == 32, "tile width");
    static_assert(DW % 16 == 0, "P.V column slice");
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

template <typename T, int DP, int MT, int NT, int STAGES, int NW>
__global__ void __launch_bounds__(NW * 32) splitkv_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                      const __grid_constant__ CUtensorMap tm_v,
                                                      const SplitParams p) {
    using C = SplitCfg<DP, MT, NT, STAGES, NW>;
    constexpr int M = C::M;
    constexpr int RPW = M / NW;  // softmax rows owned by each warp
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    allow_dependent_launch();
    const int b = blockIdx.z, hk = blockIdx.y % p.Hkv, rt = blockIdx.y / p.Hkv, split = blockIdx.x;

    TileView tv;
    if (!tile_view<M, NT>(p, b, rt, tv, split == 0)) return;
    if (split >= max(tv.nsplit, 1)) return;
    const bool single = tv.nsplit <= 1;
    const int t_begin = split * p.split_tiles;
    const int n_iter = max(0, min(tv.ntiles, t_begin + p.split_tiles) - t_begin);

    int* row_lo = reinterpret_cast<int*>(smem + C::OFF_ROW);
    int* row_hi = row_lo + M;
    float* alpha_sm = reinterpret_cast<float*>(row_hi + M);
    float* m_sm = alpha_sm + M;
    float* l_sm = m_sm + M;
    int* row_dg = reinterpret_cast<int*>(l_sm + M);
    float* row_ab = reinterpret_cast<float*>(row_dg + M);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    float* S = reinterpret_cast<float*>(smem + C::OFF_S);
    uint8_t* Ps = smem + C::OFF_P;

    if (tid < M) {
        int lo = 0, hi = -1, dg = 0;  // padding rows attend nothing
        float ab = 0.f;
        if (tid < tv.rows) {
            const int64_t i = (tv.row0 + tid) / p.G;
            const int64_t diag = i + tv.sk - tv.sq;
            lo = p.wl >= 0 ? (int)max64(0, diag - p.wl) : 0;
            hi = p.wr >= 0 ? (int)max64(-1, min64(tv.sk - 1, diag + p.wr)) : tv.sk - 1;
            dg = (int)diag;
            if (p.alibi) ab = p.alibi[hk * p.G + (int)(tv.row0 + tid - i * p.G)] * kLog2e;
        }
        row_lo[tid] = lo;
        row_hi[tid] = hi;
        row_dg[tid] = dg;
        row_ab[tid] = ab;
    }
    if (tid == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], NW);  // one arrival per warp
        fence_mbar_init();
    }
    // Q rows of the tile -> shared memory (128-byte swizzled rows, zero padded).
    {
        const T* q = static_cast<const T*>(p.q);
        constexpr int UNITS = DP / 8;
        uint8_t* qs = smem + C::OFF_Q;
        for (int idx = tid; idx < M * UNITS; idx += C::NTHR) {
            const int r = idx / UNITS, u = idx - r * UNITS;
            int4 val = make_int4(0, 0, 0, 0);
            if (r < tv.rows && u * 8 < p.D) {
                const int rho = tv.row0 + r;
                const int i = rho / p.G, g = rho - i * p.G;
                const T* src = q + (int64_t)(tv.q0 + i) * p.q_s0 + (int64_t)(hk * p.G + g) * p.q_s1 + u * 8;
                val = __ldg(reinterpret_cast<const int4*>(src));
            }
            *reinterpret_cast<int4*>(qs + (u >> 3) * (M * 128) + swz128(r, u & 7)) = val;
        }
    }
    __syncthreads();

    const uint64_t policy = l2_policy_evict_first();
    // Producers (lane 0 of every warp): pull the K/V boxes of key tile `it` of this split into
    // its stage, warp w taking the 64-column chunks c = w, w + NW, ...  One thread issuing all
    // of a stage's copies (16 at head_dim 512) held its warp, and with it the next barrier,
    // for thousands of cycles; each warp posts the bytes of its own copies before issuing them.
    auto issue = [&](int it) {
        const int stage = it % STAGES;
        const int kt = tv.kt0 + (t_begin + it) * NT;
        uint8_t* kst = smem + stage * C::STAGE_BYTES;
        uint8_t* vst = kst + C::TILE_BYTES;
        int cs[2], cb[2];
        bool live[2] = {false, false};
        uint32_t bytes = 0;
        for (int j = 0; j < p.boxes_per_tile; ++j) {
            const int key = kt + j * p.box_rows;
            if (key >= tv.sk) break;  // past the sequence: not loaded, V rows are zeroed
            if (p.paged) {
                const int page = key / p.P;
                if (page >= p.bt_cols) {
                    flag_error(p.err, PA_ERR_DEVICE_BOUNDS);
                    break;
                }
                const int blk = __ldg(p.bt + (int64_t)b * p.bt_s0 + page);
                if (blk < 0 || blk >= p.num_blocks) {
                    flag_error(p.err, PA_ERR_DEVICE_BOUNDS);
                    continue;
                }
                cs[j] = key - page * p.P;
                cb[j] = blk;
            } else {
                cs[j] = p.cu_k[b] + key;
                cb[j] = 0;
            }
            live[j] = true;
            bytes += 2u * ((C::CH - warp + NW - 1) / NW) * p.box_rows * 128u;
        }
        mbar_arrive_expect_tx(&full[stage], bytes);
        for (int j = 0; j < p.boxes_per_tile; ++j) {
            if (!live[j]) continue;
            for (int c = warp; c < C::CH; c += NW) {
                const int off = (c * NT + j * p.box_rows) * 128;
                tma_load_4d(kst + off, &tm_k, &full[stage], c * 64, hk, cs[j], cb[j], policy);
                tma_load_4d(vst + off, &tm_v, &full[stage], c * 64, hk, cs[j], cb[j], policy);
            }
        }
    };
    if (lane == 0 && !p.withhold) {
        for (int it = 0; it < min(STAGES - 1, n_iter); ++it) issue(it);
    }

    float o_acc[MT][C::DW / 8][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int n = 0; n < C::DW / 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) o_acc[mt][n][e] = 0.f;
    float m_run[RPW], l_run[RPW];
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
        m_run[k] = -INFINITY;
        l_run[k] = 0.f;
    }

    const uint32_t q_base = smem_addr(smem + C::OFF_Q);
    const uint32_t p_base = smem_addr(Ps);
    const int mi = lane >> 3, rr = lane & 7;

    for (int it = 0; it < n_iter; ++it) {
        const int stage = it % STAGES;
        const int kt = tv.kt0 + (t_begin + it) * NT;
        uint8_t* kst = smem + stage * C::STAGE_BYTES;
        uint8_t* vst = kst + C::TILE_BYTES;
        const bool ok = mbar_wait(&full[stage], (it / STAGES) & 1, p.wait_ns);

        // V rows at or past sk (tail of the last page, or pages not loaded) -> 0, so that
        // P = 0 never meets NaN or stale values in P.V.
        const int valid_rows = min(NT, tv.sk - kt);
        if (valid_rows < NT) {
            const int zr = NT - valid_rows;
            for (int idx = tid; idx < C::CH * zr * 8; idx += C::NTHR) {
                const int c = idx / (zr * 8), rem = idx - c * zr * 8;
                *reinterpret_cast<int4*>(vst + (c * NT + valid_rows + (rem >> 3)) * 128 + ((rem & 7) << 4)) =
                    make_int4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();  // this stage is rewritten by TMA later
        }

        // S = Q K^T for keys [ws*KW, ws*KW + KW) of the tile, over head-dim part kp
        const int ws = warp % C::KSLICES, kp = warp / C::KSLICES;
        float s_acc[MT][C::KW / 8][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int n = 0; n < C::KW / 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) s_acc[mt][n][e] = 0.f;
        const uint32_t k_base = smem_addr(kst);
#pragma unroll
        for (int kq = 0; kq < DP / 16 / C::KSPLIT; ++kq) {
            const int ks = kp * (DP / 16 / C::KSPLIT) + kq;
            const int c = ks >> 2, u0 = (ks & 3) * 2;
            uint32_t bf[C::KW / 8][2];
            if constexpr (C::KW >= 16) {
#pragma unroll
                for (int np = 0; np < C::KW / 16; ++np) {
                    const int key = ws * C::KW + np * 16 + rr + ((mi >> 1) << 3);
                    ldsm_x4(k_base + c * NT * 128 + swz128(key, u0 + (mi & 1)), bf[2 * np][0], bf[2 * np][1],
                            bf[2 * np + 1][0], bf[2 * np + 1][1]);
                }
            } else {
                const int key = ws * 8 + rr;
                ldsm_x2(k_base + c * NT * 128 + swz128(key, u0 + (mi & 1)), bf[0][0], bf[0][1]);
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t af[4];
                const int row = mt * 16 + rr + ((mi & 1) << 3);
                ldsm_x4(q_base + c * M * 128 + swz128(row, u0 + (mi >> 1)), af[0], af[1], af[2], af[3]);
#pragma unroll
                for (int n = 0; n < C::KW / 8; ++n) MmaOp<T>::run(s_acc[mt][n], af, bf[n][0], bf[n][1]);
            }
        }
        // raw partial scores -> shared memory (part kp)
        float* Sp = S + kp * (M * C::S_STRIDE);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int n = 0; n < C::KW / 8; ++n)
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int r = mt * 16 + (lane >> 2) + h2 * 8;
                    const int col = ws * C::KW + n * 8 + (lane & 3) * 2;
                    *reinterpret_cast<float2*>(Sp + r * C::S_STRIDE + col) =
                        make_float2(s_acc[mt][n][h2 * 2], s_acc[mt][n][h2 * 2 + 1]);
                }
        if (__syncthreads_or(!ok)) {
            if (tid == 0) flag_error(p.err, PA_ERR_DEVICE_TIMEOUT);
            return;
        }
        // the stage used by the previous iteration is free: refill it
        if (lane == 0 && it + STAGES - 1 < n_iter && !p.withhold) {
            fence_proxy_async_smem();
            issue(it + STAGES - 1);
        }

        // online softmax: warp w owns rows w, w+NW, ...; the score is scaled into the log2
        // domain (plus the position bias) and masked by select (NaN-safe)
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            const int r = warp + NW * k;
            const int lo = row_lo[r], hi = row_hi[r], dg = row_dg[r];
            const float ab = row_ab[r];
            auto score = [&](int col) {
                float sv = S[r * C::S_STRIDE + col];
#pragma unroll
                for (int kp2 = 1; kp2 < C::KSPLIT; ++kp2) sv += S[(kp2 * M + r) * C::S_STRIDE + col];
                const int j = kt + col;
                return (j >= lo && j <= hi) ? biased_log2(sv, p.scale_log2, ab, dg, j) : -INFINITY;
            };
            const float v0 = score(lane);
            const float v1 = (NT == 64) ? score(lane + 32) : -INFINITY;
            float mx = fmaxf(v0, v1);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_new = fmaxf(m_run[k], mx);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float p0 = fast_exp2(v0 - m_use);
            const float p1 = fast_exp2(v1 - m_use);
            const float alpha = fast_exp2(m_run[k] - m_use);
            float sum = p0 + p1;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            l_run[k] = l_run[k] * alpha + sum;
            m_run[k] = m_new;
            T* prow = reinterpret_cast<T*>(Ps);
            prow[(swz128(r, lane >> 3) >> 1) + (lane & 7)] = static_cast<T>(p0);
            if (NT == 64) prow[(swz128(r, (lane + 32) >> 3) >> 1) + (lane & 7)] = static_cast<T>(p1);
            if (lane == 0) alpha_sm[r] = alpha;
        }
        __syncthreads();

        // O = alpha * O + P V for output columns [warp*DW, warp*DW + DW)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const float a0 = alpha_sm[mt * 16 + (lane >> 2)];
            const float a1 = alpha_sm[mt * 16 + (lane >> 2) + 8];
#pragma unroll
            for (int n = 0; n < C::DW / 8; ++n) {
                o_acc[mt][n][0] *= a0;
                o_acc[mt][n][1] *= a0;
                o_acc[mt][n][2] *= a1;
                o_acc[mt][n][3] *= a1;
            }
        }
        const uint32_t v_base = smem_addr(vst);
#pragma unroll
        for (int ks = 0; ks < NT / 16; ++ks) {
            uint32_t af[MT][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                const int row = mt * 16 + rr + ((mi & 1) << 3);
                ldsm_x4(p_base + swz128(row, ks * 2 + (mi >> 1)), af[mt][0], af[mt][1], af[mt][2], af[mt][3]);
            }
#pragma unroll
            for (int np = 0; np < C::DW / 16; ++np) {
                const int d0 = warp * C::DW + np * 16;
                const int key = ks * 16 + rr + ((mi & 1) << 3);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(v_base + (d0 >> 6) * NT * 128 + swz128(key, ((d0 & 63) >> 3) + (mi >> 1)), b0, b1, b2, b3);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    MmaOp<T>::run(o_acc[mt][2 * np], af[mt], b0, b1);
                    MmaOp<T>::run(o_acc[mt][2 * np + 1], af[mt], b2, b3);
                }
            }
        }
    }

    // epilogue: normalise by l and write the output (or this split's partial result)
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
        if (lane == 0) {
            m_sm[warp + NW * k] = m_run[k];
            l_sm[warp + NW * k] = l_run[k];
        }
    }
    __syncthreads();
    T* out = static_cast<T*>(p.out);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int r = mt * 16 + (lane >> 2) + h2 * 8;
            if (r >= tv.rows) continue;
            const int rho = tv.row0 + r;
            const int i = rho / p.G, g = rho - i * p.G;
            const int64_t t = tv.q0 + i;
            const int h = hk * p.G + g;
            const float l = l_sm[r];
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int n = 0; n < C::DW / 8; ++n) {
                const int d = warp * C::DW + n * 8 + (lane & 3) * 2;
                if (d >= p.D) continue;
                const float x0 = o_acc[mt][n][h2 * 2] * inv, x1 = o_acc[mt][n][h2 * 2 + 1] * inv;
                if (single) {
                    *reinterpret_cast<uint32_t*>(out + t * p.o_s0 + (int64_t)h * p.o_s1 + d) = pack2<T>(x0, x1);
                } else {
                    *reinterpret_cast<float2*>(p.part_o + ((int64_t)split * p.part_stride + t * p.H + h) * p.D + d) =
                        make_float2(x0, x1);
                }
            }
        }
    if (tid < tv.rows) {
        const int r = tid;
        const int rho = tv.row0 + r;
        const int i = rho / p.G, g = rho - i * p.G;
        const int64_t t = tv.q0 + i;
        const int h = hk * p.G + g;
        const float l = l_sm[r];
        const float lse = l > 0.f ? (m_sm[r] + log2f(l)) * 0.69314718055994531f : -INFINITY;
        if (single)
            p.lse[(int64_t)h * p.lse_s0 + t + (int64_t)b * p.lse_sb] = lse;
        else
            p.part_lse[(int64_t)split * p.part_stride + t * p.H + h] = lse;
    }
}

// Launch of the tensor-core decode kernel (decode_tc.cu) for a plan with plan.tc set.
int launch_decode_tc(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& sp, const SplitPlan& plan,
                     int dtype, cudaStream_t stream, char* msg, size_t msg_len);

// lse = ln sum_s exp(lse_s); out = sum_s exp(lse_s - lse) * O_s, for the tiles that
// were split.  Grid: (rows x 64-column chunks, kv head x row tile, sequence); one CTA per
// (output row, 64 columns), each lane accumulating a pair of columns (reads of the partials
// coalesce along the head dimension).
constexpr int kCombineRows = 1;          // output rows per CTA (grid.x = rows x 64-column chunks)
constexpr int kCombineMaxSplits = 1024;  // split weights kept in shared memory

// (A minimum of 8 CTAs an SM caps it at 64 registers; with the thread count alone ptxas
// chose 32 and issued the partial loads a few at a time.)
template <typename T, int M, int NT>
__global__ void __launch_bounds__(128, 8) combine_kernel(const SplitParams p) {
    // One CTA per (row, 64 output columns).  Its 128 threads load the row's split LSEs at
    // once and turn them into weights in shared memory; warp w then sums the partial rows
    // of splits w, w + 4, ... with all of its loads in flight together, and warp 0 adds the
    // four sums: three dependent memory round trips however many splits there are (<= 256).
    __shared__ float wsm[kCombineMaxSplits];
    __shared__ float red[2][4];
    __shared__ float2 part[4][32];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.z, hk = blockIdx.y % p.Hkv, rt = blockIdx.y / p.Hkv;
    const int n_chunks = (p.D + 63) / 64;
    const int chunk = blockIdx.x % n_chunks;
    TileView tv;  // from the sequence bounds alone, which the split kernel does not write
    if (!tile_view<M, NT>(p, b, rt, tv, false)) return;
    if (tv.nsplit <= 1) return;
    const int ns = min(tv.nsplit, kCombineMaxSplits);
    const int r = blockIdx.x / n_chunks;
    if (r >= tv.rows) return;
    T* out = static_cast<T*>(p.out);
    const int rho = tv.row0 + r;
    const int i = rho / p.G, g = rho - i * p.G;
    const int64_t t = tv.q0 + i;
    const int h = hk * p.G + g;
    const int64_t row = t * p.H + h;
    // launched as a programmatic dependent of the split kernel (its launch and the lines
    // above overlap that kernel's tail): the partial results are read only after it completed
    asm volatile("griddepcontrol.wait;" ::: "memory");

    float mx = -INFINITY;
    for (int s = tid; s < ns; s += 128) {
        const float l = p.part_lse[(int64_t)s * p.part_stride + row];
        wsm[s] = l;
        mx = fmaxf(mx, l);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red[0][warp] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(red[0][0], red[0][1]), fmaxf(red[0][2], red[0][3]));
    const float m_use = (mx == -INFINITY) ? 0.f : mx;
    float sum = 0.f;
    for (int s = tid; s < ns; s += 128) {
        const float e = fast_exp2((wsm[s] - m_use) * 1.4426950408889634f);
        wsm[s] = e;
        sum += e;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0) red[1][warp] = sum;
    __syncthreads();
    sum = (red[1][0] + red[1][1]) + (red[1][2] + red[1][3]);

    const int d = chunk * 64 + lane * 2;
    float x0 = 0.f, x1 = 0.f;
    if (d < p.D) {
        const float* po = p.part_o + row * p.D + d;
        const int64_t split_stride = p.part_stride * p.D;
        constexpr int U = 16;
        for (int s0 = warp; s0 < ns; s0 += 4 * U) {
            // indices past the last split re-read the last one (in bounds, unconditional, so
            // that every load is issued before the first is used) and weigh it 0
            float2 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                v[u] = __ldg(reinterpret_cast<const float2*>(po + (int64_t)min(s0 + 4 * u, ns - 1) * split_stride));
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int s = s0 + 4 * u;
                const float wgt = s < ns ? wsm[min(s, ns - 1)] : 0.f;
                x0 = fmaf(wgt, v[u].x, x0);
                x1 = fmaf(wgt, v[u].y, x1);
            }
        }
    }
    part[warp][lane] = make_float2(x0, x1);
    __syncthreads();
    if (warp == 0 && d < p.D) {
        const float inv = sum > 0.f ? 1.f / sum : 0.f;
        const float2 a = part[0][lane], c = part[1][lane], e = part[2][lane], f = part[3][lane];
        *reinterpret_cast<uint32_t*>(out + t * p.o_s0 + (int64_t)h * p.o_s1 + d) =
            pack2<T>(((a.x + c.x) + (e.x + f.x)) * inv, ((a.y + c.y) + (e.y + f.y)) * inv);
    }
    if (chunk == 0 && tid == 0)
        p.lse[(int64_t)h * p.lse_s0 + t + (int64_t)b * p.lse_sb] = sum > 0.f ? m_use + logf(sum) : -INFINITY;
}

}  // namespace pa
