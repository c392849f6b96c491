// Decode-class paged attention on the 5th-generation tensor cores (tcgen05), with the
// operands swapped so that the keys, not the few query rows, fill the 128-row MMA.
//
// One CTA owns one (sequence, kv head, key split) with at most 32 query rows: the (query
// i, head g) pairs of the kv head's GQA group, ordered i * G + g, so every K/V byte read
// serves all G query heads.  Per tile of 128 keys:
//   S^T = K Q^T      tcgen05.mma M = 128 keys, N = NR rows (16 or 32), K = head dim;
//                    A = K tile, B = Q, both K-major in shared memory; S^T in tensor memory
//                    (lane = key, column = row), double-buffered
//   softmax          four warps, one thread per key: mask, running row maxima (lazy: updated
//                    only when a row's maximum grows by more than 2^8, which is exact after
//                    the final division), P = exp2(S - m) written as P^T rows to shared memory
//   O^T += V^T P^T   tcgen05.mma M = 128 head-dim columns per chunk, N = NR rows, K = keys;
//                    A = V tile MN-major, B = P^T K-major; O^T in tensor memory
// Keys fill the MMA rows, so a decode row count of 4..32 wastes no tensor work, and the
// head dim only sets the number of 128-column chunks: head_dim 512 keeps S^T (2 x NR
// columns) and O^T (4 x NR columns) in 256 of the 512 tensor-memory columns.
//
// K and V arrive by TMA through the block table (the paged layout of "flash-attn-varlen
// paged expects k/v tensors of rank 4", What it means), page-aligned boxes of 64 head-dim
// columns, into two rings: K in 16 KB units (128 keys x 64 columns, one 16-deep slice of
// the Q.K^T reduction each), V in 32 KB units (128 keys x 128 columns, one O^T chunk each).
// Each ring has its own MMA-issuing warp, so the keys of the next tiles stream in while the
// softmax and P.V of the current tile run.  One thread issuing TMA copies of page-sized boxes
// sustains only ~13 B/clk (measured on GB300: the issue cost grows with the box's 128-byte
// rows), so two producer warps feed each ring, sharing its copies round robin; each posts the
// bytes of its own copies on the unit's barrier before issuing them.
//
// Roles (320 threads): warps 0..3 softmax and epilogue (warp w reaches tensor-memory lanes
// 32 w .. 32 w + 31), warp 4 S issuer (owns the tensor memory), warp 5 P.V issuer, warps 6, 7
// K producers, warps 8, 9 V producers.
//
// Mask (bottom-right aligned): query i of a sequence with sq queries and sk keys attends
// key j iff 0 <= j < sk, j >= i + sk - sq - window_left (window_left >= 0) and
// j <= i + sk - sq + window_right (window_right >= 0).
#include <cstdio>
#include <cstdlib>
#include <type_traits>

#include "splitkv_kernel.cuh"
#include "tc_common.cuh"

namespace pa {
namespace {

constexpr int kTcNT = 128;  // keys per tile
template <int NR>
struct TcRoles {
    static constexpr int PROD = 4;  // producer warps 6..9: two for the K ring, two for the V ring
    static constexpr int THREADS = (6 + PROD) * 32;
};

template <int DP, int NR, int KR, int VR>
struct TcCfg {
    static constexpr int CH = DP / 128;              // 128-column head-dim chunks (V units per tile)
    static constexpr int KH = DP / 64;               // 64-column halves (K units per tile)
    static constexpr int KUNIT = 128 * 128;          // 128 keys x 64 columns (16 KB)
    static constexpr int VUNIT = 2 * KUNIT;          // 128 keys x 128 columns (32 KB)
    static constexpr int Q_CHUNK = NR * 128;         // NR rows x 64 columns
    static constexpr int P_BUF = 2 * NR * 128;       // NR rows x 128 keys
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = KR * KUNIT;
    static constexpr int OFF_Q = OFF_V + VR * VUNIT;
    static constexpr int OFF_P = OFF_Q + KH * Q_CHUNK;
    static constexpr int OFF_ROW = OFF_P + 2 * P_BUF;     // lo, hi, dg (int), ab (float) per row
    static constexpr int OFF_RED = OFF_ROW + 4 * NR * 4;  // [4 warps][NR] floats, then 2 x 4 votes
    static constexpr int OFF_BAR = (OFF_RED + 4 * NR * 4 + 8 * 4 + 15) & ~15;
    // k_full[KR], k_empty[KR], v_full[VR], v_empty[VR], s_full[2], p_full[2], pv_done[2], drain[2]
    static constexpr int NBAR = 2 * KR + 2 * VR + 8;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem base, abort flag, rank pick
    static constexpr int OFF_IDS = OFF_MISC + 16;
    static constexpr int MAX_BOXES = 512;
    static constexpr int SMEM = OFF_IDS + MAX_BOXES * 4 + 1024;
    static constexpr uint32_t T_S = 0;       // S^T buffers: columns [0, NR), [NR, 2 NR)
    static constexpr uint32_t T_O = 2 * NR;  // O^T chunk c: columns [2 NR + c NR, ...)
    static constexpr uint32_t TMEM_COLS = (2 * NR + CH * NR) <= 32    ? 32
                                          : (2 * NR + CH * NR) <= 64  ? 64
                                          : (2 * NR + CH * NR) <= 128 ? 128
                                                                      : 256;
    static_assert(DP % 128 == 0 && NR % 16 == 0 && NR <= 32, "shape");
    static_assert(2 * NR + CH * NR <= 256, "tensor memory");
    static_assert(KR >= 2 && VR >= 2, "rings");
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                        unsigned int* err, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            *abort_flag = 1u;
            flag_error(err, PA_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
}

// Reduce-scatter of NR per-thread values over the warp: afterwards lane l holds the maximum
// (MAX) or sum over all 32 lanes of value (l mod NR).
template <int NR, bool MAX>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[NR], int lane) {
#pragma unroll
    for (int half = NR / 2; half >= 1; half >>= 1) {
        const bool upper = (lane & half) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            const float recv = __shfl_xor_sync(0xffffffffu, send, half);
            v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
        }
    }
    float r = v[0];
    if (NR == 16) {  // lanes l and l ^ 16 hold the two halves' partial results of one value
        const float o = __shfl_xor_sync(0xffffffffu, r, 16);
        r = MAX ? fmaxf(r, o) : r + o;
    }
    return r;
}

template <typename T, int DP, int NR, int KR, int VR>
__global__ void __launch_bounds__(TcRoles<NR>::THREADS, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const SplitParams p) {
    using C = TcCfg<DP, NR, KR, VR>;
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr int CH = C::CH, KH = C::KH;
    constexpr int kTcThreads = TcRoles<NR>::THREADS, kTcProd = TcRoles<NR>::PROD;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    allow_dependent_launch();

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* k_full = bars;
    uint64_t* k_empty = k_full + KR;
    uint64_t* v_full = k_empty + KR;
    uint64_t* v_empty = v_full + VR;
    uint64_t* s_full = v_empty + VR;  // [2]: S^T(j) complete, j % 2
    uint64_t* p_full = s_full + 2;    // [2]: the softmax warps have written P^T(j), j % 2
    uint64_t* pv_done = p_full + 2;   // [2]: P.V(j) complete, j % 2
    uint64_t* drain = pv_done + 2;    // [2]: every MMA of the S / P.V issuer complete
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile uint32_t* abort_flag = tmem_slot + 1;
    int* pick = reinterpret_cast<int*>(tmem_slot + 2);
    int* row_lo = reinterpret_cast<int*>(smem + C::OFF_ROW);
    int* row_hi = row_lo + NR;
    int* row_dg = row_hi + NR;
    float* row_ab = reinterpret_cast<float*>(row_dg + NR);
    float* red = reinterpret_cast<float*>(smem + C::OFF_RED);            // [4][NR]
    volatile int* vote = reinterpret_cast<volatile int*>(red + 4 * NR);  // [2][4]

    // ---- which sequence: longest first (ties by index), as the warp-sliced decode kernel
    int b = (int)blockIdx.z;
    if (p.order) {
        b = p.order[blockIdx.z];
    } else if (p.rank_in_cta) {
        int* rank_len = reinterpret_cast<int*>(smem + C::OFF_IDS);  // reused below for block ids
        if (tid < p.batch) rank_len[tid] = p.cu_k[tid + 1] - p.cu_k[tid];
        if (tid == 0) *pick = (int)blockIdx.z;
        __syncthreads();
        if (tid < p.batch) {
            const int ls = rank_len[tid];
            int rank = 0;
            for (int t = 0; t < p.batch; ++t) {
                const int lt = rank_len[t];
                rank += (lt > ls) || (lt == ls && t < tid);
            }
            if (rank == (int)blockIdx.z) *pick = tid;
        }
        __syncthreads();
        b = *pick;
        __syncthreads();  // rank_len is overwritten by the block ids below
    }
    const int hk = blockIdx.y % p.Hkv, split = blockIdx.x;

    TileView tv;
    if (!tile_view<NR, kTcNT>(p, b, 0, tv, split == 0)) return;
    if (split >= max(tv.nsplit, 1)) return;
    const bool single = tv.nsplit <= 1;
    const int t_begin = split * p.split_tiles;
    const int n_iter = max(0, min(tv.ntiles, t_begin + p.split_tiles) - t_begin);

    // ---- set-up: barriers (thread 128), tensor memory (warp 5), row metadata, q -> smem
    if (tid == 128) {
        for (int s = 0; s < KR; ++s) {
            mbar_init(&k_full[s], kTcProd / 2);  // both producers of the ring arrive, posting their own bytes
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < VR; ++s) {
            mbar_init(&v_full[s], kTcProd / 2);
            mbar_init(&v_empty[s], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], 4);  // one arrive per softmax warp
            mbar_init(&pv_done[x], 1);
            mbar_init(&drain[x], 1);
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 4) {
        tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
        tc::tmem_relinquish();
    }
    if (tid < NR) {
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
    {  // q rows -> shared memory: K-major, 128-byte swizzled rows of 64 columns, zero padded
        const T* q = static_cast<const T*>(p.q);
        constexpr int UNITS = DP / 8;
        uint8_t* qs = smem + C::OFF_Q;
        for (int idx = tid; idx < NR * UNITS; idx += kTcThreads) {
            const int r = idx / UNITS, u = idx - r * UNITS;
            int4 val = make_int4(0, 0, 0, 0);
            if (r < tv.rows && u * 8 < p.D) {
                const int rho = tv.row0 + r;
                const int i = rho / p.G, g = rho - i * p.G;
                val = __ldg(reinterpret_cast<const int4*>(q + (int64_t)(tv.q0 + i) * p.q_s0 +
                                                          (int64_t)(hk * p.G + g) * p.q_s1 + u * 8));
            }
            *reinterpret_cast<int4*>(qs + (u >> 3) * C::Q_CHUNK + swz128(r, u & 7)) = val;
        }
        fence_proxy_async_smem();  // generic-proxy writes, read by the tensor cores
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp >= 4) {
    if (warp >= 6) {
        // ---------------- TMA producers (warps 6..9): two per ring ----------------
        // Warps 6, 7 feed the K ring (16 KB units: one box per page piece), warps 8, 9 the V ring
        // (32 KB units: two 64-column boxes per page piece), so that neither ring's copies wait
        // behind the other's free slots.  Within a ring, copy number n of a unit goes to the
        // ring's producer n % 2.  Both producers of a ring visit every unit in order: each waits
        // for the slot to be free, arrives on the unit's full barrier (arrival count 2) posting
        // the bytes of its own copies, and only then issues them, so the barrier's transaction
        // count never runs ahead of the bytes announced.
        constexpr int PER_RING = kTcProd / 2;
        const bool is_k = warp < 6 + PER_RING;
        const int pi = (warp - 6) % PER_RING;
        int* ids = reinterpret_cast<int*>(smem + C::OFF_IDS);
        const int boxes_per_tile = kTcNT / p.box_rows;
        const int kbeg = tv.kt0 + t_begin * kTcNT;
        const int n_boxes = min(n_iter * boxes_per_tile, C::MAX_BOXES);
        const int32_t* bt_row = p.paged ? p.bt + (int64_t)b * p.bt_s0 : nullptr;
        for (int bi = (warp - 6) * 32 + lane; bi < n_boxes; bi += kTcProd * 32) {
            const int key = kbeg + bi * p.box_rows;
            ids[bi] = p.paged ? box_block(bt_row, p.bt_cols, p.num_blocks, p.P, key, tv.sk, p.err)
                              : (key < tv.sk ? 0 : -1);
        }
        named_barrier_sync(3, kTcProd * 32);  // the staged block ids are visible to every producer
        if (lane == 0 && !p.withhold) {
            const CUtensorMap* map = is_k ? &tm_k : &tm_v;
            prefetch_tmap(map);
            const uint64_t policy = l2_policy_evict_first();
            const int per = is_k ? boxes_per_tile : 2 * boxes_per_tile;  // copies per unit
            const int units = is_k ? KH : CH;                              // units per tile
            const int ring = is_k ? KR : VR;
            bool ok = true;
            for (int it = 0; ok && it < n_iter; ++it) {
                const int kt = kbeg + it * kTcNT;
                int blk[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int bi = it * boxes_per_tile + jj;
                    const int key = kt + jj * p.box_rows;
                    blk[jj] = jj >= boxes_per_tile ? -1
                              : bi < C::MAX_BOXES  ? ids[bi]
                              : (p.paged ? box_block(bt_row, p.bt_cols, p.num_blocks, p.P, key, tv.sk, p.err)
                                         : (key < tv.sk ? 0 : -1));
                }
                for (int c = 0; c < units; ++c) {
                    const int u = it * units + c;  // unit number in the ring
                    const int slot = u % ring;
                    uint64_t* fullb = is_k ? &k_full[slot] : &v_full[slot];
                    if (u >= ring && !tc_wait(is_k ? &k_empty[slot] : &v_empty[slot], ((u / ring) - 1) & 1,
                                              abort_flag, p.err, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    // (blk is read through selects: a runtime index would put it in local memory)
                    auto blk_of = [&](int jj) { return jj == 0 ? blk[0] : jj == 1 ? blk[1] : jj == 2 ? blk[2] : blk[3]; };
                    uint32_t mine = 0;
                    for (int op = pi; op < per; op += PER_RING)
                        if (blk_of(is_k ? op : op >> 1) >= 0) mine += (uint32_t)p.box_rows * 128u;
                    mbar_arrive_expect_tx(fullb, mine);
                    for (int op = pi; op < per; op += PER_RING) {
                        const int jj = is_k ? op : op >> 1, h = is_k ? 0 : op & 1;
                        const int bj = blk_of(jj);
                        if (bj < 0) continue;
                        const int key = kt + jj * p.box_rows;
                        const int c2 = p.paged ? key - (key / p.P) * p.P : p.cu_k[b] + key;
                        const int c3 = p.paged ? bj : 0;
                        if (is_k)
                            tma_load_4d(smem + C::OFF_K + slot * C::KUNIT + jj * p.box_rows * 128, map, fullb, c * 64,
                                        hk, c2, c3, policy);
                        else
                            tma_load_4d(smem + C::OFF_V + slot * C::VUNIT + h * C::KUNIT + jj * p.box_rows * 128, map,
                                        fullb, c * 128 + h * 64, hk, c2, c3, policy);
                    }
                }
            }
            // Leave only once the last units of this ring have landed: every earlier unit was
            // consumed before its slot was reused, so no copy of this producer is then still in
            // flight when the CTA's shared memory is released.  (Only the final ring-full is
            // waited for: a slot has no later unit, so its phase is unambiguous.)  Bounded like
            // every other wait; after an abort, units the other producer never issued run out.
            const int nu = n_iter * units;
            for (int k = max(0, nu - ring); k < nu; ++k)
                mbar_wait(is_k ? &k_full[k % ring] : &v_full[k % ring], (k / ring) & 1, p.wait_ns);
        }
        return;  // the other roles synchronise among themselves with named barrier 1
    }

    {
        // ---------------- MMA issuers: warp 4 S^T = K Q^T, warp 5 O^T += V^T P^T ----------------
        auto wait_all = [&](uint64_t* bar, uint32_t parity) {
            const bool r = __all_sync(0xffffffffu, tc_wait(bar, parity, abort_flag, p.err, p.wait_ns));
            tc::fence_after_sync();
            return r;
        };
        const bool is_s = warp == 4;
        bool ok = true;
        if (is_s) {
            constexpr uint32_t IDESC_S = tc::idesc_f16(128, NR, kBF16, false, false);
            const uint64_t d_k = tc::smem_desc_sw128(smem_addr(smem + C::OFF_K), 16, 1024);
            const uint64_t d_q = tc::smem_desc_sw128(smem_addr(smem + C::OFF_Q), 16, 1024);
            for (int j = 0; ok && j < n_iter; ++j) {
                // S buffer j % 2 was last read by the softmax of tile j - 2
                if (j >= 2 && !(ok = wait_all(&p_full[j & 1], ((j >> 1) - 1) & 1))) break;
                for (int h = 0; h < KH; ++h) {
                    const int u = j * KH + h, slot = u % KR;
                    if (!(ok = wait_all(&k_full[slot], (u / KR) & 1))) break;
                    {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t a = d_k + (uint64_t)((slot * C::KUNIT + kk * 32) >> 4);
                            const uint64_t bq = d_q + (uint64_t)((h * C::Q_CHUNK + kk * 32) >> 4);
                            tc::mma_ss_elect(tmem + C::T_S + (j & 1) * NR, a, bq, IDESC_S, (h | kk) ? 1u : 0u);
                        }
                        tc::commit_elect(&k_empty[slot]);
                        if (h == KH - 1) tc::commit_elect(&s_full[j & 1]);
                    }
                    __syncwarp();
                }
            }
        } else {
            constexpr uint32_t IDESC_O = tc::idesc_f16(128, NR, kBF16, true, false);
            const uint64_t d_v = tc::smem_desc_sw128(smem_addr(smem + C::OFF_V), C::KUNIT, 1024);
            const uint64_t d_p = tc::smem_desc_sw128(smem_addr(smem + C::OFF_P), 16, 1024);
            for (int j = 0; ok && j < n_iter; ++j) {
                if (!(ok = wait_all(&p_full[j & 1], (j >> 1) & 1))) break;
                const int valid = min(kTcNT, tv.sk - (tv.kt0 + (t_begin + j) * kTcNT));
                for (int c = 0; c < CH; ++c) {
                    const int u = j * CH + c, slot = u % VR;
                    if (!(ok = wait_all(&v_full[slot], (u / VR) & 1))) break;
                    if (valid < kTcNT) {  // V rows at or past sk -> 0 (P = 0 there; 0 * NaN is not 0)
                        uint8_t* vst = smem + C::OFF_V + slot * C::VUNIT;
                        const int zr = kTcNT - valid;
                        for (int idx = lane; idx < 2 * zr * 8; idx += 32) {
                            const int h = idx / (zr * 8), rem = idx - h * zr * 8;
                            *reinterpret_cast<int4*>(vst + h * C::KUNIT + (valid + (rem >> 3)) * 128 +
                                                     ((rem & 7) << 4)) = make_int4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        tc::fence_after_sync();
                    }
                    {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t a = d_v + (uint64_t)((slot * C::VUNIT + kk * 2048) >> 4);
                            const uint64_t bp = d_p + (uint64_t)(((j & 1) * C::P_BUF + (kk >> 2) * (NR * 128) +
                                                                  (kk & 3) * 32) >> 4);
                            tc::mma_ss_elect(tmem + C::T_O + c * NR, a, bp, IDESC_O, (j > 0 || kk > 0) ? 1u : 0u);
                        }
                        tc::commit_elect(&v_empty[slot]);
                        if (c == CH - 1) tc::commit_elect(&pv_done[j & 1]);
                    }
                    __syncwarp();
                }
            }
        }
        // every MMA this issuer started has completed before the tensor memory is released
        if (lane == 0) {
            tc::commit(&drain[is_s ? 0 : 1]);
            mbar_wait(&drain[is_s ? 0 : 1], 0, p.wait_ns);  // not cut short by an abort: MMAs may be in flight
        }
        __syncwarp();
        tc::fence_before_sync();
        named_barrier_sync(1, 192);
        if (is_s) {
            tc::fence_after_sync();
            tc::tmem_dealloc(tmem, C::TMEM_COLS);
        }
        return;
    }
    }  // warps 4..

    // ---------------- softmax (warps 0..3): thread = key 32 warp + lane of the tile ----------------
    // Control flow is uniform over the four warps: a warp whose wait fails (or that sees the
    // abort flag) still takes part in every named barrier, and all of them leave the loop
    // together, right after the per-tile vote.
    const uint32_t lane_addr = (uint32_t)(32 * warp) << 16;
    const int kk_me = 32 * warp + lane;
    // m[r]: running maximum of row r (log2 domain), the same in every thread.  lrow: the sum
    // of P over this warp's keys for row (lane mod NR), reduced over the warp every tile (one
    // register instead of NR per-thread partial sums).
    float m[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) m[r] = -INFINITY;
    float lrow = 0.f;
    // m_mine = m[lane mod NR], kept apart (updated by the same rule) so that no register array
    // is ever indexed by the lane: such an index would put the array in local memory
    const int myrow = lane & (NR - 1);
    float m_mine = -INFINITY;
    // the tile's keys are attended by every row (no masking needed) when the tile lies inside
    // the intersection of all rows' intervals
    int lo_max = 0, hi_min = INT32_MAX;
    for (int r = 0; r < tv.rows; ++r) {
        lo_max = max(lo_max, row_lo[r]);
        hi_min = min(hi_min, row_hi[r]);
    }
    const bool any_alibi = p.alibi != nullptr;
    bool ok = true;
    for (int j = 0; j < n_iter; ++j) {
        const int kt = tv.kt0 + (t_begin + j) * kTcNT;
        bool alive = !*abort_flag &&
                     __all_sync(0xffffffffu, tc_wait(&s_full[j & 1], (j >> 1) & 1, abort_flag, p.err, p.wait_ns));
        tc::fence_after_sync();
        float x[NR];
        bool grow = false;
        if (alive) {
            uint32_t sr[NR];
            tc::ld_cols<NR>(tmem + lane_addr + C::T_S + (j & 1) * NR, sr);
            tc::wait_ld();
            const int key = kt + kk_me;
            const bool inside = kt >= lo_max && kt + kTcNT - 1 <= hi_min && tv.rows == NR;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                float v = __uint_as_float(sr[r]);
                if (any_alibi)
                    v = biased_log2(v, p.scale_log2, row_ab[r], row_dg[r], key);
                else
                    v *= p.scale_log2;
                if (!inside) v = (key >= row_lo[r] && key <= row_hi[r]) ? v : -INFINITY;
                x[r] = v;
                grow |= v > m[r] + 8.f;  // lazy running maximum: only a growth past 2^8 counts
            }
        } else {
#pragma unroll
            for (int r = 0; r < NR; ++r) x[r] = -INFINITY;
        }
        const bool wgrow = __any_sync(0xffffffffu, grow);
        if (lane == 0) vote[(j & 1) * 4 + warp] = alive ? (wgrow ? 1 : 0) : 2;
        named_barrier_sync(2, 128);
        const int v0 = vote[(j & 1) * 4 + 0], v1 = vote[(j & 1) * 4 + 1], v2 = vote[(j & 1) * 4 + 2],
                  v3 = vote[(j & 1) * 4 + 3];
        if ((v0 | v1 | v2 | v3) & 2) {  // some warp gave up: all leave here
            ok = false;
            break;
        }
        if ((v0 | v1 | v2 | v3) & 1) {
            float t[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) t[r] = x[r];
            const float wmax = warp_reduce_scatter<NR, true>(t, lane);
            if (lane < NR) red[warp * NR + lane] = wmax;
            named_barrier_sync(2, 128);
            float alpha[NR];
            bool resc = false;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const float mx = fmaxf(fmaxf(red[r], red[NR + r]), fmaxf(red[2 * NR + r], red[3 * NR + r]));
                alpha[r] = 1.f;
                if (mx > m[r] + 8.f) {
                    alpha[r] = fast_exp2(m[r] - mx);  // 0 when m was -inf
                    m[r] = mx;
                    resc = true;
                }
            }
            {  // the same update for this lane's row of the running sum
                const float mx = fmaxf(fmaxf(red[myrow], red[NR + myrow]), fmaxf(red[2 * NR + myrow], red[3 * NR + myrow]));
                if (mx > m_mine + 8.f) {
                    lrow *= fast_exp2(m_mine - mx);
                    m_mine = mx;
                }
            }
            named_barrier_sync(2, 128);  // red is rewritten by the next reduction
            // (resc is the same in every thread: all of them read the same maxima)
            if (resc && j > 0) {
                // O^T holds P.V(j-1) accumulated with the old maxima: wait for it, rescale
                if (__all_sync(0xffffffffu, tc_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, p.err,
                                                    p.wait_ns))) {
                    tc::fence_after_sync();
#pragma unroll 1
                    for (int c = 0; c < CH; ++c) {
                        uint32_t o[NR];
                        tc::ld_cols<NR>(tmem + lane_addr + C::T_O + c * NR, o);
                        tc::wait_ld();
#pragma unroll
                        for (int r = 0; r < NR; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha[r]);
                        tc::st_cols<NR>(tmem + lane_addr + C::T_O + c * NR, o);
                    }
                    tc::wait_st();
                }  // else the abort flag is set: the next vote ends the loop
            }
        }
        // P = exp2(x - m); this thread's key column of P^T (in place of x)
#pragma unroll
        for (int r = 0; r < NR; ++r) x[r] = fast_exp2(x[r] - (m[r] == -INFINITY ? 0.f : m[r]));
        // P^T buffer j % 2 was last read by P.V(j-2)
        if (j < 2 || __all_sync(0xffffffffu, tc_wait(&pv_done[j & 1], ((j - 2) >> 1) & 1, abort_flag, p.err,
                                                      p.wait_ns))) {
            uint8_t* pb = smem + C::OFF_P + (j & 1) * C::P_BUF + (kk_me >> 6) * (NR * 128);
            const int u16 = (kk_me & 63) >> 3, e = kk_me & 7;
#pragma unroll
            for (int r = 0; r < NR; ++r) *reinterpret_cast<T*>(pb + swz128(r, u16) + e * 2) = static_cast<T>(x[r]);
            fence_proxy_async_smem();
        }
        lrow += warp_reduce_scatter<NR, false>(x, lane);  // this tile's sums over the warp's keys
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[j & 1]);
    }

    // ---- epilogue: l over the CTA, O^T / l -> out (or this split's partial result) ----
    if (ok && n_iter > 0)
        ok = __all_sync(0xffffffffu, tc_wait(&pv_done[(n_iter - 1) & 1], ((n_iter - 1) >> 1) & 1, abort_flag, p.err,
                                             p.wait_ns));
    tc::fence_after_sync();
    if (lane < NR) red[warp * NR + lane] = lrow;
    named_barrier_sync(2, 128);
    float inv[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const float L = red[r] + red[NR + r] + red[2 * NR + r] + red[3 * NR + r];
        inv[r] = L > 0.f ? 1.f / L : 0.f;
    }
    if (ok && !*abort_flag) {
        T* out = static_cast<T*>(p.out);
#pragma unroll 1
        for (int c = 0; c < CH; ++c) {
            const int d = c * 128 + kk_me;  // O^T lane = head-dim column within the chunk
            uint32_t o[NR];
            if (n_iter > 0) {
                tc::ld_cols<NR>(tmem + lane_addr + C::T_O + c * NR, o);
                tc::wait_ld();
            } else {
#pragma unroll
                for (int r = 0; r < NR; ++r) o[r] = 0u;
            }
            if (d >= p.D) continue;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r >= tv.rows) break;
                const int rho = tv.row0 + r;
                const int i = rho / p.G, g = rho - i * p.G;
                const int64_t t = tv.q0 + i;
                const int h = hk * p.G + g;
                const float val = __uint_as_float(o[r]) * inv[r];
                if (single)
                    out[t * p.o_s0 + (int64_t)h * p.o_s1 + d] = static_cast<T>(val);
                else
                    p.part_o[((int64_t)split * p.part_stride + t * p.H + h) * p.D + d] = val;
            }
        }
        if (warp == 0 && lane < tv.rows) {
            const int r = lane;
            const int rho = tv.row0 + r;
            const int i = rho / p.G, g = rho - i * p.G;
            const int64_t t = tv.q0 + i;
            const int h = hk * p.G + g;
            const float L = red[r] + red[NR + r] + red[2 * NR + r] + red[3 * NR + r];
            const float lse = L > 0.f ? (m_mine + log2f(L)) * 0.69314718055994531f : -INFINITY;  // r == myrow
            if (single)
                p.lse[(int64_t)h * p.lse_s0 + t + (int64_t)b * p.lse_sb] = lse;
            else
                p.part_lse[(int64_t)split * p.part_stride + t * p.H + h] = lse;
        }
    }
    tc::fence_before_sync();
    named_barrier_sync(1, 192);  // with the MMA issuers; warp 4 then releases the tensor memory
}

template <int DP>
struct TcRings;  // ring depths (K units of 16 KB, V units of 32 KB) per padded head dim
template <>
struct TcRings<128> {
    static constexpr int K = 6, V = 3;
};
template <>
struct TcRings<256> {
    static constexpr int K = 5, V = 3;
};
template <>
struct TcRings<512> {
    static constexpr int K = 4, V = 3;
};

template <typename T, int DP, int NR>
int run_decode_tc(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& sp, const SplitPlan& plan,
                  cudaStream_t stream, char* msg, size_t msg_len) {
    using C = TcCfg<DP, NR, TcRings<DP>::K, TcRings<DP>::V>;
    auto kern = decode_tc_kernel<T, DP, NR, TcRings<DP>::K, TcRings<DP>::V>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "cudaFuncSetAttribute(decode_tc, %d bytes): %s", C::SMEM, cudaGetErrorString(e));
            return PA_ERR_CUDA;
        }
        configured = true;
    }
    if (sp.order) {
        const int rc = launch_longest_first(sp.cu_k, sp.batch, const_cast<int*>(sp.order), stream, msg, msg_len);
        if (rc != PA_OK) return rc;
    }
    dim3 grid(plan.max_splits, sp.Hkv, sp.batch);
    NvtxRange nv("pa::decode_tc_kernel");
    timer_begin(PA_KC_SPLITKV, stream);
    kern<<<grid, TcRoles<NR>::THREADS, C::SMEM, stream>>>(tk, tv, sp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "decode_tc launch: %s", cudaGetErrorString(e));
        return PA_ERR_CUDA;
    }
    timer_end(PA_KC_SPLITKV, stream);
    count_launches(1);
    return PA_OK;
}

template <typename T, int DP, int NR>
int tc_occupancy_one() {
    using C = TcCfg<DP, NR, TcRings<DP>::K, TcRings<DP>::V>;
    static int n = [] {
        auto kern = decode_tc_kernel<T, DP, NR, TcRings<DP>::K, TcRings<DP>::V>;
        int v = 0;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, TcRoles<NR>::THREADS, C::SMEM) != cudaSuccess) {
            (void)cudaGetLastError();
            return 1;
        }
        return v > 0 ? v : 1;
    }();
    return n;
}

template <typename T>
int tc_occupancy_t(int dp, int nr) {
    if (dp == 128) return nr == 16 ? tc_occupancy_one<T, 128, 16>() : tc_occupancy_one<T, 128, 32>();
    if (dp == 256) return nr == 16 ? tc_occupancy_one<T, 256, 16>() : tc_occupancy_one<T, 256, 32>();
    return nr == 16 ? tc_occupancy_one<T, 512, 16>() : tc_occupancy_one<T, 512, 32>();
}

template <typename T>
int launch_tc_t(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& sp, const SplitPlan& plan,
                cudaStream_t stream, char* msg, size_t msg_len) {
    const int nr = plan.mt == 1 ? 16 : 32;
#define PA_TC_CASE(DPV, NRV) \
    if (plan.dp == DPV && nr == NRV) return run_decode_tc<T, DPV, NRV>(tk, tv, sp, plan, stream, msg, msg_len);
    PA_TC_CASE(128, 16)
    PA_TC_CASE(128, 32)
    PA_TC_CASE(256, 16)
    PA_TC_CASE(256, 32)
    PA_TC_CASE(512, 16)
    PA_TC_CASE(512, 32)
#undef PA_TC_CASE
    snprintf(msg, msg_len, "no tensor-core decode kernel for head_dim tile %d, rows %d", plan.dp, nr);
    return PA_ERR_UNSUPPORTED;
}

}  // namespace

int decode_tc_occupancy(int dtype, int dp, int nr) {
    return dtype == PA_BF16 ? tc_occupancy_t<__nv_bfloat16>(dp, nr) : tc_occupancy_t<__half>(dp, nr);
}

int launch_decode_tc(const CUtensorMap& tk, const CUtensorMap& tv, const SplitParams& sp, const SplitPlan& plan,
                     int dtype, cudaStream_t stream, char* msg, size_t msg_len) {
    return dtype == PA_BF16 ? launch_tc_t<__nv_bfloat16>(tk, tv, sp, plan, stream, msg, msg_len)
                            : launch_tc_t<__half>(tk, tv, sp, plan, stream, msg, msg_len);
}

}  // namespace pa
