// Tensor-core prefill / chunked-prefill kernels for paged varlen attention (sm_103a).
//
// Two persistent kernels, one CTA per SM, each taking work items from a device counter:
//   prefill_kernel     head_dim <= 128: an item is two consecutive 128-row query tiles (A, B)
//                      of one (sequence, kv head), so every K/V tile feeds both;
//   prefill256_kernel  head_dim 129..256: an item is one 128-row query tile (two tiles' O
//                      would not fit the 512 TMEM columns beside the S buffers).
// A tile's rows are the (query i, head g) pairs of the kv head's GQA group, ordered i G + g,
// so each K/V tile feeds all G query heads.  A tile holds floor(128 / G) whole queries; when
// G does not divide 128 its last 128 mod G rows are padding (masked, never written).
// Roles (384 threads, three warpgroups):
//   warp 0      takes the items (atomic add on the counter, a scan of cu_seqlens_q) and
//               publishes each in a shared-memory slot; loads q and the K tiles by TMA
//               through the block table (one box per page piece; the paged layout of
//               "flash-attn-varlen paged expects k/v tensors of rank 4", What it means)
//   warp 2      loads the V tiles
//   warps 1, 3  MMA issuers (one elected lane each; warp 1 also owns the tensor memory):
//               S = Q K_j^T (tcgen05.mma, A and B from shared memory, S in TMEM) and
//               O += P V_j  (tcgen05.mma, A = P from TMEM, B = V from shared memory)
//   warps 4..11 softmax: each warp owns 16 rows (TMEM lanes), four threads per row; reads S
//               from TMEM, masks, keeps the running max and sum, writes P (16-bit) over the
//               columns of S it came from, and rescales O in TMEM only when the running max
//               grew by more than 2^8 (otherwise the stale max stays: exact after the final
//               division); writes out O and the log-sum-exp at the end of an item.
// Every barrier and ring continues from item to item through running counters, so the
// producers load the next item while the issuers and the softmax finish the current one.
//
// Mask (bottom-right aligned): query i of a sequence with sq queries and sk keys attends
// key j iff 0 <= j < sk, j >= i + sk - sq - window_left (window_left >= 0), and
// j <= i + sk - sq + window_right (window_right >= 0).

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <type_traits>

#include "tc_common.cuh"

namespace pa {
namespace {

constexpr int kPrefillThreads = 384;  // three warpgroups
// Register split (setmaxnreg): the launch gives 384 x 168; warpgroup 0 (producer, MMA
// issuers, V producer) drops to 72 and the two softmax warpgroups rise to 216:
// 128 x 72 + 256 x 216 = 64,512, the launch total.
constexpr int kRegsControl = 72, kRegsSoftmax = 216;

struct PrefillParams {
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
    int64_t num_blocks, total_q;
    int paged;
    int box_rows, boxes_per_tile;
    int max_sq, max_sk;
    float scale_log2;
    int wl, wr;
    const float* alibi;  // per-query-head slopes of the linear position bias, or nullptr
    int rows_cap;
    int pairs;     // an upper bound of the number of work units (tile pairs or tiles) per kv head
    int* counter;  // the take counter of (work unit, kv head) items, zeroed before the launch
    unsigned int* err;
    uint64_t wait_ns;  // bound on every wait
    int withhold;      // test hook: issue no loads
};


// Layout of prefill_kernel at padded head dim DP (64 or 128).
template <int DP>
struct PfCfg {
    static constexpr int CH = DP / 64;              // 64-column (128-byte) chunks
    static constexpr int Q_TILE = CH * 128 * 128;   // one 128-row q tile
    static constexpr int KV_TILE = CH * 128 * 128;  // 128 keys x DP
    static constexpr int KS = 3;                    // K stages
    static constexpr int VS = DP == 64 ? 3 : 2;     // V stages
    static constexpr int OFF_Q = 0;                 // q tile A, then q tile B
    static constexpr int OFF_K = 2 * Q_TILE;
    static constexpr int OFF_V = OFF_K + KS * KV_TILE;
    static constexpr int OFF_BAR = OFF_V + VS * KV_TILE;
    // q_full, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], s_full[2], p_full[2], pv_done[2],
    // drain[2], item_ready[2], item_free[2], q_free
    static constexpr int NBAR = 1 + 2 * KS + 2 * VS + 13;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem base, abort flag
    static constexpr int OFF_SLOT = OFF_MISC + 16;       // two item slots
    static constexpr int OFF_IDS = OFF_SLOT + 128;       // block-id windows of the K and V producers
    static constexpr int WIN = 128;                      // boxes per window
    static constexpr int SMEM = OFF_IDS + 2 * WIN * 4 + 1024;
    static constexpr uint32_t T_S0 = 0, T_S1 = 128;        // S (then P) of tiles A and B
    static constexpr uint32_t T_O0 = 256, T_O1 = 256 + DP;  // O of tiles A and B
    static_assert(256 + 2 * DP <= 512, "TMEM columns");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

// Bounded wait that also gives up as soon as another role of the CTA has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
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

// Issues the K (or V) boxes of the CTA's 128-key tile number `j` (first key kt0 + 128 j)
// into `dst`.  ids[j * boxes_per_tile + jj] holds the physical block of box jj, or a
// negative value for a box that is not loaded.
__device__ __forceinline__ void issue_kv_tile(const PrefillParams& p, const CUtensorMap* map, uint8_t* dst,
                                              uint64_t* bar, const int* ids, int j, int hk, int kt0, int k0,
                                              int CH) {
    const int kt = kt0 + j * 128;
    int blk[4];
    uint32_t bytes = 0;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        blk[jj] = jj < p.boxes_per_tile ? ids[j * p.boxes_per_tile + jj] : -1;
        if (blk[jj] >= 0) bytes += (uint32_t)(CH * p.box_rows * 128);
    }
    mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        if (blk[jj] < 0) continue;
        const int key = kt + jj * p.box_rows;
        const int c2 = p.paged ? key - (key / p.P) * p.P : k0 + key;
        const int c3 = p.paged ? blk[jj] : 0;
        for (int c = 0; c < CH; ++c)
            tma_load_4d(dst + (c * 128 + jj * p.box_rows) * 128, map, bar, c * 64, hk, c2, c3, 0ull);
    }
}

// 4 x 4 transpose of 32-bit values over the four threads of a quad (t = lane % 4): thread t
// holds a[j] = M[t][j] on entry and a[j] = M[j][t] on exit.  Two butterfly stages: lanes t and
// t ^ 1 swap the odd/even entries of each pair, then lanes t and t ^ 2 swap the pairs.
__device__ __forceinline__ void quad_transpose(uint32_t (&a)[4], int t) {
    const bool b = t & 1, h = t & 2;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const uint32_t r = __shfl_xor_sync(0xffffffffu, b ? a[2 * c] : a[2 * c + 1], 1);
        if (b) a[2 * c] = r; else a[2 * c + 1] = r;
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const uint32_t r = __shfl_xor_sync(0xffffffffu, h ? a[e] : a[2 + e], 2);
        if (h) a[e] = r; else a[2 + e] = r;
    }
}

// The work of one item.  Warp 0 computes it and publishes it in a slot; every role reads it.
struct PfItem {
    int b, u, hk, q0, sq, sk, k0, i0, kt0, n_tiles, has_b, bad;
};
static_assert(sizeof(PfItem) <= 64, "item slot");

__device__ __forceinline__ void pf_item(const PrefillParams& p, int qpt, PfItem& it) {
    it.q0 = p.cu_q[it.b];
    const int q1 = p.cu_q[it.b + 1];
    it.k0 = p.cu_k[it.b];
    const int k1 = p.cu_k[it.b + 1];
    it.sq = q1 - it.q0;
    it.sk = k1 - it.k0;
    it.bad = it.sq < 0 || it.sk < 0 || it.sq > p.max_sq || it.sk > p.max_sk || it.q0 < 0 || q1 > p.total_q ||
             (!p.paged && (it.k0 < 0 || k1 > p.num_blocks));
    it.n_tiles = 0;
    if (it.bad) return;
    it.i0 = it.u * 2 * qpt;
    it.has_b = it.i0 + qpt < it.sq;
    const int i_last = min(it.sq - 1, it.i0 + (it.has_b ? 2 : 1) * qpt - 1);
    const int64_t cdiag = (int64_t)it.sk - it.sq;
    const int64_t lo = p.wl >= 0 ? max64(0, it.i0 + cdiag - p.wl) : 0;
    const int64_t hi = p.wr >= 0 ? min64((int64_t)it.sk - 1, i_last + cdiag + p.wr) : (int64_t)it.sk - 1;
    it.kt0 = hi >= lo ? (int)(lo & ~int64_t(127)) : 0;
    it.n_tiles = hi >= lo ? (int)((hi - it.kt0) / 128 + 1) : 0;
}

// ---------------------------------------------------------------------------------------------
// prefill_kernel: head_dim <= 128, items of two query tiles.
//
// Per item the issuers order their products S_X(0), PV_X(0), S_X(1), PV_X(1), ... (X = A for
// warp 1, B for warp 3): the in-order pipe of one issuing thread is what lets S_X(j+1)
// overwrite P_X(j).  The two tiles ping-pong: while the softmax works on one tile, the tensor
// pipe runs the other tile's P.V and next Q.K^T.  TMEM columns: S_A [0,128), S_B [128,256),
// O_A [256, 256+DP), O_B [256+DP, 256+2 DP).  Between items:
//   * each producer stages the block ids of its own item's boxes (a window of C::WIN boxes,
//     restaged when a tile runs past it);
//   * the next q tiles are loaded once both issuers have committed q_free after the last
//     Q.K^T of the item that read them;
//   * the first P.V of an item (which overwrites O_X) waits for P_X(0), which the softmax
//     hands over only after its epilogue has read O_X of the previous item;
//   * the V stage of an item's last key tile is released by the epilogue (after P.V).
// A CTA per tile pair instead spent ~20 % of its time outside the steady state (launch,
// set-up, block-id staging, the first loads, the epilogue); the persistent form measured
// 2.3 % faster on the causal prefill batch and 9 % at head_dim 64.
// ALIBI: the scores carry the linear position bias -slope_h * |diagonal - key| (a separate
// instantiation, so the unbiased softmax has no extra arithmetic).
template <typename T, int DP, bool ALIBI>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
    using C = PfCfg<DP>;
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* k_empty = k_full + C::KS;
    uint64_t* v_full = k_empty + C::KS;
    uint64_t* v_empty = v_full + C::VS;
    uint64_t* s_full = v_empty + C::VS;    // [tile]
    uint64_t* p_full = s_full + 2;         // [tile]
    uint64_t* pv_done = p_full + 2;        // [tile]: the tile's last P.V of the item has completed
    uint64_t* drain = pv_done + 2;         // [issuer]
    uint64_t* item_ready = drain + 2;      // [slot]
    uint64_t* item_free = item_ready + 2;  // [slot]
    uint64_t* q_free = item_free + 2;      // both issuers' Q.K^T of the item have completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile uint32_t* abort_flag = tmem_slot + 1;
    PfItem* slots = reinterpret_cast<PfItem*>(smem + C::OFF_SLOT);
    if (tid == 64) {
        mbar_init(q_full, 1);
        for (int s = 0; s < C::KS; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 2);  // one arrive per query tile (softmax side)
        }
        for (int s = 0; s < C::VS; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 2);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], 8);  // one arrive per softmax warp
            mbar_init(&pv_done[x], 1);
            mbar_init(&drain[x], 1);
            mbar_init(&item_ready[x], 1);
            mbar_init(&item_free[x], 11);  // the V producer, two issuers, eight softmax warps
        }
        mbar_init(q_free, 2);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int qpt = 128 / p.G;    // whole queries per 128-row tile
    const int trows = qpt * p.G;  // rows of a tile that hold queries (the rest are padding)
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
        const bool r = __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, p.err, p.wait_ns));
        tc::fence_after_sync();
        return r;
    };
    // item k of this CTA, from slot k % 2 (b < 0: no more items)
    auto take_slot = [&](int k, PfItem& it) -> bool {
        if (!wait_all(&item_ready[k & 1], (k >> 1) & 1)) return false;
        it = slots[k & 1];
        __syncwarp();
        if (lane == 0) mbar_arrive(&item_free[k & 1]);
        return true;
    };
    // Issues the item's key tiles into a K or V ring from this warp (lane 0 issues); the whole
    // warp stages the block ids of up to C::WIN boxes at a time.  Returns false on an abort.
    auto produce = [&](const PfItem& it, const CUtensorMap* map, uint8_t* ring, uint64_t* fullb, uint64_t* emptyb,
                       int stages, int g0, int* win) -> bool {
        const int32_t* bt_row = p.paged ? p.bt + (int64_t)it.b * p.bt_s0 : nullptr;
        const int win_tiles = C::WIN / p.boxes_per_tile;
        int jw = -win_tiles;  // first tile of the staged window
        for (int j = 0; j < it.n_tiles; ++j) {
            if (j >= jw + win_tiles) {  // stage the window that starts at tile j
                jw = j;
                __syncwarp();
                const int n_boxes = min((it.n_tiles - j) * p.boxes_per_tile, C::WIN);
                for (int bi = lane; bi < n_boxes; bi += 32) {
                    const int key = it.kt0 + j * 128 + bi * p.box_rows;
                    win[bi] = p.paged ? box_block(bt_row, p.bt_cols, p.num_blocks, p.P, key, it.sk, p.err)
                                      : (key < it.sk ? 0 : -1);
                }
                __syncwarp();
            }
            const int g = g0 + j, s = g % stages;
            if (g >= stages && !wait_all(&emptyb[s], ((g / stages) - 1) & 1)) return false;
            if (lane == 0)
                issue_kv_tile(p, map, ring + s * C::KV_TILE, &fullb[s], win, j - jw, it.hk, it.kt0 + jw * 128, it.k0,
                              C::CH);
        }
        return true;
    };

    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
    if (warp == 0) {
        // ---------------- item taker, q and K producer ----------------
        // Items: w = pair * Hkv + kv head over the pairs of 128-row tiles of prefill-class
        // sequences, sequence by sequence, each sequence's last (longest causal) pair first; a
        // pair index past the list ends it.  (Taking the kv heads outermost, so that all SMs
        // read the same head's K/V tiles at once, measured 8 % slower.)
        const int total = p.pairs * p.Hkv;
        int* win = reinterpret_cast<int*>(smem + C::OFF_IDS);
        if (!p.withhold) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
        }
        int w_next = lane == 0 ? atomicAdd(p.counter, 1) : 0;
        int ld = 0, gk = 0;  // items with loads so far, K tiles issued so far
        for (int k = 0;; ++k) {
            const int w = __shfl_sync(0xffffffffu, w_next, 0);
            PfItem it{};
            it.b = -1;
            if (w < total) {
                const int pair = w / p.Hkv;
                it.hk = w - pair * p.Hkv;
                int remaining = pair;
                for (int base = 0; base < p.batch && it.b < 0; base += 32) {
                    const int bb = base + lane;
                    int pairs = 0;
                    if (bb < p.batch) {
                        const int sqb = p.cu_q[bb + 1] - p.cu_q[bb];
                        pairs = (int64_t)sqb * p.G > p.rows_cap ? (sqb + 2 * qpt - 1) / (2 * qpt) : 0;
                    }
                    int incl = pairs;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const int v = __shfl_up_sync(0xffffffffu, incl, off);
                        if (lane >= off) incl += v;
                    }
                    const unsigned hit = __ballot_sync(0xffffffffu, remaining < incl);
                    if (hit) {
                        const int src = __ffs(hit) - 1;
                        const int excl = __shfl_sync(0xffffffffu, incl - pairs, src);
                        const int cnt = __shfl_sync(0xffffffffu, pairs, src);
                        it.b = base + src;
                        it.u = cnt - 1 - (remaining - excl);
                    } else {
                        remaining -= __shfl_sync(0xffffffffu, incl, 31);
                    }
                }
                if (it.b >= 0) pf_item(p, qpt, it);
            }
            // the next claim's latency overlaps this item's loads
            if (it.b >= 0 && lane == 0) w_next = atomicAdd(p.counter, 1);
            if (k >= 2 && !wait_all(&item_free[k & 1], ((k >> 1) - 1) & 1)) break;
            if (lane == 0) {
                slots[k & 1] = it;
                mbar_arrive(&item_ready[k & 1]);  // release: the slot's stores precede the arrive
            }
            if (it.b < 0) break;
            if (it.bad) {
                if (lane == 0) flag_error(p.err, PA_ERR_DEVICE_BOUNDS);
                continue;
            }
            if (it.n_tiles == 0) continue;
            // the q tiles, once the previous item's last Q.K^T products have completed (issuing
            // the item's first K tile before this wait measured 2-3 % slower)
            if (ld >= 1 && !wait_all(q_free, (ld - 1) & 1)) break;
            if (lane == 0 && !p.withhold) {
                mbar_arrive_expect_tx(q_full, (it.has_b ? 2 : 1) * C::CH * trows * 128);
                for (int x = 0; x < (it.has_b ? 2 : 1); ++x)
                    for (int c = 0; c < C::CH; ++c)
                        tma_load_4d(smem + C::OFF_Q + x * C::Q_TILE + c * 128 * 128, &tm_q, q_full, c * 64,
                                    it.hk * p.G, it.q0 + it.i0 + x * qpt, 0, 0ull);
            }
            if (!p.withhold && !produce(it, &tm_k, smem + C::OFF_K, k_full, k_empty, C::KS, gk, win)) break;
            gk += it.n_tiles;
            ++ld;
        }
    } else if (warp == 2) {
        // ---------------- V producer ----------------
        int* win = reinterpret_cast<int*>(smem + C::OFF_IDS) + C::WIN;
        if (!p.withhold) prefetch_tmap(&tm_v);
        int gv = 0;
        for (int k = 0;; ++k) {
            PfItem it;
            if (!take_slot(k, it) || it.b < 0) break;
            if (it.bad || it.n_tiles == 0) continue;
            if (!p.withhold && !produce(it, &tm_v, smem + C::OFF_V, v_full, v_empty, C::VS, gv, win)) break;
            gv += it.n_tiles;
        }
    } else {
        // ---------------- MMA issuers: warp 1 for tile A, warp 3 for tile B ----------------
        // Per issuer S_x(0), PV_x(0), S_x(1), ..., and across items the next item's S_x(0)
        // follows this item's last P.V in the same thread's order.  A tcgen05.mma costs its
        // issuing thread ~50-100 cycles, close to the 64 cycles a 128x128x16 product occupies
        // the pipe, so each tile has its own issuer.
        constexpr uint32_t IDESC_S = tc::idesc_f16(128, 128, kBF16, false, false);
        constexpr uint32_t IDESC_O = tc::idesc_f16(128, DP, kBF16, false, true);
        const int x = warp == 1 ? 0 : 1;
        const uint64_t da = tc::smem_desc_sw128(smem_addr(smem + C::OFF_Q + x * C::Q_TILE), 16, 1024);
        const uint64_t dk0 = tc::smem_desc_sw128(smem_addr(smem + C::OFF_K), 16, 1024);
        const uint64_t dv0 = tc::smem_desc_sw128(smem_addr(smem + C::OFF_V), 128 * 128, 1024);
        const uint32_t d_s = tmem + (x ? C::T_S1 : C::T_S0);
        const uint32_t d_o = tmem + (x ? C::T_O1 : C::T_O0);
        // lq: items with loads so far; gk, gv: ring positions; sx: this tile's S count
        int lq = 0, gk = 0, gv = 0, sx = 0;
        bool ok = true;
        auto issue_s = [&](int g) {  // S_x = Q_x K^T of the K tile at ring position g
            const uint64_t db = dk0 + (uint64_t)((g % C::KS) * (C::KV_TILE >> 4));
#pragma unroll
            for (int kk = 0; kk < DP / 16; ++kk) {
                const uint64_t off = (uint64_t)((kk >> 2) * (128 * 128 / 16) + (kk & 3) * 2);
                tc::mma_ss_elect(d_s, da + off, db + off, IDESC_S, kk > 0 ? 1u : 0u);
            }
            tc::commit_elect(&s_full[x]);
        };
        for (int k = 0; ok; ++k) {
            PfItem it;
            if (!take_slot(k, it) || it.b < 0) break;
            if (it.bad || it.n_tiles == 0) continue;
            const int n = it.n_tiles;
            if (x == 0 || it.has_b) {
                if (!(ok = wait_all(q_full, lq & 1))) break;
                if (!(ok = wait_all(&k_full[gk % C::KS], (gk / C::KS) & 1))) break;
                // q_free takes two arrivals an item, each when an issuer's last Q.K^T of it has
                // completed; without tile B both come from this issuer (were issuer 1 to arrive
                // at once for such an item, it could arrive for the next one too before this
                // issuer finished, and the next q tiles would overwrite q this item still reads)
                const int qf = it.has_b ? 1 : 2;
                issue_s(gk);  // the whole warp, one elected lane issuing
                if (n == 1)      // the item's last Q.K^T is issued
                    for (int c = 0; c < qf; ++c) tc::commit_elect(q_free);
                __syncwarp();
                for (int j = 0; ok && j < n; ++j) {
                    const int g_v = gv + j;
                    if (!(ok = wait_all(&v_full[g_v % C::VS], (g_v / C::VS) & 1))) break;
                    uint8_t* vst = smem + C::OFF_V + (g_v % C::VS) * C::KV_TILE;
                    const int valid = min(128, it.sk - (it.kt0 + j * 128));
                    if (valid < 128) {  // keys at or past sk: zero V rows so P = 0 never meets NaN
                        const int zr = 128 - valid;
                        for (int idx = lane; idx < C::CH * zr * 8; idx += 32) {
                            const int c = idx / (zr * 8), rem = idx - c * zr * 8;
                            *reinterpret_cast<int4*>(vst + (c * 128 + valid + (rem >> 3)) * 128 + ((rem & 7) << 4)) =
                                make_int4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        tc::fence_after_sync();
                    }
                    const bool more = j + 1 < n;
                    const int g_k = gk + j + 1;
                    if (more && !(ok = wait_all(&k_full[g_k % C::KS], (g_k / C::KS) & 1))) break;
                    if (!(ok = wait_all(&p_full[x], (sx + j) & 1))) break;
                    {  // the whole warp, one elected lane issuing
                        const uint64_t db = dv0 + (uint64_t)((g_v % C::VS) * (C::KV_TILE >> 4));
                        const uint32_t first = j > 0 ? 1u : 0u;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            tc::mma_ts_elect(d_o, d_s + kk * 8, db + (uint64_t)(kk * (2048 / 16)), IDESC_O,
                                             kk > 0 ? 1u : first);
                        if (j + 1 == n) tc::commit_elect(&pv_done[x]);
                        if (more) {
                            issue_s(g_k);
                            if (j + 2 == n)
                                for (int c = 0; c < qf; ++c) tc::commit_elect(q_free);
                        }
                    }
                    __syncwarp();
                }
                if (!ok) break;
                sx += n;
            }  // no tile B: issuer 0 arrives on q_free for both
            __syncwarp();
            gk += n;
            gv += n;
            ++lq;
        }
        // every MMA this issuer started has completed before tensor memory is released
        if (lane == 0) {
            tc::commit(&drain[x]);
            mbar_wait(&drain[x], 0, p.wait_ns);  // not cut short by an abort: MMAs may be in flight
        }
        __syncwarp();
    }
    } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    {
        // ---------------- softmax: warps 4..11, tile A and then tile B at every key tile ----------------
        // Warp w reaches TMEM lanes 32 (w % 4) .. +31 and takes the half hh = (w - 4) / 4 of
        // them: lanes lb .. lb + 15 with lb = 32 (w % 4) + 16 hh.  Thread t holds rows
        // lb + t/4 (q = 0) and lb + t/4 + 8 (q = 1) of each tile; the four threads of a quad
        // split a row's 128 keys (keys 8k + 2 (t % 4) + {0, 1}, k = 0..15), so row maxima and
        // sums are quad reductions and P lands in the columns its own thread read S from.
        const int lg = warp & 3, hh = (warp - 4) >> 2;
        const int gid = lane >> 2, tig = lane & 3;
        const int lb = lg * 32 + hh * 16;
        const uint32_t lane_addr = (uint32_t)lb << 16;
        T* out = static_cast<T*>(p.out);
        struct TileRows {
            int lo[2], hi[2];
            float m[2], l[2];
            int dg[2];
            float ab[2];
        };
        // This thread's two rows of a tile, lb + gid + 8q: query qi[q] of the tile, head gi[q] of
        // the group (the same in every item); rows at or past trows are padding.
        int qi[2], gi[2];
        bool pad[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int r = lb + gid + 8 * q;
            qi[q] = r / p.G;
            gi[q] = r - qi[q] * p.G;
            pad[q] = r >= trows;
        }
        int gk = 0, gv = 0, sa = 0, sb = 0, aa = 0, ab_ = 0;  // ring positions, S and P.V counts
        bool ok = true;
        for (int k = 0; ok; ++k) {
            PfItem it;
            if (!take_slot(k, it) || it.b < 0) break;
            if (it.bad) continue;
            const int b = it.b, hk = it.hk;
            const int64_t cdiag = (int64_t)it.sk - it.sq;
            const int64_t rows_total = (int64_t)it.sq * p.G;
            auto tile_rho = [&](int x, int r) -> int64_t { return (int64_t)(it.i0 + x * qpt) * p.G + r; };
            auto row_live = [&](int x, int r) { return r < trows && tile_rho(x, r) < rows_total; };
            if (it.n_tiles == 0) {  // no row attends any key: out = 0, lse = -inf
                const int x = (warp - 4) >> 2, r = (warp & 3) * 32 + lane;
                if (row_live(x, r)) {
                    const int64_t rho = tile_rho(x, r);
                    const int i = (int)(rho / p.G), g = (int)(rho - (int64_t)i * p.G);
                    const int64_t t = it.q0 + i;
                    const int h = hk * p.G + g;
                    for (int d = 0; d < p.D; d += 8)
                        *reinterpret_cast<int4*>(out + t * p.o_s0 + (int64_t)h * p.o_s1 + d) = make_int4(0, 0, 0, 0);
                    p.lse[(int64_t)h * p.lse_s0 + t + (int64_t)b * p.lse_sb] = -INFINITY;
                }
                continue;
            }
            const int n = it.n_tiles;
            // query index (within the sequence) of row q of tile x, and whether it holds a query
            auto qrow = [&](int x, int q) { return it.i0 + x * qpt + qi[q]; };
            auto live = [&](int x, int q) { return !pad[q] && qrow(x, q) < it.sq; };
            auto init_rows = [&](int x, TileRows& st) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    st.lo[q] = 0;
                    st.hi[q] = -1;
                    st.dg[q] = 0;
                    st.ab[q] = 0.f;
                    if (live(x, q)) {
                        const int64_t diag = qrow(x, q) + cdiag;
                        st.lo[q] = p.wl >= 0 ? (int)max64(0, diag - p.wl) : 0;
                        st.hi[q] = p.wr >= 0 ? (int)max64(-1, min64((int64_t)it.sk - 1, diag + p.wr)) : it.sk - 1;
                        if (ALIBI) {
                            st.dg[q] = (int)diag;
                            st.ab[q] = p.alibi[hk * p.G + gi[q]] * kLog2e;
                        }
                    }
                    st.m[q] = -INFINITY;
                    st.l[q] = 0.f;
                }
            };
            TileRows rows_a, rows_b;
            init_rows(0, rows_a);
            init_rows(1, rows_b);

            // One key tile of one query tile: S -> running max -> (rare) O rescale -> P.
            auto step = [&](int x, TileRows& st, int j) -> bool {
                const int kt = it.kt0 + j * 128;
                const int sc = (x ? sb : sa) + j;
                if (!__all_sync(0xffffffffu, wait_bar(&s_full[x], sc & 1, abort_flag, p.err, p.wait_ns))) return false;
                tc::fence_after_sync();
                const uint32_t s_addr = tmem + lane_addr + (x ? C::T_S1 : C::T_S0);
                const uint32_t o_addr = tmem + lane_addr + (x ? C::T_O1 : C::T_O0);
                float sv[64];
                tc::ld_16x256b_x8(s_addr, *reinterpret_cast<float(*)[32]>(&sv[0]));
                tc::ld_16x256b_x8(s_addr + 64, *reinterpret_cast<float(*)[32]>(&sv[32]));
                if (warp == 4 && lane == 0) {
                    const uint32_t nrel = it.has_b ? 1u : 2u;
                    mbar_arrive_n(&k_empty[(gk + j) % C::KS], nrel);
                    if (j > 0) mbar_arrive_n(&v_empty[(gv + j - 1) % C::VS], nrel);
                }
                tc::wait_ld();
                if (!(kt >= max(st.lo[0], st.lo[1]) && kt + 127 <= min(st.hi[0], st.hi[1]))) {
#pragma unroll
                    for (int kk = 0; kk < 16; ++kk)
#pragma unroll
                        for (int q = 0; q < 2; ++q)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int key = kt + 8 * kk + 2 * tig + e;
                                float& v = sv[4 * kk + 2 * q + e];
                                v = (key >= st.lo[q] && key <= st.hi[q]) ? v : -INFINITY;
                            }
                }
                float sl = p.scale_log2;
                if (ALIBI) {
                    if (p.wr == 0) {  // causal: the bias is linear in the key left of the diagonal
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const float base = st.ab[q] * (float)(kt + 2 * tig - st.dg[q]);
#pragma unroll
                            for (int kk = 0; kk < 16; ++kk) {
                                float b0, b1;
                                ffma2(b0, b1, st.ab[q], st.ab[q], (float)(8 * kk), (float)(8 * kk + 1), base, base);
                                float& v0 = sv[4 * kk + 2 * q];
                                float& v1 = sv[4 * kk + 2 * q + 1];
                                ffma2(v0, v1, v0, v1, sl, sl, b0, b1);
                            }
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const float d0 = (float)(st.dg[q] - kt - 2 * tig);
#pragma unroll
                            for (int kk = 0; kk < 16; ++kk)
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    float& v = sv[4 * kk + 2 * q + e];
                                    v = fmaf(-st.ab[q], fabsf(d0 - (float)(8 * kk + e)), v * sl);
                                }
                        }
                    }
                    sl = 1.f;
                }
                float lm[2];
                bool grow = false;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float c0 = fmaxf(sv[2 * q], sv[2 * q + 1]), c1 = fmaxf(sv[4 + 2 * q], sv[5 + 2 * q]);
#pragma unroll
                    for (int kk = 2; kk < 16; kk += 2) {
                        c0 = max3f(c0, sv[4 * kk + 2 * q], sv[4 * kk + 2 * q + 1]);
                        c1 = max3f(c1, sv[4 * kk + 4 + 2 * q], sv[4 * kk + 5 + 2 * q]);
                    }
                    lm[q] = fmaxf(c0, c1);
                    grow |= lm[q] * sl > st.m[q] + 8.f;
                }
                float alpha[2] = {1.f, 1.f};
                if (__any_sync(0xffffffffu, grow)) {
                    bool resc = false;
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        float mx = lm[q];
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                        const float m_cand = mx * sl;
                        if (m_cand > st.m[q] + 8.f) {
                            alpha[q] = fast_exp2(st.m[q] - m_cand);
                            st.m[q] = m_cand;
                            resc = true;
                        }
                    }
                    // O_x's last P.V (PV_x(j-1)) precedes S_x(j) on its issuer: complete now
                    if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
                        for (int cc = 0; cc < DP / 64; ++cc) {
                            float o[32];
                            tc::ld_16x256b_x8(o_addr + cc * 64, o);
                            tc::wait_ld();
                            uint32_t ob[32];
#pragma unroll
                            for (int e = 0; e < 32; ++e) ob[e] = __float_as_uint(o[e] * alpha[(e >> 1) & 1]);
                            tc::st_16x256b_x8(o_addr + cc * 64, ob);
                        }
                    }
                }
                float nm[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) nm[q] = st.m[q] == -INFINITY ? 0.f : -st.m[q];
                float sums[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t pk[32];
#pragma unroll
                for (int kk = 0; kk < 16; ++kk)
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        float x0, x1;
                        ffma2(x0, x1, sv[4 * kk + 2 * q], sv[4 * kk + 2 * q + 1], sl, sl, nm[q], nm[q]);
                        const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                        fadd2_acc(sums[2 * q], sums[2 * q + 1], p0, p1);
                        pk[2 * kk + q] = pack2<T>(p0, p1);
                    }
#pragma unroll
                for (int q = 0; q < 2; ++q) st.l[q] = st.l[q] * alpha[q] + (sums[2 * q] + sums[2 * q + 1]);
                tc::st_16x128b_x16(s_addr, pk);
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[x]);
                return true;
            };

            auto epilogue = [&](int x, TileRows& st) -> bool {
                if (!__all_sync(0xffffffffu,
                                wait_bar(&pv_done[x], (x ? ab_ : aa) & 1, abort_flag, p.err, p.wait_ns)))
                    return false;
                tc::fence_after_sync();
                // P.V of the item's last key tile has completed: its V stage is free
                if (warp == 4 && lane == 0) mbar_arrive_n(&v_empty[(gv + n - 1) % C::VS], it.has_b ? 1u : 2u);
                const uint32_t o_addr = tmem + lane_addr + (x ? C::T_O1 : C::T_O0);
                float inv[2];
                T* orow[2];
                bool valid[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float l = st.l[q];
                    l += __shfl_xor_sync(0xffffffffu, l, 1);
                    l += __shfl_xor_sync(0xffffffffu, l, 2);
                    inv[q] = l > 0.f ? 1.f / l : 0.f;
                    valid[q] = live(x, q);
                    const int64_t t = it.q0 + qrow(x, q);
                    const int h = hk * p.G + gi[q];
                    orow[q] = out + t * p.o_s0 + (int64_t)h * p.o_s1;
                    if (valid[q] && tig == 0)
                        p.lse[(int64_t)h * p.lse_s0 + t + (int64_t)b * p.lse_sb] =
                            l > 0.f ? (st.m[q] + log2f(l)) * 0.69314718055994531f : -INFINITY;
                }
                // O[row][8k + 2 tig + {0,1}] sits in thread tig of the row's quad; a 4 x 4
                // transpose over the quad gives thread tig the eight columns of groups tig and
                // tig + 4 of each 64-column chunk, written as two 16-byte stores (a warp's store
                // then covers 64 contiguous bytes of each of its eight rows instead of 16)
#pragma unroll 1
                for (int cc = 0; cc < DP / 64; ++cc) {
                    float o[32];
                    tc::ld_16x256b_x8(o_addr + cc * 64, o);
                    tc::wait_ld();
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        uint32_t w[8];
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            w[kk] = pack2<T>(o[4 * kk + 2 * q] * inv[q], o[4 * kk + 2 * q + 1] * inv[q]);
                        quad_transpose(*reinterpret_cast<uint32_t(*)[4]>(&w[0]), tig);
                        quad_transpose(*reinterpret_cast<uint32_t(*)[4]>(&w[4]), tig);
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const int d = cc * 64 + 32 * hf + 8 * tig;
                            if (valid[q] && d < p.D)
                                *reinterpret_cast<uint4*>(orow[q] + d) =
                                    make_uint4(w[4 * hf], w[4 * hf + 1], w[4 * hf + 2], w[4 * hf + 3]);
                        }
                    }
                }
                // this warp's reads of O_x are complete before its next arrival on p_full[x]
                tc::fence_before_sync();
                return true;
            };

            for (int j = 0; ok && j < n; ++j) {
                ok = step(0, rows_a, j);
                if (ok && it.has_b) ok = step(1, rows_b, j);
            }
            if (ok) ok = epilogue(0, rows_a);
            if (ok && it.has_b) ok = epilogue(1, rows_b);
            sa += n;
            ++aa;
            if (it.has_b) {
                sb += n;
                ++ab_;
            }
            gk += n;
            gv += n;
        }
        tc::fence_before_sync();
    }
    }
    __syncwarp();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// Tile shape of prefill256_kernel.  DP: padded head dim, NT: keys per K/V tile (the width of
// an S buffer), NSB: S buffers, KS / VS: K and V ring stages.
template <int DP_, int NT_, int NSB_, int KS_, int VS_>
struct P2Cfg {
    static constexpr int DP = DP_, CH = DP / 64, NT = NT_, NSB = NSB_;
    static constexpr int Q_TILE = CH * 128 * 128;  // one 128-row q tile
    static constexpr int KV_TILE = CH * NT * 128;  // NT keys x DP columns
    static constexpr int KS = KS_, VS = VS_;
    static_assert(NSB * NT + DP <= 512, "TMEM columns");
};
using P2Cfg256 = P2Cfg<256, 64, 4, 3, 2>;

// Issues the K (or V) boxes of the CTA's NT-key tile number `j` (first key kt0 + NT j) into
// `dst` (chunk-major: 64-column chunk c holds rows [NT c, NT c + NT) of 128 bytes).
template <int NT, int CH>
__device__ __forceinline__ void issue_kv_tile_nt(const PrefillParams& p, const CUtensorMap* map, uint8_t* dst,
                                                 uint64_t* bar, const int* ids, int j, int hk, int kt0, int k0) {
    constexpr int MB = NT / 32;  // most boxes a tile takes (32-row boxes)
    const int kt = kt0 + j * NT;
    int blk[MB];
    uint32_t bytes = 0;
#pragma unroll
    for (int jj = 0; jj < MB; ++jj) {
        blk[jj] = jj < p.boxes_per_tile ? ids[j * p.boxes_per_tile + jj] : -1;
        if (blk[jj] >= 0) bytes += (uint32_t)(CH * p.box_rows * 128);
    }
    mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
    for (int jj = 0; jj < MB; ++jj) {
        if (blk[jj] < 0) continue;
        const int key = kt + jj * p.box_rows;
        const int c2 = p.paged ? key - (key / p.P) * p.P : k0 + key;
        const int c3 = p.paged ? blk[jj] : 0;
        for (int c = 0; c < CH; ++c)
            tma_load_4d(dst + (c * NT + jj * p.box_rows) * 128, map, bar, c * 64, hk, c2, c3, 0ull);
    }
}
// ---------------------------------------------------------------------------------------------
// prefill256_kernel: head_dim 129..256, items of one 128-row query tile.
//
// Two query tiles whose O takes 256 columns each would need more than the 512 TMEM columns,
// and 128-key K/V stages (64 KB each) do not fit twice beside a 64 KB q tile in shared
// memory.  So an item is one query tile of one (sequence, kv head) (q by TMA into shared
// memory, 64 KB); K and V come in 64-key tiles (32 KB) through a 3-deep K ring and a 2-deep
// V ring.  S is quadruple-buffered over consecutive key tiles (64 columns each), so the
// Q.K^T issuer (warp 1) runs up to three tiles ahead of the softmax while the pipe also
// computes P.V (warp 3).  TMEM columns: S0..S3 [0,256), O [256,512).  (With two S buffers the
// chain P.V(j) -> Q.K^T(j+2) -> softmax(j+2) bounded the kernel at ~1,950 cycles a tile.)  A
// 128x64x16 product keeps the tensor pipe ~32 cycles and costs its issuing thread about twice
// that, so one thread issuing both products of a tile bounded the kernel; two issuers share
// the work.  The P.V issuer commits PV(g) to buf_free[g % 4]; the Q.K^T issuer waits for it
// before S(g+4) reuses the columns P(g) was read from, and the softmax waits for PV(g-1)
// there before it hands over P(g) -- only then may it rescale O -- and releases V stage g-1.
// Each waiter takes a buffer's phases in order, and the next phase of a buffer needs work the
// waiter has not yet released, so no wait can see a barrier two phases ahead.  The softmax
// releases K stage g once S(g) is complete.  g counts the CTA's key tiles over its items.
// The same structure at head_dim 128 (three 128-column S buffers) ran no faster than
// prefill_kernel: one query tile per K/V tile doubles the L2 -> shared memory traffic, and
// with every SM in its steady state the L2 delivered ~9 TB/s, ~2,100 cycles a tile against
// ~1,540 with fewer SMs loading.  Between items:
//   * warp 0 takes the next item one claim ahead (atomic add, then a scan of cu_seqlens_q)
//     and publishes its description in one of two slots (item_ready / item_free);
//   * the next q tile is loaded once the Q.K^T issuer has committed q_free after the last
//     S of the item that read it; the next item's first S go into the S buffers the item's
//     last P.V does not read, while the softmax writes out O;
//   * the first P.V of an item (which overwrites O) waits for P(0), which the softmax hands
//     over only after it has read O of the previous item;
//   * the V stage of an item's last key tile is released by the softmax after the last P.V.
template <int DP>
struct PtCfg {
    static_assert(DP == 256, "instantiated for head dim 129..256");
    using B = P2Cfg256;
    static constexpr int CH = B::CH, NT = B::NT, NSB = B::NSB, KS = B::KS, VS = B::VS;
    static constexpr int Q_TILE = B::Q_TILE, KV_TILE = B::KV_TILE;
    static constexpr int OFF_Q = 0, OFF_K = Q_TILE, OFF_V = OFF_K + KS * KV_TILE, OFF_BAR = OFF_V + VS * KV_TILE;
    // q_full, q_free, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], s_full[NSB],
    // p_full[NSB], buf_free[NSB], drain[2], item_ready[2], item_free[2]
    static constexpr int NBAR = 2 + 2 * KS + 2 * VS + 3 * NSB + 6;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem base, abort flag
    static constexpr int OFF_SLOT = OFF_MISC + 16;       // two item slots
    static constexpr int OFF_IDS = OFF_SLOT + 128;       // block-id windows of the K and V producers
    static constexpr int WIN = 128;                      // boxes per window
    static constexpr int SMEM = OFF_IDS + 2 * WIN * 4 + 1024;
    static constexpr uint32_t T_S = 0, T_O = NSB * NT;  // S buffer x at T_S + NT x
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

// Item of the single-tile kernel: query tile u (queries u qpt ..) of sequence b.
__device__ __forceinline__ void pt_item(const PrefillParams& p, int qpt, int nt, PfItem& it) {
    it.q0 = p.cu_q[it.b];
    const int q1 = p.cu_q[it.b + 1];
    it.k0 = p.cu_k[it.b];
    const int k1 = p.cu_k[it.b + 1];
    it.sq = q1 - it.q0;
    it.sk = k1 - it.k0;
    it.bad = it.sq < 0 || it.sk < 0 || it.sq > p.max_sq || it.sk > p.max_sk || it.q0 < 0 || q1 > p.total_q ||
             (!p.paged && (it.k0 < 0 || k1 > p.num_blocks));
    it.n_tiles = 0;
    it.has_b = 0;
    if (it.bad) return;
    it.i0 = it.u * qpt;
    const int i_last = min(it.sq - 1, it.i0 + qpt - 1);
    const int64_t cdiag = (int64_t)it.sk - it.sq;
    const int64_t lo = p.wl >= 0 ? max64(0, it.i0 + cdiag - p.wl) : 0;
    const int64_t hi = p.wr >= 0 ? min64((int64_t)it.sk - 1, i_last + cdiag + p.wr) : (int64_t)it.sk - 1;
    it.kt0 = hi >= lo ? (int)(lo & ~int64_t(nt - 1)) : 0;
    it.n_tiles = hi >= lo ? (int)((hi - it.kt0) / nt + 1) : 0;
}

template <typename T, int DP, bool ALIBI>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    prefill256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
    using C = PtCfg<DP>;
    constexpr int NT = C::NT, NSB = C::NSB, KS = C::KS, VS = C::VS;
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* q_full = bars;
    uint64_t* q_free = bars + 1;
    uint64_t* k_full = bars + 2;
    uint64_t* k_empty = k_full + KS;
    uint64_t* v_full = k_empty + KS;
    uint64_t* v_empty = v_full + VS;
    uint64_t* s_full = v_empty + VS;      // [S buffer]
    uint64_t* p_full = s_full + NSB;      // [S buffer]
    uint64_t* buf_free = p_full + NSB;    // [S buffer]: the P.V that read it has completed
    uint64_t* drain = buf_free + NSB;     // [issuer]
    uint64_t* item_ready = drain + 2;     // [slot]
    uint64_t* item_free = item_ready + 2; // [slot]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile uint32_t* abort_flag = tmem_slot + 1;
    PfItem* slots = reinterpret_cast<PfItem*>(smem + C::OFF_SLOT);
    if (tid == 64) {
        mbar_init(q_full, 1);
        mbar_init(q_free, 1);
        for (int s = 0; s < KS; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < VS; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int x = 0; x < NSB; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], 8);  // one arrive per softmax warp
            mbar_init(&buf_free[x], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&drain[x], 1);
            mbar_init(&item_ready[x], 1);
            mbar_init(&item_free[x], 11);  // the V producer, two issuers, eight softmax warps
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int qpt = 128 / p.G;    // whole queries per tile
    const int trows = qpt * p.G;  // rows of the tile that hold queries (the rest are padding)
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
        const bool r = __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, p.err, p.wait_ns));
        tc::fence_after_sync();
        return r;
    };
    // item k of this CTA, from slot k % 2 (b < 0: no more items)
    auto take_slot = [&](int k, PfItem& it) -> bool {
        if (!wait_all(&item_ready[k & 1], (k >> 1) & 1)) return false;
        it = slots[k & 1];
        __syncwarp();
        if (lane == 0) mbar_arrive(&item_free[k & 1]);
        return true;
    };
    // first key of the item's key tile j (taken in increasing order; the reverse order,
    // diagonal first, measured 3 % slower)
    auto key_tile = [&](const PfItem& it, int j) { return it.kt0 + j * NT; };
    // Issues the item's key tiles into a K or V ring (lane 0 issues); the whole warp stages
    // the block ids of up to C::WIN boxes at a time.  Returns false on an abort.
    auto produce = [&](const PfItem& it, const CUtensorMap* map, uint8_t* ring, uint64_t* fullb, uint64_t* emptyb,
                       int stages, int g0, int* win) -> bool {
        const int32_t* bt_row = p.paged ? p.bt + (int64_t)it.b * p.bt_s0 : nullptr;
        const int bpt = p.boxes_per_tile, win_tiles = C::WIN / bpt;
        int jw = -win_tiles;  // first tile (in processing order) of the staged window
        for (int j = 0; j < it.n_tiles; ++j) {
            if (j >= jw + win_tiles) {  // stage the window that starts at tile j
                jw = j;
                __syncwarp();
                const int n_boxes = min((it.n_tiles - j) * bpt, C::WIN);
                for (int bi = lane; bi < n_boxes; bi += 32) {
                    const int jt = bi / bpt;
                    const int key = key_tile(it, j + jt) + (bi - jt * bpt) * p.box_rows;
                    win[bi] = p.paged ? box_block(bt_row, p.bt_cols, p.num_blocks, p.P, key, it.sk, p.err)
                                      : (key < it.sk ? 0 : -1);
                }
                __syncwarp();
            }
            const int g = g0 + j, s = g % stages;
            if (g >= stages && !wait_all(&emptyb[s], ((g / stages) - 1) & 1)) return false;
            if (lane == 0)
                issue_kv_tile_nt<NT, C::CH>(p, map, ring + s * C::KV_TILE, &fullb[s], win + (j - jw) * bpt, 0, it.hk,
                                            key_tile(it, j), it.k0);
        }
        return true;
    };

    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
    if (warp == 0) {
        // ---------------- item taker, q and K producer ----------------
        // Items: w = tile * Hkv + kv head over the tiles of prefill-class sequences, sequence
        // by sequence, each sequence's last tile first; a tile index past the list ends it.
        const int total = p.pairs * p.Hkv;
        int* win = reinterpret_cast<int*>(smem + C::OFF_IDS);
        if (!p.withhold) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
        }
        int w_next = lane == 0 ? atomicAdd(p.counter, 1) : 0;
        int ld = 0, gk = 0;  // items with loads so far, K tiles issued so far
        for (int k = 0;; ++k) {
            const int w = __shfl_sync(0xffffffffu, w_next, 0);
            PfItem it{};
            it.b = -1;
            if (w < total) {
                const int tile = w / p.Hkv;
                it.hk = w - tile * p.Hkv;
                int remaining = tile;
                for (int base = 0; base < p.batch && it.b < 0; base += 32) {
                    const int bb = base + lane;
                    int tiles = 0;
                    if (bb < p.batch) {
                        const int sqb = p.cu_q[bb + 1] - p.cu_q[bb];
                        tiles = (int64_t)sqb * p.G > p.rows_cap ? (sqb + qpt - 1) / qpt : 0;
                    }
                    int incl = tiles;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const int v = __shfl_up_sync(0xffffffffu, incl, off);
                        if (lane >= off) incl += v;
                    }
                    const unsigned hit = __ballot_sync(0xffffffffu, remaining < incl);
                    if (hit) {
                        const int src = __ffs(hit) - 1;
                        const int excl = __shfl_sync(0xffffffffu, incl - tiles, src);
                        const int cnt = __shfl_sync(0xffffffffu, tiles, src);
                        it.b = base + src;
                        it.u = cnt - 1 - (remaining - excl);
                    } else {
                        remaining -= __shfl_sync(0xffffffffu, incl, 31);
                    }
                }
                if (it.b >= 0) pt_item(p, qpt, NT, it);
            }
            // the next claim's latency overlaps this item's loads
            if (it.b >= 0 && lane == 0) w_next = atomicAdd(p.counter, 1);
            if (k >= 2 && !wait_all(&item_free[k & 1], ((k >> 1) - 1) & 1)) break;
            if (lane == 0) {
                slots[k & 1] = it;
                mbar_arrive(&item_ready[k & 1]);  // release: the slot's stores precede the arrive
            }
            if (it.b < 0) break;  // past the last tile: so is every later item
            if (it.bad) {
                if (lane == 0) flag_error(p.err, PA_ERR_DEVICE_BOUNDS);
                continue;
            }
            if (it.n_tiles == 0) continue;
            // the q tile, once the previous item's last Q.K^T has completed
            if (ld >= 1 && !wait_all(q_free, (ld - 1) & 1)) break;
            if (lane == 0 && !p.withhold) {
                mbar_arrive_expect_tx(q_full, C::CH * trows * 128);
                for (int c = 0; c < C::CH; ++c)
                    tma_load_4d(smem + C::OFF_Q + c * 128 * 128, &tm_q, q_full, c * 64, it.hk * p.G, it.q0 + it.i0,
                                0, 0ull);
            }
            if (!p.withhold && !produce(it, &tm_k, smem + C::OFF_K, k_full, k_empty, KS, gk, win)) break;
            gk += it.n_tiles;
            ++ld;
        }
    } else if (warp == 2) {
        // ---------------- V producer ----------------
        int* win = reinterpret_cast<int*>(smem + C::OFF_IDS) + C::WIN;
        if (!p.withhold) prefetch_tmap(&tm_v);
        int gv = 0;
        for (int k = 0;; ++k) {
            PfItem it;
            if (!take_slot(k, it) || it.b < 0) break;
            if (it.bad || it.n_tiles == 0) continue;
            if (!p.withhold && !produce(it, &tm_v, smem + C::OFF_V, v_full, v_empty, VS, gv, win)) break;
            gv += it.n_tiles;
        }
    } else if (warp == 1) {
        // ---------------- Q.K^T issuer: S(g) into S buffer g % NSB ----------------
        constexpr uint32_t IDESC_S = tc::idesc_f16(128, NT, kBF16, false, false);
        const uint64_t da = tc::smem_desc_sw128(smem_addr(smem + C::OFF_Q), 16, 1024);
        const uint64_t dk0 = tc::smem_desc_sw128(smem_addr(smem + C::OFF_K), 16, 1024);
        int lq = 0, gk = 0, gs = 0;  // items with loads, K ring position, S sequence number
        bool ok = true;
        for (int k = 0; ok; ++k) {
            PfItem it;
            if (!take_slot(k, it) || it.b < 0) break;
            if (it.bad || it.n_tiles == 0) continue;
            const int n = it.n_tiles;
            if (!(ok = wait_all(q_full, lq & 1))) break;
            for (int j = 0; ok && j < n; ++j) {
                const int g = gs + j, x = g % NSB;
                // the S buffer's previous P has been read by its P.V
                if (g >= NSB && !(ok = wait_all(&buf_free[x], ((g / NSB) - 1) & 1))) break;
                const int gkj = gk + j;
                if (!(ok = wait_all(&k_full[gkj % KS], (gkj / KS) & 1))) break;
                {  // the whole warp, one elected lane issuing
                    const uint64_t db = dk0 + (uint64_t)((gkj % KS) * (C::KV_TILE >> 4));
                    const uint32_t d_s = tmem + C::T_S + NT * x;
#pragma unroll
                    for (int kk = 0; kk < DP / 16; ++kk) {
                        const uint64_t oa = (uint64_t)((kk >> 2) * (128 * 128 / 16) + (kk & 3) * 2);
                        const uint64_t ob = (uint64_t)((kk >> 2) * (NT * 128 / 16) + (kk & 3) * 2);
                        tc::mma_ss_elect(d_s, da + oa, db + ob, IDESC_S, kk > 0 ? 1u : 0u);
                    }
                    tc::commit_elect(&s_full[x]);
                    if (j + 1 == n) tc::commit_elect(q_free);  // the item's last read of the q tile
                }
                __syncwarp();
            }
            gs += n;
            gk += n;
            ++lq;
        }
        if (lane == 0) {  // every MMA this issuer started has completed before TMEM is released
            tc::commit(&drain[0]);
            mbar_wait(&drain[0], 0, p.wait_ns);  // not cut short by an abort: MMAs may be in flight
        }
        __syncwarp();
    } else {
        // ---------------- P.V issuer: O += P(g) V ----------------
        constexpr uint32_t IDESC_O = tc::idesc_f16(128, DP, kBF16, false, true);
        const uint64_t dv0 = tc::smem_desc_sw128(smem_addr(smem + C::OFF_V), NT * 128, 1024);
        const uint32_t t_o = tmem + C::T_O;
        int gv = 0, gs = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            PfItem it;
            if (!take_slot(k, it) || it.b < 0) break;
            if (it.bad || it.n_tiles == 0) continue;
            const int n = it.n_tiles;
            for (int j = 0; ok && j < n; ++j) {
                const int g = gs + j, gvj = gv + j;
                if (!(ok = wait_all(&v_full[gvj % VS], (gvj / VS) & 1))) break;
                uint8_t* vst = smem + C::OFF_V + (gvj % VS) * C::KV_TILE;
                const int valid = min(NT, it.sk - key_tile(it, j));
                if (valid < NT) {  // keys at or past sk: zero V rows so P = 0 never meets NaN
                    const int zr = NT - valid;
                    for (int idx = lane; idx < C::CH * zr * 8; idx += 32) {
                        const int c = idx / (zr * 8), rem = idx - c * zr * 8;
                        *reinterpret_cast<int4*>(vst + (c * NT + valid + (rem >> 3)) * 128 + ((rem & 7) << 4)) =
                            make_int4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    tc::fence_after_sync();
                }
                if (!(ok = wait_all(&p_full[g % NSB], (g / NSB) & 1))) break;
                {  // the whole warp, one elected lane issuing
                    const uint64_t db = dv0 + (uint64_t)((gvj % VS) * (C::KV_TILE >> 4));
                    const uint32_t a_p = tmem + C::T_S + NT * (g % NSB);
#pragma unroll
                    for (int kk = 0; kk < NT / 16; ++kk)
                        tc::mma_ts_elect(t_o, a_p + kk * 8, db + (uint64_t)(kk * (2048 / 16)), IDESC_O,
                                         kk > 0 ? 1u : (j > 0 ? 1u : 0u));
                    tc::commit_elect(&buf_free[g % NSB]);
                }
                __syncwarp();
            }
            gs += n;
            gv += n;
        }
        if (lane == 0) {
            tc::commit(&drain[1]);
            mbar_wait(&drain[1], 0, p.wait_ns);
        }
        __syncwarp();
    }
    } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    {
        // ---------------- softmax: warps 4..11 ----------------
        // Warp w reaches TMEM lanes 32 (w % 4) .. +31 and takes half hh = (w - 4) / 4 of them:
        // lanes lb .. lb + 15, lb = 32 (w % 4) + 16 hh.  Thread t holds rows lb + t/4 (q = 0)
        // and lb + t/4 + 8 (q = 1); the four threads of a quad split a row's NT keys (keys
        // 8k + 2 (t % 4) + {0, 1}).
        constexpr int NK = NT / 8;  // 8-key groups of a tile
        const int lg = warp & 3, hh = (warp - 4) >> 2;
        const int gid = lane >> 2, tig = lane & 3;
        const int lb = lg * 32 + hh * 16;
        const uint32_t lane_addr = (uint32_t)lb << 16;
        const uint32_t o_addr = tmem + lane_addr + C::T_O;
        T* out = static_cast<T*>(p.out);
        // this thread's rows of a tile: query qi[q] of the tile, head gi[q] of the group
        int qi[2], gi[2];
        bool pad[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int r = lb + gid + 8 * q;
            qi[q] = r / p.G;
            gi[q] = r - qi[q] * p.G;
            pad[q] = r >= trows;
        }
        int gk = 0, gv = 0, gs = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            PfItem it;
            if (!take_slot(k, it) || it.b < 0) break;
            if (it.bad) continue;
            const int b = it.b, hk = it.hk, n = it.n_tiles;
            const int64_t cdiag = (int64_t)it.sk - it.sq;
            if (n == 0) {  // no row of the tile attends any key: out = 0, lse = -inf
                if (warp < 8) {
                    const int r = (warp & 3) * 32 + lane;
                    const int i = it.i0 + r / p.G, g = r - (r / p.G) * p.G;
                    if (r < trows && i < it.sq) {
                        const int64_t t = it.q0 + i;
                        const int h = hk * p.G + g;
                        for (int d = 0; d < p.D; d += 8)
                            *reinterpret_cast<int4*>(out + t * p.o_s0 + (int64_t)h * p.o_s1 + d) =
                                make_int4(0, 0, 0, 0);
                        p.lse[(int64_t)h * p.lse_s0 + t + (int64_t)b * p.lse_sb] = -INFINITY;
                    }
                }
                continue;
            }
            int lo_r[2], hi_r[2], dg_r[2];
            float ab_r[2], m_r[2], l_r[2];
            bool valid[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int i = it.i0 + qi[q];
                valid[q] = !pad[q] && i < it.sq;
                lo_r[q] = 0;
                hi_r[q] = -1;
                dg_r[q] = 0;
                ab_r[q] = 0.f;
                if (valid[q]) {
                    const int64_t diag = i + cdiag;
                    lo_r[q] = p.wl >= 0 ? (int)max64(0, diag - p.wl) : 0;
                    hi_r[q] = p.wr >= 0 ? (int)max64(-1, min64((int64_t)it.sk - 1, diag + p.wr)) : it.sk - 1;
                    if (ALIBI) {
                        dg_r[q] = (int)diag;
                        ab_r[q] = p.alibi[hk * p.G + gi[q]] * kLog2e;
                    }
                }
                m_r[q] = -INFINITY;
                l_r[q] = 0.f;
            }

            // One key tile: S -> running max -> P; O rescaled (rarely) once PV(j-1) is complete.
            auto step = [&](int j) -> bool {
                const int g = gs + j, x = g % NSB;
                const int kt = key_tile(it, j);
                if (!__all_sync(0xffffffffu, wait_bar(&s_full[x], (g / NSB) & 1, abort_flag, p.err, p.wait_ns)))
                    return false;
                tc::fence_after_sync();
                const uint32_t s_addr = tmem + lane_addr + C::T_S + NT * x;
                // sv[4k + 2q + e] = S[row q][key 8k + 2 tig + e]
                float sv[NT / 2];
#pragma unroll
                for (int hf = 0; hf < NT / 64; ++hf)
                    tc::ld_16x256b_x8(s_addr + 64 * hf, *reinterpret_cast<float(*)[32]>(&sv[32 * hf]));
                if (warp == 4 && lane == 0) mbar_arrive(&k_empty[(gk + j) % KS]);  // S(g) complete: K stage free
                tc::wait_ld();
                if (!(kt >= max(lo_r[0], lo_r[1]) && kt + NT - 1 <= min(hi_r[0], hi_r[1]))) {
#pragma unroll
                    for (int kk = 0; kk < NK; ++kk)
#pragma unroll
                        for (int q = 0; q < 2; ++q)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int key = kt + 8 * kk + 2 * tig + e;
                                float& v = sv[4 * kk + 2 * q + e];
                                v = (key >= lo_r[q] && key <= hi_r[q]) ? v : -INFINITY;
                            }
                }
                float sl = p.scale_log2;  // softmax_scale > 0 on this path
                if (ALIBI) {
                    if (p.wr == 0) {  // causal: the bias is linear in the key left of the diagonal
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const float base = ab_r[q] * (float)(kt + 2 * tig - dg_r[q]);
#pragma unroll
                            for (int kk = 0; kk < NK; ++kk) {
                                float b0, b1;
                                ffma2(b0, b1, ab_r[q], ab_r[q], (float)(8 * kk), (float)(8 * kk + 1), base, base);
                                float& v0 = sv[4 * kk + 2 * q];
                                float& v1 = sv[4 * kk + 2 * q + 1];
                                ffma2(v0, v1, v0, v1, sl, sl, b0, b1);
                            }
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const float d0 = (float)(dg_r[q] - kt - 2 * tig);  // distance of key kt + 2 tig
#pragma unroll
                            for (int kk = 0; kk < NK; ++kk)
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    float& v = sv[4 * kk + 2 * q + e];
                                    v = fmaf(-ab_r[q], fabsf(d0 - (float)(8 * kk + e)), v * sl);
                                }
                        }
                    }
                    sl = 1.f;
                }
                // running max with the lazy rescale: exact row maxima and an O rescale only
                // when some row of the warp grew by more than 2^8
                float lm[2];
                bool grow = false;
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float c0 = fmaxf(sv[2 * q], sv[2 * q + 1]), c1 = fmaxf(sv[4 + 2 * q], sv[5 + 2 * q]);
#pragma unroll
                    for (int kk = 2; kk < NK; kk += 2) {
                        c0 = max3f(c0, sv[4 * kk + 2 * q], sv[4 * kk + 2 * q + 1]);
                        c1 = max3f(c1, sv[4 * kk + 4 + 2 * q], sv[4 * kk + 5 + 2 * q]);
                    }
                    lm[q] = fmaxf(c0, c1);
                    grow |= lm[q] * sl > m_r[q] + 8.f;
                }
                float alpha[2] = {1.f, 1.f};
                bool resc = false;
                if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        float mx = lm[q];
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                        const float m_cand = mx * sl;
                        if (m_cand > m_r[q] + 8.f) {
                            alpha[q] = fast_exp2(m_r[q] - m_cand);
                            m_r[q] = m_cand;
                            resc = true;
                        }
                    }
                }
                float nm[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) nm[q] = m_r[q] == -INFINITY ? 0.f : -m_r[q];
                float sums[4] = {0.f, 0.f, 0.f, 0.f};
                // pk[2k + q] = P[row q][packed column 4k + tig] = (keys 8k + 2 tig, +1)
                uint32_t pk[NK * 2];
#pragma unroll
                for (int kk = 0; kk < NK; ++kk)
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        float x0, x1;
                        ffma2(x0, x1, sv[4 * kk + 2 * q], sv[4 * kk + 2 * q + 1], sl, sl, nm[q], nm[q]);
                        const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                        fadd2_acc(sums[2 * q], sums[2 * q + 1], p0, p1);
                        pk[2 * kk + q] = pack2<T>(p0, p1);
                    }
#pragma unroll
                for (int q = 0; q < 2; ++q) l_r[q] = l_r[q] * alpha[q] + (sums[2 * q] + sums[2 * q + 1]);
                if (j > 0) {
                    // PV(g-1) complete: O holds every earlier tile, V stage j-1 is free
                    if (!__all_sync(0xffffffffu, wait_bar(&buf_free[(g - 1) % NSB], ((g - 1) / NSB) & 1, abort_flag,
                                                          p.err, p.wait_ns)))
                        return false;
                    tc::fence_after_sync();
                    if (warp == 4 && lane == 0) mbar_arrive(&v_empty[(gv + j - 1) % VS]);
                    if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
                        for (int cc = 0; cc < DP / 64; ++cc) {
                            float o[32];
                            tc::ld_16x256b_x8(o_addr + cc * 64, o);
                            tc::wait_ld();
                            uint32_t ob[32];
#pragma unroll
                            for (int e = 0; e < 32; ++e) ob[e] = __float_as_uint(o[e] * alpha[(e >> 1) & 1]);
                            tc::st_16x256b_x8(o_addr + cc * 64, ob);
                        }
                    }
                }
                // P overwrites the first NT / 2 columns of the S it came from (this thread's cells)
                if constexpr (NT == 64)
                    tc::st_16x128b_x8(s_addr, pk);
                else
                    tc::st_16x128b_x16(s_addr, pk);
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[x]);
                return true;
            };

            for (int j = 0; ok && j < n; ++j) ok = step(j);
            const int gl = gs + n - 1;  // the item's last tile
            if (ok) ok = __all_sync(0xffffffffu, wait_bar(&buf_free[gl % NSB], (gl / NSB) & 1, abort_flag, p.err,
                                                          p.wait_ns));
            if (ok) {
                tc::fence_after_sync();
                if (warp == 4 && lane == 0) mbar_arrive(&v_empty[(gv + n - 1) % VS]);  // last P.V complete
                float inv[2];
                T* orow[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float l = l_r[q];
                    l += __shfl_xor_sync(0xffffffffu, l, 1);
                    l += __shfl_xor_sync(0xffffffffu, l, 2);
                    inv[q] = l > 0.f ? 1.f / l : 0.f;
                    const int64_t t = it.q0 + it.i0 + qi[q];
                    const int h = hk * p.G + gi[q];
                    orow[q] = out + t * p.o_s0 + (int64_t)h * p.o_s1;
                    if (valid[q] && tig == 0)
                        p.lse[(int64_t)h * p.lse_s0 + t + (int64_t)b * p.lse_sb] =
                            l > 0.f ? (m_r[q] + log2f(l)) * 0.69314718055994531f : -INFINITY;
                }
                // a 4 x 4 transpose over each quad gives thread tig the eight columns of groups
                // tig and tig + 4 of a 64-column chunk: two 16-byte stores per row and chunk
#pragma unroll 1
                for (int cc = 0; cc < DP / 64; ++cc) {
                    float o[32];
                    tc::ld_16x256b_x8(o_addr + cc * 64, o);
                    tc::wait_ld();
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        uint32_t w[8];
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            w[kk] = pack2<T>(o[4 * kk + 2 * q] * inv[q], o[4 * kk + 2 * q + 1] * inv[q]);
                        quad_transpose(*reinterpret_cast<uint32_t(*)[4]>(&w[0]), tig);
                        quad_transpose(*reinterpret_cast<uint32_t(*)[4]>(&w[4]), tig);
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const int d = cc * 64 + 32 * hf + 8 * tig;
                            if (valid[q] && d < p.D)
                                *reinterpret_cast<uint4*>(orow[q] + d) =
                                    make_uint4(w[4 * hf], w[4 * hf + 1], w[4 * hf + 2], w[4 * hf + 3]);
                        }
                    }
                }
                // this warp's reads of O are complete before its next arrival on p_full
                tc::fence_before_sync();
            }
            gs += n;
            gk += n;
            gv += n;
        }
        tc::fence_before_sync();
    }
    }
    __syncwarp();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}
// Tensor maps: q as (D, H, total_q, 1) with box (64, G, 128 / G, 1); K/V as (D, Hkv, page,
// blocks) with box (64, 1, box_rows, 1) (non-paged: (D, Hkv, keys, 1)).
int prefill_maps(const Args& a, const PrefillParams& pp, CUtensorMap* tq, CUtensorMap* tk, CUtensorMap* tv,
                 char* msg, size_t msg_len) {
    {
        const uint64_t dims[4] = {(uint64_t)a.D, (uint64_t)a.H, (uint64_t)a.total_q, 1};
        const uint64_t strides[3] = {(uint64_t)a.q_s1 * 2, (uint64_t)a.q_s0 * 2, (uint64_t)a.q_s0 * 2 * a.total_q};
        const uint32_t box[4] = {64u, (uint32_t)pp.G, (uint32_t)(128 / pp.G), 1u};
        int rc = encode_tmap_4d(tq, a.dtype, a.q, dims, strides, box, 1, msg, msg_len);
        if (rc != PA_OK) return rc;
    }
    uint64_t dims[4], strides[3];
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
    const uint32_t box[4] = {64u, 1u, (uint32_t)pp.box_rows, 1u};
    int rc = encode_tmap_4d(tk, a.dtype, a.k, dims, strides, box, 1, msg, msg_len);
    if (rc != PA_OK) return rc;
    return encode_tmap_4d(tv, a.dtype, a.v, dims, strides, box, 1, msg, msg_len);
}

// Zeroes the item counter on `stream` and launches one CTA per SM (at most one per item).
// `sms` caches the SM count and doubles as the once-per-instantiation configuration flag.
template <typename Kern>
int launch_persistent(Kern kern, int smem, int& sms, const Args& a, const PrefillParams& pp, const char* name,
                      cudaStream_t stream, char* msg, size_t msg_len) {
    if (!sms) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        int dev = 0, n = 0;
        if (e == cudaSuccess) e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "configuring %s (%d bytes of shared memory): %s", name, smem, cudaGetErrorString(e));
            return PA_ERR_CUDA;
        }
        sms = n;
    }
    CUtensorMap tq, tk, tv;
    int rc = prefill_maps(a, pp, &tq, &tk, &tv, msg, msg_len);
    if (rc != PA_OK) return rc;
    // the kernels count items, and every CTA claims one past the last, in int
    if ((int64_t)pp.pairs * a.Hkv + sms >= (int64_t)INT32_MAX) {
        snprintf(msg, msg_len, "%s: %lld work items (tiles x kv heads) exceed the item counter's range", name,
                 (long long)pp.pairs * a.Hkv);
        return PA_ERR_UNSUPPORTED;
    }
    const int items = pp.pairs * a.Hkv;
    NvtxRange nv(name);
    cudaError_t e = cudaMemsetAsync(pp.counter, 0, sizeof(int), stream);
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "%s: zeroing the item counter: %s", name, cudaGetErrorString(e));
        return PA_ERR_CUDA;
    }
    timer_begin(PA_KC_PREFILL, stream);
    kern<<<std::min(sms, items), kPrefillThreads, smem, stream>>>(tq, tk, tv, pp);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "%s launch: %s", name, cudaGetErrorString(e));
        return PA_ERR_CUDA;
    }
    timer_end(PA_KC_PREFILL, stream);
    count_launches(1);
    return PA_OK;
}

template <typename T, int DP, bool ALIBI>
int run_prefill(const Args& a, const PrefillParams& pp, char* msg, size_t msg_len) {
    static int sms = 0;
    return launch_persistent(prefill_kernel<T, DP, ALIBI>, PfCfg<DP>::SMEM, sms, a, pp, "pa::prefill_kernel", a.stream,
                             msg, msg_len);
}

template <typename T, bool ALIBI>
int run_prefill256(const Args& a, const PrefillParams& pp, char* msg, size_t msg_len) {
    static int sms = 0;
    return launch_persistent(prefill256_kernel<T, 256, ALIBI>, PtCfg<256>::SMEM, sms, a, pp, "pa::prefill256_kernel",
                             a.stream, msg, msg_len);
}

}  // namespace

int prefill_rows_threshold() { return 32; }

bool prefill_supported(const Args& a) {
    static const bool disabled = std::getenv("PA_DISABLE_TC_PREFILL") != nullptr;
    if (disabled) return false;
    const int G = a.H / a.Hkv;
    if (a.D > 256 || G > 128) return false;
    if (!(a.scale > 0.f)) return false;
    if ((int64_t)a.max_sq * G <= prefill_rows_threshold()) return false;  // nothing for it to do
    if (a.total_q <= 0 || a.q_s1 * 2 % 16 != 0 || a.q_s0 * 2 % 16 != 0) return false;
    // a q tensor map needs a 16-byte aligned base: rows of wider heads then take the general kernel
    if (a.D > 128 && reinterpret_cast<uintptr_t>(a.q) % 16 != 0) return false;
    return true;
}

// Upper bound of the prefill kernel's work items per kv head, from the call's sizes alone:
// query tiles (head dim above 128) or tile pairs of 128 / G whole queries each, summed over
// the sequences, is at most ceil(total_q / per item) + batch and at most batch x
// ceil(max_seqlen_q / per item).
static int64_t prefill_items_per_head(const Args& a) {
    const int64_t per = (a.D > 128 ? 1 : 2) * (128 / (a.H / a.Hkv));
    return std::min<int64_t>(((int64_t)a.total_q + per - 1) / per + a.batch,
                             (int64_t)a.batch * (((int64_t)a.max_sq + per - 1) / per));
}

int64_t prefill_items_bound(const Args& a) { return prefill_items_per_head(a) * a.Hkv; }

int launch_prefill(const Args& a, int* counter, unsigned int* err, char* msg, size_t msg_len) {
    if (!counter) {
        snprintf(msg, msg_len, "the prefill kernels need a device item counter");
        return PA_ERR_ARG;
    }
    PrefillParams pp{};
    pp.counter = counter;
    pp.out = a.out;
    pp.o_s0 = a.o_s0;
    pp.o_s1 = a.o_s1;
    pp.lse = a.lse;
    pp.lse_s0 = a.lse_s0;
    pp.lse_sb = a.lse_sb;
    pp.cu_q = a.cu_q;
    pp.cu_k = a.cu_k;
    pp.bt = a.block_table;
    pp.bt_s0 = a.bt_s0;
    pp.bt_cols = a.bt_cols;
    pp.batch = a.batch;
    pp.H = a.H;
    pp.Hkv = a.Hkv;
    pp.G = a.H / a.Hkv;
    pp.D = a.D;
    pp.P = a.paged ? a.page : 1;
    pp.num_blocks = a.num_blocks;
    pp.total_q = a.total_q;
    pp.paged = a.paged ? 1 : 0;
    pp.max_sq = a.max_sq;
    pp.max_sk = a.max_sk;
    pp.scale_log2 = a.scale * 1.4426950408889634f;
    pp.alibi = a.alibi;
    pp.wl = a.wl;
    pp.wr = a.wr;
    pp.rows_cap = prefill_rows_threshold();
    pp.err = err;
    pp.wait_ns = a.wait_ns;
    pp.withhold = a.withhold_loads;
    const bool alibi = a.alibi != nullptr;
    if (a.D > 128) {  // items of one query tile, 64-key K/V tiles
        pp.box_rows = a.paged ? (a.page % 64 == 0 ? 64 : 32) : 64;
        pp.boxes_per_tile = 64 / pp.box_rows;
        pp.pairs = (int)prefill_items_per_head(a);  // query tiles
        if (a.dtype == PA_BF16)
            return alibi ? run_prefill256<__nv_bfloat16, true>(a, pp, msg, msg_len)
                         : run_prefill256<__nv_bfloat16, false>(a, pp, msg, msg_len);
        return alibi ? run_prefill256<__half, true>(a, pp, msg, msg_len) : run_prefill256<__half, false>(a, pp, msg, msg_len);
    }
    // items of two query tiles, 128-key K/V tiles
    pp.box_rows = a.paged ? ((a.page % 128 == 0) ? 128 : (a.page % 64 == 0) ? 64 : 32) : 128;
    pp.boxes_per_tile = 128 / pp.box_rows;
    pp.pairs = (int)prefill_items_per_head(a);  // tile pairs (2 qpt queries each)
    const int dp = a.D <= 64 ? 64 : 128;
    if (a.dtype == PA_BF16) {
        if (alibi)
            return dp == 64 ? run_prefill<__nv_bfloat16, 64, true>(a, pp, msg, msg_len)
                            : run_prefill<__nv_bfloat16, 128, true>(a, pp, msg, msg_len);
        return dp == 64 ? run_prefill<__nv_bfloat16, 64, false>(a, pp, msg, msg_len)
                        : run_prefill<__nv_bfloat16, 128, false>(a, pp, msg, msg_len);
    }
    if (alibi)
        return dp == 64 ? run_prefill<__half, 64, true>(a, pp, msg, msg_len)
                        : run_prefill<__half, 128, true>(a, pp, msg, msg_len);
    return dp == 64 ? run_prefill<__half, 64, false>(a, pp, msg, msg_len)
                    : run_prefill<__half, 128, false>(a, pp, msg, msg_len);
}

}  // namespace pa
