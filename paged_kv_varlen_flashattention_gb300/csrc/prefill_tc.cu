// Tensor-core prefill / chunked-prefill kernel for paged varlen attention (sm_103a).
//
// One CTA owns two 128-row query tiles (A and B, consecutive) of one (sequence, kv head);
// a tile's rows are the (query i, head g) pairs of the kv head's GQA group, ordered
// i * G + g, so each K/V tile feeds all G query heads and both query tiles.  A tile holds
// floor(128 / G) whole queries; when G does not divide 128 its last 128 mod G rows are
// padding (masked, never written).
// Roles (384 threads, three warpgroups):
//   warps 0, 2  TMA producers (warp 0: both q tiles once, then K tiles; warp 2: V tiles),
//               128 keys per tile through the block table (one box per page piece; the
//               paged layout of "flash-attn-varlen paged expects k/v tensors of rank 4",
//               What it means), each blocking on its own ring's empty barriers
//   warps 1, 3  MMA issuers for tiles A and B (one elected lane each; warp 1 also owns the
//               tensor memory):
//               S_X = Q_X K_j^T  (tcgen05.mma, A and B from shared memory, S in TMEM)
//               O_X += P_X V_j   (tcgen05.mma, A = P from TMEM, B = V from shared memory)
//   warps 4..11 softmax, all eight on tile A and then on tile B at every key tile: each
//               warp owns 16 rows (TMEM lanes), four threads per row; reads S from TMEM,
//               masks, keeps the running max and sum, writes P (16-bit) over the columns of
//               S it came from, and rescales O in TMEM only when the running max grew by
//               more than 2^8 (otherwise the stale max stays: exact after the final division).
// The two tiles ping-pong: while the softmax works on one tile, the tensor pipe runs the
// other tile's P.V and next Q.K^T.  TMEM columns: S_A [0,128), S_B [128,256),
// O_A [256, 256+DP), O_B [256+DP, 256+2 DP).
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
    int pairs;  // grid.x: an upper bound of the number of tile pairs
    unsigned int* err;
    uint64_t wait_ns;  // bound on every wait
    int withhold;      // test hook: issue no loads
};

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
    // drain[2]
    static constexpr int NBAR = 1 + 2 * KS + 2 * VS + 8;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem base, abort flag, picked pair
    static constexpr int OFF_IDS = OFF_MISC + 16;         // block id of every TMA box of the CTA
    static constexpr int MAX_BOXES = 256;
    static constexpr int SMEM = OFF_IDS + (MAX_BOXES + 4) * 4 + 1024;
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
    const int hk = blockIdx.y;

    // ---- set-up that does not depend on the work item, overlapped with the scan below:
    // warp 1 allocates tensor memory, warp 2 initialises the barriers.
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* k_empty = k_full + C::KS;
    uint64_t* v_full = k_empty + C::KS;
    uint64_t* v_empty = v_full + C::VS;
    uint64_t* s_full = v_empty + C::VS;  // [tile]
    uint64_t* p_full = s_full + 2;       // [tile]
    uint64_t* pv_done = p_full + 2;      // [tile]: the tile's last P.V has completed
    uint64_t* drain = pv_done + 2;       // [issuer]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile uint32_t* abort_flag = tmem_slot + 1;
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
        }
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }

    // ---- which (sequence, tile pair) this CTA owns: the blockIdx.x-th pair of the list of
    // all pairs of 128-row tiles of prefill-class sequences, sequence by sequence, each
    // sequence's last pair (the longest under a causal mask) first.  Warp 0 scans
    // cu_seqlens_q 32 sequences at a time with a prefix sum of pair counts.
    int* pick = reinterpret_cast<int*>(smem + C::OFF_MISC + 8);
    const int qpt = 128 / p.G;     // whole queries per 128-row tile
    const int trows = qpt * p.G;   // rows of a tile that hold queries (the rest are padding)
    if (warp == 0) {
        int remaining = (int)blockIdx.x, found_b = -1, found_u = 0;
        for (int base = 0; base < p.batch && found_b < 0; base += 32) {
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
                found_b = base + src;
                found_u = cnt - 1 - (remaining - excl);
            } else {
                remaining -= __shfl_sync(0xffffffffu, incl, 31);
            }
        }
        if (lane == 0) {
            pick[0] = found_b;
            pick[1] = found_u;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int b = pick[0], u = pick[1];
    // every early exit below is uniform over the CTA; warp 1 returns the tensor memory
    auto leave = [&]() {
        if (warp == 1) tc::tmem_dealloc(tmem, 512);
    };
    if (b < 0) {  // past the last pair
        leave();
        return;
    }

    // ---- this CTA's work (uniform over the CTA) ----
    const int q0 = p.cu_q[b], q1 = p.cu_q[b + 1];
    const int k0 = p.cu_k[b], k1 = p.cu_k[b + 1];
    const int sq = q1 - q0, sk = k1 - k0;
    if (sq < 0 || sk < 0 || sq > p.max_sq || sk > p.max_sk || q0 < 0 || q1 > p.total_q ||
        (!p.paged && (k0 < 0 || k1 > p.num_blocks))) {
        if (tid == 0) flag_error(p.err, PA_ERR_DEVICE_BOUNDS);
        leave();
        return;
    }
    const int64_t rows_total = (int64_t)sq * p.G;
    const int i0 = u * 2 * qpt;         // first query of tile A
    const bool has_b = i0 + qpt < sq;   // tile B holds at least one query
    // row (i * G + g) of row r of tile x, and whether that row holds a query of the sequence
    auto tile_rho = [&](int x, int r) -> int64_t { return (int64_t)(i0 + x * qpt) * p.G + r; };
    auto row_live = [&](int x, int r) { return r < trows && tile_rho(x, r) < rows_total; };
    const int i_last = min(sq - 1, i0 + (has_b ? 2 : 1) * qpt - 1);
    const int64_t cdiag = (int64_t)sk - sq;
    const int64_t lo = p.wl >= 0 ? max64(0, i0 + cdiag - p.wl) : 0;
    const int64_t hi = p.wr >= 0 ? min64((int64_t)sk - 1, i_last + cdiag + p.wr) : (int64_t)sk - 1;
    const int kt0 = hi >= lo ? (int)(lo & ~int64_t(127)) : 0;
    const int n_tiles = hi >= lo ? (int)((hi - kt0) / 128 + 1) : 0;

    T* out = static_cast<T*>(p.out);
    if (n_tiles == 0) {  // no row of the pair attends any key: out = 0, lse = -inf
        if (warp >= 4) {
            const int x = (warp - 4) >> 2, r = (warp & 3) * 32 + lane;
            const int64_t rho = tile_rho(x, r);
            if (row_live(x, r)) {
                const int i = (int)(rho / p.G), g = (int)(rho - (int64_t)i * p.G);
                const int64_t t = q0 + i;
                const int h = hk * p.G + g;
                for (int d = 0; d < p.D; d += 8)
                    *reinterpret_cast<int4*>(out + t * p.o_s0 + (int64_t)h * p.o_s1 + d) = make_int4(0, 0, 0, 0);
                p.lse[(int64_t)h * p.lse_s0 + t + (int64_t)b * p.lse_sb] = -INFINITY;
            }
        }
        leave();
        return;
    }

    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
    if (warp == 0 || warp == 2) {
        // ---------------- TMA producers: warp 0 loads q and K, warp 2 loads V ----------------
        // Physical block of every box of this CTA's key range, staged once by warp 0.
        int* ids = reinterpret_cast<int*>(smem + C::OFF_IDS);
        const int n_boxes = min(n_tiles * p.boxes_per_tile, C::MAX_BOXES);
        const int32_t* bt_row = p.paged ? p.bt + (int64_t)b * p.bt_s0 : nullptr;
        if (warp == 0) {
            if (lane == 0 && !p.withhold) {  // the q tiles first: their latency overlaps the id lookups
                prefetch_tmap(&tm_q);
                mbar_arrive_expect_tx(q_full, (has_b ? 2 : 1) * C::CH * trows * 128);
                for (int x = 0; x < (has_b ? 2 : 1); ++x)
                    for (int c = 0; c < C::CH; ++c)
                        tma_load_4d(smem + C::OFF_Q + x * C::Q_TILE + c * 128 * 128, &tm_q, q_full, c * 64,
                                    hk * p.G, q0 + i0 + x * qpt, 0, 0ull);
            }
            for (int bi = lane; bi < n_boxes; bi += 32) {
                const int key = kt0 + bi * p.box_rows;
                ids[bi] = p.paged ? box_block(bt_row, p.bt_cols, p.num_blocks, p.P, key, sk, p.err)
                                  : (key < sk ? 0 : -1);
            }
        }
        named_barrier_sync(2, 64);  // warps 0 and 2: the staged ids are visible
        const bool is_k = warp == 0;
        if (lane == 0 && !p.withhold) {
            const CUtensorMap* map = is_k ? &tm_k : &tm_v;
            prefetch_tmap(map);
            const int stages = is_k ? C::KS : C::VS;
            uint64_t* fullb = is_k ? k_full : v_full;
            uint64_t* emptyb = is_k ? k_empty : v_empty;
            uint8_t* ring = smem + (is_k ? C::OFF_K : C::OFF_V);
            int spill[4];  // block ids of one tile past the staged range
            for (int j = 0; j < n_tiles; ++j) {
                const int s = j % stages;
                if (j >= stages && !wait_bar(&emptyb[s], ((j / stages) - 1) & 1, abort_flag, p.err, p.wait_ns))
                    break;
                const int* tile = ids;
                int jt = j, kb = kt0;
                if ((j + 1) * p.boxes_per_tile > C::MAX_BOXES) {
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int key = kt0 + j * 128 + jj * p.box_rows;
                        spill[jj] = jj >= p.boxes_per_tile ? -1
                                    : p.paged ? box_block(bt_row, p.bt_cols, p.num_blocks, p.P, key, sk, p.err)
                                              : (key < sk ? 0 : -1);
                    }
                    tile = spill;
                    jt = 0;
                    kb = kt0 + j * 128;
                }
                issue_kv_tile(p, map, ring + s * C::KV_TILE, &fullb[s], tile, jt, hk, kb, k0, C::CH);
            }
        }
    } else if (warp == 1 || warp == 3) {
        // ---------------- MMA issuers: warp 1 for tile A, warp 3 for tile B ----------------
        // A tcgen05.mma costs its issuing thread ~50 cycles, close to the 64 cycles a
        // 128x128x16 product takes; two issuers keep the pipe fed while each also waits on
        // its tile's barriers.  Per issuer the order is S_x(0), PV_x(0), S_x(1), PV_x(1), ...
        // so S_x(j+1) overwrites the P_x(j) columns only after PV_x(j) (in-order per thread).
        constexpr uint32_t IDESC_S = tc::idesc_f16(128, 128, kBF16, false, false);
        constexpr uint32_t IDESC_O = tc::idesc_f16(128, DP, kBF16, false, true);
        const int x = warp == 1 ? 0 : 1;
        const bool active = x == 0 || has_b;  // without tile B, warp 3 only releases the stages
        // Shared-memory descriptors are built once; the start-address field (address / 16,
        // bits 0..13) then advances by a compile-time constant per MMA.
        const uint64_t da = tc::smem_desc_sw128(smem_addr(smem + C::OFF_Q + x * C::Q_TILE), 16, 1024);
        const uint64_t dk0 = tc::smem_desc_sw128(smem_addr(smem + C::OFF_K), 16, 1024);
        const uint64_t dv0 = tc::smem_desc_sw128(smem_addr(smem + C::OFF_V), 128 * 128, 1024);
        const uint32_t d_s = tmem + (x ? C::T_S1 : C::T_S0);
        const uint32_t d_o = tmem + (x ? C::T_O1 : C::T_O0);
        auto wait_all = [&](uint64_t* bar, uint32_t parity) {
            const bool r = __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, p.err, p.wait_ns));
            tc::fence_after_sync();
            return r;
        };
        // S_x(j) = Q_x K_j^T into S buffer x; releases K stage j once complete
        auto issue_s = [&](int j) {
            if (active) {
                const uint64_t db = dk0 + (uint64_t)((j % C::KS) * (C::KV_TILE >> 4));
#pragma unroll
                for (int kk = 0; kk < DP / 16; ++kk) {
                    const uint64_t off = (uint64_t)((kk >> 2) * (128 * 128 / 16) + (kk & 3) * 2);
                    tc::mma_ss(d_s, da + off, db + off, IDESC_S, kk > 0 ? 1u : 0u);
                }
                tc::commit(&s_full[x]);
            }
        };
        // Stages are released on the softmax side (see there); an issuer without a tile idles.
        bool ok = active && wait_all(q_full, 0);
        if (ok && n_tiles > 0 && (ok = wait_all(&k_full[0], 0))) {
            if (lane == 0) issue_s(0);
            __syncwarp();
        }
        for (int j = 0; ok && j < n_tiles; ++j) {
            // Everything that does not depend on P_x(j) is settled first (V_j and K_{j+1}
            // resident, V_j's rows past the last key zeroed), so that once the softmax hands
            // over P_x(j), PV_x(j) and S_x(j+1) issue back to back.
            if (!(ok = wait_all(&v_full[j % C::VS], (j / C::VS) & 1))) break;
            if (active) {
                uint8_t* vst = smem + C::OFF_V + (j % C::VS) * C::KV_TILE;
                const int valid = min(128, sk - (kt0 + j * 128));
                if (valid < 128) {  // keys at or past sk: zero V rows so P = 0 never meets NaN
                    // (both issuers write the same zeros; each orders its own writes before its MMAs)
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
            }
            const bool more = j + 1 < n_tiles;
            if (more && !(ok = wait_all(&k_full[(j + 1) % C::KS], ((j + 1) / C::KS) & 1))) break;
            // O_x += P_x(j) V_j, P_x read from the columns of S buffer x
            if (active && !(ok = wait_all(&p_full[x], j & 1))) break;
            if (lane == 0) {
                if (active) {
                    const uint64_t db = dv0 + (uint64_t)((j % C::VS) * (C::KV_TILE >> 4));
                    const uint32_t first = j > 0 ? 1u : 0u;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc::mma_ts(d_o, d_s + kk * 8, db + (uint64_t)(kk * (2048 / 16)), IDESC_O, kk > 0 ? 1u : first);
                    if (j + 1 == n_tiles) tc::commit(&pv_done[x]);
                }
                if (more) issue_s(j + 1);
            }
            __syncwarp();
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
        // ---------------- softmax: warps 4..11, tile A then tile B at every key tile ----------------
        // Warp w reaches TMEM lanes 32 (w % 4) .. +31 and takes the half hh = (w - 4) / 4 of
        // them: lanes lb .. lb + 15 with lb = 32 (w % 4) + 16 hh.  Thread t holds rows
        // lb + t/4 (q = 0) and lb + t/4 + 8 (q = 1) of each tile; the four threads of a quad
        // split a row's 128 keys (keys 8k + 2 (t % 4) + {0, 1}, k = 0..15), so row maxima and
        // sums are quad reductions and P lands in the columns its own thread read S from.
        const int lg = warp & 3, hh = (warp - 4) >> 2;
        const int gid = lane >> 2, tig = lane & 3;
        const int lb = lg * 32 + hh * 16;
        const uint32_t lane_addr = (uint32_t)lb << 16;
        struct TileRows {
            int lo[2], hi[2];  // attended key range of each row (empty for padding rows)
            float m[2], l[2];  // running max (log2 domain) and this thread's share of the sum
            int dg[2];         // the row's bottom-right aligned diagonal key (ALIBI)
            float ab[2];       // its bias slope times log2(e) (ALIBI)
        };
        auto init_rows = [&](int x, TileRows& st) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int64_t rho = tile_rho(x, lb + gid + 8 * q);
                st.lo[q] = 0;
                st.hi[q] = -1;
                st.dg[q] = 0;
                st.ab[q] = 0.f;
                if (row_live(x, lb + gid + 8 * q)) {
                    const int64_t diag = rho / p.G + cdiag;
                    st.lo[q] = p.wl >= 0 ? (int)max64(0, diag - p.wl) : 0;
                    st.hi[q] = p.wr >= 0 ? (int)max64(-1, min64((int64_t)sk - 1, diag + p.wr)) : sk - 1;
                    if (ALIBI) {
                        st.dg[q] = (int)diag;
                        st.ab[q] = p.alibi[hk * p.G + (int)(rho - (rho / p.G) * p.G)] * kLog2e;
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
            const int kt = kt0 + j * 128;
            if (!__all_sync(0xffffffffu, wait_bar(&s_full[x], j & 1, abort_flag, p.err, p.wait_ns))) return false;
            tc::fence_after_sync();
            const uint32_t s_addr = tmem + lane_addr + (x ? C::T_S1 : C::T_S0);
            const uint32_t o_addr = tmem + lane_addr + (x ? C::T_O1 : C::T_O0);
            // sv[4k + 2q + e] = S[row q][key 8k + 2 tig + e]
            float sv[64];
            tc::ld_16x256b_x8(s_addr, *reinterpret_cast<float(*)[32]>(&sv[0]));
            tc::ld_16x256b_x8(s_addr + 64, *reinterpret_cast<float(*)[32]>(&sv[32]));
            // S_x(j) is complete, and so is PV_x(j-1), which its issuer started before it: this
            // tile is done with K stage j and V stage j-1.  (Released here, while the TMEM load
            // is in flight, instead of by tcgen05.commit: that spares the issuers two commits
            // per key tile.)
            if (warp == 4 && lane == 0) {
                const uint32_t n = has_b ? 1u : 2u;
                mbar_arrive_n(&k_empty[j % C::KS], n);
                if (j > 0) mbar_arrive_n(&v_empty[(j - 1) % C::VS], n);
            }
            tc::wait_ld();
            if (!(kt >= max(st.lo[0], st.lo[1]) && kt + 127 <= min(st.hi[0], st.hi[1]))) {
#pragma unroll
                for (int k = 0; k < 16; ++k)
#pragma unroll
                    for (int q = 0; q < 2; ++q)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int key = kt + 8 * k + 2 * tig + e;
                            float& v = sv[4 * k + 2 * q + e];
                            v = (key >= st.lo[q] && key <= st.hi[q]) ? v : -INFINITY;
                        }
            }
            // With the position bias, S becomes the biased score in the log2 domain here and
            // the rest runs with a unit scale.
            float sl = p.scale_log2;  // softmax_scale > 0 on this path
            if (ALIBI) {
                if (p.wr == 0) {
                    // causal: every attended key is at or left of the diagonal, where the
                    // bias ab * (key - dg) is linear in the key (masked keys stay -inf)
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const float base = st.ab[q] * (float)(kt + 2 * tig - st.dg[q]);  // key kt + 2 tig
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            float b0, b1;
                            ffma2(b0, b1, st.ab[q], st.ab[q], (float)(8 * k), (float)(8 * k + 1), base, base);
                            float& v0 = sv[4 * k + 2 * q];
                            float& v1 = sv[4 * k + 2 * q + 1];
                            ffma2(v0, v1, v0, v1, sl, sl, b0, b1);
                        }
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const float d0 = (float)(st.dg[q] - kt - 2 * tig);  // distance of key kt + 2 tig
#pragma unroll
                        for (int k = 0; k < 16; ++k)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                float& v = sv[4 * k + 2 * q + e];
                                v = fmaf(-st.ab[q], fabsf(d0 - (float)(8 * k + e)), v * sl);
                            }
                    }
                }
                sl = 1.f;
            }
            // Running max: each thread first checks its own 32 keys of each row against the
            // running max; only when some row of the warp grew past it by more than 2^8 (the
            // first tile, or a jump in the scores) are the exact row maxima taken over the quad
            // and O rescaled.
            float lm[2];
            bool grow = false;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float c0 = fmaxf(sv[2 * q], sv[2 * q + 1]), c1 = fmaxf(sv[4 + 2 * q], sv[5 + 2 * q]);
#pragma unroll
                for (int k = 2; k < 16; k += 2) {
                    c0 = max3f(c0, sv[4 * k + 2 * q], sv[4 * k + 2 * q + 1]);
                    c1 = max3f(c1, sv[4 * k + 4 + 2 * q], sv[4 * k + 5 + 2 * q]);
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
                // O_x was accumulated with the old maximum.  Its last P.V (PV_x(j-1)) precedes
                // S_x(j) in the tensor pipe, so it is complete once S_x(j) is.
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
            // pk[2k + q] = P[row q][packed column 4k + tig] = (keys 8k + 2 tig, 8k + 2 tig + 1),
            // the register order of the 16x128b store
            uint32_t pk[32];
#pragma unroll
            for (int k = 0; k < 16; ++k)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float x0, x1;
                    ffma2(x0, x1, sv[4 * k + 2 * q], sv[4 * k + 2 * q + 1], sl, sl, nm[q], nm[q]);
                    const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                    fadd2_acc(sums[2 * q], sums[2 * q + 1], p0, p1);
                    pk[2 * k + q] = pack2<T>(p0, p1);
                }
#pragma unroll
            for (int q = 0; q < 2; ++q) st.l[q] = st.l[q] * alpha[q] + (sums[2 * q] + sums[2 * q + 1]);
            // P overwrites the first 64 columns of the S it came from (this thread's own cells)
            tc::st_16x128b_x16(s_addr, pk);
            tc::wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[x]);
            return true;
        };

        auto epilogue = [&](int x, TileRows& st) -> bool {
            if (!__all_sync(0xffffffffu, wait_bar(&pv_done[x], 0, abort_flag, p.err, p.wait_ns))) return false;
            tc::fence_after_sync();
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
                const int64_t rho = tile_rho(x, lb + gid + 8 * q);
                valid[q] = row_live(x, lb + gid + 8 * q);
                const int i = (int)(rho / p.G), g = (int)(rho - (int64_t)i * p.G);
                const int64_t t = q0 + i;
                const int h = hk * p.G + g;
                orow[q] = out + t * p.o_s0 + (int64_t)h * p.o_s1;
                if (valid[q] && tig == 0)
                    p.lse[(int64_t)h * p.lse_s0 + t + (int64_t)b * p.lse_sb] =
                        l > 0.f ? (st.m[q] + log2f(l)) * 0.69314718055994531f : -INFINITY;
            }
#pragma unroll 1
            for (int cc = 0; cc < DP / 64; ++cc) {
                float o[32];
                tc::ld_16x256b_x8(o_addr + cc * 64, o);
                tc::wait_ld();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int d = cc * 64 + 8 * k + 2 * tig;
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        if (valid[q] && d < p.D)
                            *reinterpret_cast<uint32_t*>(orow[q] + d) =
                                pack2<T>(o[4 * k + 2 * q] * inv[q], o[4 * k + 2 * q + 1] * inv[q]);
                }
            }
            return true;
        };

        bool ok = true;
        for (int j = 0; ok && j < n_tiles; ++j) {
            ok = step(0, rows_a, j);
            if (ok && has_b) ok = step(1, rows_b, j);
        }
        if (ok) ok = epilogue(0, rows_a);
        if (ok && has_b) epilogue(1, rows_b);
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

template <typename T, int DP, bool ALIBI>
int run_prefill(const Args& a, const PrefillParams& pp, cudaStream_t stream, char* msg, size_t msg_len) {
    using C = PfCfg<DP>;
    // tensor maps: q as (D, H, total_q, 1), box (64, G, 128 / G, 1); K/V as in the split-KV path
    CUtensorMap tq, tk, tv;
    {
        const uint64_t dims[4] = {(uint64_t)a.D, (uint64_t)a.H, (uint64_t)a.total_q, 1};
        const uint64_t strides[3] = {(uint64_t)a.q_s1 * 2, (uint64_t)a.q_s0 * 2, (uint64_t)a.q_s0 * 2 * a.total_q};
        const uint32_t box[4] = {64u, (uint32_t)pp.G, (uint32_t)(128 / pp.G), 1u};
        int rc = encode_tmap_4d(&tq, a.dtype, a.q, dims, strides, box, 1, msg, msg_len);
        if (rc != PA_OK) return rc;
    }
    {
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
        int rc = encode_tmap_4d(&tk, a.dtype, a.k, dims, strides, box, 1, msg, msg_len);
        if (rc != PA_OK) return rc;
        rc = encode_tmap_4d(&tv, a.dtype, a.v, dims, strides, box, 1, msg, msg_len);
        if (rc != PA_OK) return rc;
    }
    auto kern = prefill_kernel<T, DP, ALIBI>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "cudaFuncSetAttribute(prefill, %d bytes): %s", C::SMEM, cudaGetErrorString(e));
            return PA_ERR_CUDA;
        }
        configured = true;
    }
    dim3 grid(pp.pairs, a.Hkv, 1);
    NvtxRange nv("pa::prefill_kernel");
    timer_begin(PA_KC_PREFILL, stream);
    kern<<<grid, kPrefillThreads, C::SMEM, stream>>>(tq, tk, tv, pp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "prefill launch: %s", cudaGetErrorString(e));
        return PA_ERR_CUDA;
    }
    timer_end(PA_KC_PREFILL, stream);
    count_launches(1);
    return PA_OK;
}

// ---------------------------------------------------------------------------------------------
// Head dim 129..256: one 128-row query tile per CTA, q held in tensor memory.
//
// Two query tiles whose O takes 256 columns each would need more than the 512 TMEM columns,
// and 128-key K/V stages (64 KB each) do not fit twice beside a 64 KB q tile in shared
// memory.  So a CTA owns one query tile of one (sequence, kv head) (q by TMA into shared
// memory, 64 KB); K and V come in 64-key tiles (32 KB) through a 3-deep K ring and a 2-deep
// V ring.  S is quadruple-buffered over consecutive key tiles (64 columns each), so the
// Q.K^T issuer runs up to three tiles ahead of the softmax while the pipe also computes P.V.
// TMEM columns: S0..S3 [0,256), O [256,512).  (With q in tensor memory and two S buffers
// the chain P.V(j) -> Q.K^T(j+2) -> softmax(j+2) bounded the kernel at ~1,950 cycles a tile.)
// Roles: warp 0 K producer, warp 2 V producer, warp 1 the Q.K^T issuer (and TMEM owner),
// warp 3 the P.V issuer, warps 4..11 softmax (two warps per 32-lane TMEM quarter, 16 rows
// each).  A 128x64x16 product keeps the tensor pipe ~32 cycles and costs its issuing thread
// about twice that, so one thread issuing both products of a tile bounded the kernel
// (40 % tensor-pipe activity, 935 TFLOP/s); two issuers share the work.  The P.V issuer
// commits PV(j) to buf_free[j % 4]; the Q.K^T issuer waits for it before S(j+4) reuses the
// columns P(j) was read from, and the softmax waits for PV(j-1) there before it hands over
// P(j) -- only then may it rescale O -- and releases V stage j-1.  Each waiter takes a
// buffer's phases in order, and the next phase of a buffer needs work the waiter has not yet
// released, so no wait can see a barrier two phases ahead.  The softmax releases K stage j
// once S(j) is complete.
struct P2Cfg {
    static constexpr int DP = 256, CH = 4, NT = 64, NSB = 4;  // NSB: S buffers
    static constexpr int Q_TILE = CH * 128 * 128;  // one 128-row q tile: 64 KB
    static constexpr int KV_TILE = CH * NT * 128;  // 64 keys x 256 columns: 32 KB
    static constexpr int KS = 3, VS = 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = Q_TILE;
    static constexpr int OFF_V = OFF_K + KS * KV_TILE;
    static constexpr int OFF_BAR = OFF_V + VS * KV_TILE;
    // q_full, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], s_full[NSB], p_full[NSB],
    // buf_free[NSB], drain[2]
    static constexpr int NBAR = 1 + 2 * KS + 2 * VS + 3 * NSB + 2;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem base, abort flag, picked tile
    static constexpr int OFF_IDS = OFF_MISC + 16;
    static constexpr int MAX_BOXES = 256;
    static constexpr int SMEM = OFF_IDS + (MAX_BOXES + 4) * 4 + 1024;
    static constexpr uint32_t T_S = 0, T_O = 256;  // S buffer x at T_S + 64 x
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

// Issues the K (or V) boxes of the CTA's 64-key tile number `j` (first key kt0 + 64 j) into
// `dst` (chunk-major: 64-column chunk c holds rows [64 c, 64 c + 64) of 128 bytes).
__device__ __forceinline__ void issue_kv_tile64(const PrefillParams& p, const CUtensorMap* map, uint8_t* dst,
                                                uint64_t* bar, const int* ids, int j, int hk, int kt0, int k0) {
    const int kt = kt0 + j * 64;
    int blk[2];
    uint32_t bytes = 0;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        blk[jj] = jj < p.boxes_per_tile ? ids[j * p.boxes_per_tile + jj] : -1;
        if (blk[jj] >= 0) bytes += (uint32_t)(P2Cfg::CH * p.box_rows * 128);
    }
    mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        if (blk[jj] < 0) continue;
        const int key = kt + jj * p.box_rows;
        const int c2 = p.paged ? key - (key / p.P) * p.P : k0 + key;
        const int c3 = p.paged ? blk[jj] : 0;
        for (int c = 0; c < P2Cfg::CH; ++c)
            tma_load_4d(dst + (c * 64 + jj * p.box_rows) * 128, map, bar, c * 64, hk, c2, c3, 0ull);
    }
}

template <typename T, bool ALIBI>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    prefill256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
    using C = P2Cfg;
    constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hk = blockIdx.y;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* k_empty = k_full + C::KS;
    uint64_t* v_full = k_empty + C::KS;
    uint64_t* v_empty = v_full + C::VS;
    uint64_t* s_full = v_empty + C::VS;     // [S buffer]
    uint64_t* p_full = s_full + C::NSB;     // [S buffer]
    uint64_t* buf_free = p_full + C::NSB;   // [S buffer]: the P.V that read it has completed
    uint64_t* drain = buf_free + C::NSB;    // [issuer]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile uint32_t* abort_flag = tmem_slot + 1;
    if (tid == 64) {
        mbar_init(q_full, 1);
        for (int s = 0; s < C::KS; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < C::VS; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int x = 0; x < C::NSB; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], 8);
            mbar_init(&buf_free[x], 1);
        }
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }

    // ---- which (sequence, query tile) this CTA owns: the blockIdx.x-th of all 128-row tiles of
    // prefill-class sequences, sequence by sequence, each sequence's last tile first.
    int* pick = reinterpret_cast<int*>(smem + C::OFF_MISC + 8);
    const int qpt = 128 / p.G;    // whole queries per tile
    const int trows = qpt * p.G;  // rows of the tile that hold queries (the rest are padding)
    if (warp == 0) {
        int remaining = (int)blockIdx.x, found_b = -1, found_u = 0;
        for (int base = 0; base < p.batch && found_b < 0; base += 32) {
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
                found_b = base + src;
                found_u = cnt - 1 - (remaining - excl);
            } else {
                remaining -= __shfl_sync(0xffffffffu, incl, 31);
            }
        }
        if (lane == 0) {
            pick[0] = found_b;
            pick[1] = found_u;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int b = pick[0], u = pick[1];
    auto leave = [&]() {  // every early exit below is uniform over the CTA
        if (warp == 1) tc::tmem_dealloc(tmem, 512);
    };
    if (b < 0) {
        leave();
        return;
    }
    const int q0 = p.cu_q[b], q1 = p.cu_q[b + 1];
    const int k0 = p.cu_k[b], k1 = p.cu_k[b + 1];
    const int sq = q1 - q0, sk = k1 - k0;
    if (sq < 0 || sk < 0 || sq > p.max_sq || sk > p.max_sk || q0 < 0 || q1 > p.total_q ||
        (!p.paged && (k0 < 0 || k1 > p.num_blocks))) {
        if (tid == 0) flag_error(p.err, PA_ERR_DEVICE_BOUNDS);
        leave();
        return;
    }
    const int64_t rows_total = (int64_t)sq * p.G;
    const int i0 = u * qpt;  // first query of the tile
    auto tile_rho = [&](int r) -> int64_t { return (int64_t)i0 * p.G + r; };
    auto row_live = [&](int r) { return r < trows && tile_rho(r) < rows_total; };
    const int i_last = min(sq - 1, i0 + qpt - 1);
    const int64_t cdiag = (int64_t)sk - sq;
    const int64_t lo = p.wl >= 0 ? max64(0, i0 + cdiag - p.wl) : 0;
    const int64_t hi = p.wr >= 0 ? min64((int64_t)sk - 1, i_last + cdiag + p.wr) : (int64_t)sk - 1;
    const int kt0 = hi >= lo ? (int)(lo & ~int64_t(63)) : 0;
    const int n_tiles = hi >= lo ? (int)((hi - kt0) / 64 + 1) : 0;

    T* out = static_cast<T*>(p.out);
    if (n_tiles == 0) {  // no row of the tile attends any key: out = 0, lse = -inf
        if (warp >= 4 && warp < 8) {
            const int r = (warp & 3) * 32 + lane;
            if (row_live(r)) {
                const int64_t rho = tile_rho(r);
                const int i = (int)(rho / p.G), g = (int)(rho - (int64_t)i * p.G);
                const int64_t t = q0 + i;
                const int h = hk * p.G + g;
                for (int d = 0; d < p.D; d += 8)
                    *reinterpret_cast<int4*>(out + t * p.o_s0 + (int64_t)h * p.o_s1 + d) = make_int4(0, 0, 0, 0);
                p.lse[(int64_t)h * p.lse_s0 + t + (int64_t)b * p.lse_sb] = -INFINITY;
            }
        }
        leave();
        return;
    }

    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl));
    if (warp == 0 || warp == 2) {
        // ---------------- TMA producers: warp 0 K tiles, warp 2 V tiles ----------------
        int* ids = reinterpret_cast<int*>(smem + C::OFF_IDS);
        const int n_boxes = min(n_tiles * p.boxes_per_tile, C::MAX_BOXES);
        const int32_t* bt_row = p.paged ? p.bt + (int64_t)b * p.bt_s0 : nullptr;
        if (warp == 0) {
            if (lane == 0 && !p.withhold) {  // the q tile first: its latency overlaps the id lookups
                prefetch_tmap(&tm_q);
                mbar_arrive_expect_tx(q_full, C::CH * trows * 128);
                for (int c = 0; c < C::CH; ++c)
                    tma_load_4d(smem + C::OFF_Q + c * 128 * 128, &tm_q, q_full, c * 64, hk * p.G, q0 + i0, 0, 0ull);
            }
            for (int bi = lane; bi < n_boxes; bi += 32) {
                const int key = kt0 + bi * p.box_rows;
                ids[bi] = p.paged ? box_block(bt_row, p.bt_cols, p.num_blocks, p.P, key, sk, p.err)
                                  : (key < sk ? 0 : -1);
            }
        }
        named_barrier_sync(2, 64);  // warps 0 and 2: the staged ids are visible
        const bool is_k = warp == 0;
        if (lane == 0 && !p.withhold) {
            const CUtensorMap* map = is_k ? &tm_k : &tm_v;
            prefetch_tmap(map);
            const int stages = is_k ? C::KS : C::VS;
            uint64_t* fullb = is_k ? k_full : v_full;
            uint64_t* emptyb = is_k ? k_empty : v_empty;
            uint8_t* ring = smem + (is_k ? C::OFF_K : C::OFF_V);
            int spill[2];  // block ids of one tile past the staged range
            for (int j = 0; j < n_tiles; ++j) {
                const int s = j % stages;
                if (j >= stages && !wait_bar(&emptyb[s], ((j / stages) - 1) & 1, abort_flag, p.err, p.wait_ns))
                    break;
                const int* tile = ids;
                int jt = j, kb = kt0;
                if ((j + 1) * p.boxes_per_tile > C::MAX_BOXES) {
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int key = kt0 + j * 64 + jj * p.box_rows;
                        spill[jj] = jj >= p.boxes_per_tile ? -1
                                    : p.paged ? box_block(bt_row, p.bt_cols, p.num_blocks, p.P, key, sk, p.err)
                                              : (key < sk ? 0 : -1);
                    }
                    tile = spill;
                    jt = 0;
                    kb = kt0 + j * 64;
                }
                issue_kv_tile64(p, map, ring + s * C::KV_TILE, &fullb[s], tile, jt, hk, kb, k0);
            }
        }
    } else {
        // ---------------- MMA issuers: warp 1 Q.K^T, warp 3 P.V ----------------
        constexpr uint32_t IDESC_S = tc::idesc_f16(128, 64, kBF16, false, false);
        constexpr uint32_t IDESC_O = tc::idesc_f16(128, 256, kBF16, false, true);
        const bool s_issuer = warp == 1;
        auto s_buf = [&](int j) { return tmem + C::T_S + 64 * (j % C::NSB); };
        auto wait_all = [&](uint64_t* bar, uint32_t parity) {
            const bool r = __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, p.err, p.wait_ns));
            tc::fence_after_sync();
            return r;
        };
        if (s_issuer) {
            // S(j) = Q K_j^T into S buffer j % NSB (A: the q tile, B: K stage, both K-major)
            const uint64_t da = tc::smem_desc_sw128(smem_addr(smem + C::OFF_Q), 16, 1024);
            const uint64_t dk0 = tc::smem_desc_sw128(smem_addr(smem + C::OFF_K), 16, 1024);
            bool ok = wait_all(q_full, 0);
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int x = j % C::NSB;
                if (j >= C::NSB && !(ok = wait_all(&buf_free[x], ((j / C::NSB) - 1) & 1))) break;
                if (!(ok = wait_all(&k_full[j % C::KS], (j / C::KS) & 1))) break;
                if (lane == 0) {
                    const uint64_t db = dk0 + (uint64_t)((j % C::KS) * (C::KV_TILE >> 4));
#pragma unroll
                    for (int kk = 0; kk < C::DP / 16; ++kk) {
                        const uint64_t oa = (uint64_t)((kk >> 2) * (128 * 128 / 16) + (kk & 3) * 2);
                        const uint64_t ob = (uint64_t)((kk >> 2) * (64 * 128 / 16) + (kk & 3) * 2);
                        tc::mma_ss(s_buf(j), da + oa, db + ob, IDESC_S, kk > 0 ? 1u : 0u);
                    }
                    tc::commit(&s_full[x]);
                }
                __syncwarp();
            }
        } else {
            // O += P(j) V_j, P(j) in the first 32 columns of S buffer j % NSB
            const uint64_t dv0 = tc::smem_desc_sw128(smem_addr(smem + C::OFF_V), 64 * 128, 1024);
            const uint32_t t_o = tmem + C::T_O;
            bool ok = true;
            for (int j = 0; ok && j < n_tiles; ++j) {
                if (!(ok = wait_all(&v_full[j % C::VS], (j / C::VS) & 1))) break;
                uint8_t* vst = smem + C::OFF_V + (j % C::VS) * C::KV_TILE;
                const int valid = min(64, sk - (kt0 + j * 64));
                if (valid < 64) {  // keys at or past sk: zero V rows so P = 0 never meets NaN
                    const int zr = 64 - valid;
                    for (int idx = lane; idx < C::CH * zr * 8; idx += 32) {
                        const int c = idx / (zr * 8), rem = idx - c * zr * 8;
                        *reinterpret_cast<int4*>(vst + (c * 64 + valid + (rem >> 3)) * 128 + ((rem & 7) << 4)) =
                            make_int4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    tc::fence_after_sync();
                }
                if (!(ok = wait_all(&p_full[j % C::NSB], (j / C::NSB) & 1))) break;
                if (lane == 0) {
                    const uint64_t db = dv0 + (uint64_t)((j % C::VS) * (C::KV_TILE >> 4));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_ts(t_o, s_buf(j) + kk * 8, db + (uint64_t)(kk * (2048 / 16)), IDESC_O,
                                   kk > 0 ? 1u : (j > 0 ? 1u : 0u));
                    tc::commit(&buf_free[j % C::NSB]);
                }
                __syncwarp();
            }
        }
        // every MMA this issuer started has completed before tensor memory is released
        if (lane == 0) {
            uint64_t* d = &drain[s_issuer ? 0 : 1];
            tc::commit(d);
            mbar_wait(d, 0, p.wait_ns);  // not cut short by an abort: MMAs may be in flight
        }
        __syncwarp();
    }
    } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    {
        // ---------------- softmax: warps 4..11 ----------------
        // Warp w reaches TMEM lanes 32 (w % 4) .. +31 and takes half hh = (w - 4) / 4 of them:
        // lanes lb .. lb + 15, lb = 32 (w % 4) + 16 hh.  Thread t holds rows lb + t/4 (q = 0)
        // and lb + t/4 + 8 (q = 1); the four threads of a quad split a row's 64 keys (keys
        // 8k + 2 (t % 4) + {0, 1}, k = 0..7).
        const int lg = warp & 3, hh = (warp - 4) >> 2;
        const int gid = lane >> 2, tig = lane & 3;
        const int lb = lg * 32 + hh * 16;
        const uint32_t lane_addr = (uint32_t)lb << 16;

        int lo_r[2], hi_r[2], dg_r[2];
        float ab_r[2], m_r[2], l_r[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int r = lb + gid + 8 * q;
            lo_r[q] = 0;
            hi_r[q] = -1;
            dg_r[q] = 0;
            ab_r[q] = 0.f;
            if (row_live(r)) {
                const int64_t rho = tile_rho(r);
                const int64_t diag = rho / p.G + cdiag;
                lo_r[q] = p.wl >= 0 ? (int)max64(0, diag - p.wl) : 0;
                hi_r[q] = p.wr >= 0 ? (int)max64(-1, min64((int64_t)sk - 1, diag + p.wr)) : sk - 1;
                if (ALIBI) {
                    dg_r[q] = (int)diag;
                    ab_r[q] = p.alibi[hk * p.G + (int)(rho - (rho / p.G) * p.G)] * kLog2e;
                }
            }
            m_r[q] = -INFINITY;
            l_r[q] = 0.f;
        }
        const uint32_t o_addr = tmem + lane_addr + C::T_O;

        // One key tile: S -> running max -> P; O rescaled (rarely) once PV(j-1) is complete.
        auto step = [&](int j) -> bool {
            const int kt = kt0 + j * 64;
            if (!__all_sync(0xffffffffu,
                            wait_bar(&s_full[j % C::NSB], (j / C::NSB) & 1, abort_flag, p.err, p.wait_ns)))
                return false;
            tc::fence_after_sync();
            const uint32_t s_addr = tmem + lane_addr + C::T_S + 64 * (j % C::NSB);
            // sv[4k + 2q + e] = S[row q][key 8k + 2 tig + e]
            float sv[32];
            tc::ld_16x256b_x8(s_addr, sv);
            if (warp == 4 && lane == 0) mbar_arrive(&k_empty[j % C::KS]);  // S(j) is complete: K stage j is free
            tc::wait_ld();
            if (!(kt >= max(lo_r[0], lo_r[1]) && kt + 63 <= min(hi_r[0], hi_r[1]))) {
#pragma unroll
                for (int k = 0; k < 8; ++k)
#pragma unroll
                    for (int q = 0; q < 2; ++q)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int key = kt + 8 * k + 2 * tig + e;
                            float& v = sv[4 * k + 2 * q + e];
                            v = (key >= lo_r[q] && key <= hi_r[q]) ? v : -INFINITY;
                        }
            }
            float sl = p.scale_log2;  // softmax_scale > 0 on this path
            if (ALIBI) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const float d0 = (float)(dg_r[q] - kt - 2 * tig);  // distance of key kt + 2 tig
#pragma unroll
                    for (int k = 0; k < 8; ++k)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            float& v = sv[4 * k + 2 * q + e];
                            v = fmaf(-ab_r[q], fabsf(d0 - (float)(8 * k + e)), v * sl);
                        }
                }
                sl = 1.f;
            }
            // running max with the lazy rescale of the 128-key kernel: exact row maxima and
            // an O rescale only when some row of the warp grew by more than 2^8
            float lm[2];
            bool grow = false;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float c0 = fmaxf(sv[2 * q], sv[2 * q + 1]), c1 = fmaxf(sv[4 + 2 * q], sv[5 + 2 * q]);
#pragma unroll
                for (int k = 2; k < 8; k += 2) {
                    c0 = max3f(c0, sv[4 * k + 2 * q], sv[4 * k + 2 * q + 1]);
                    c1 = max3f(c1, sv[4 * k + 4 + 2 * q], sv[4 * k + 5 + 2 * q]);
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
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 8; ++k)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float x0, x1;
                    ffma2(x0, x1, sv[4 * k + 2 * q], sv[4 * k + 2 * q + 1], sl, sl, nm[q], nm[q]);
                    const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                    fadd2_acc(sums[2 * q], sums[2 * q + 1], p0, p1);
                    pk[2 * k + q] = pack2<T>(p0, p1);
                }
#pragma unroll
            for (int q = 0; q < 2; ++q) l_r[q] = l_r[q] * alpha[q] + (sums[2 * q] + sums[2 * q + 1]);
            if (j > 0) {
                // PV(j-1) complete: O holds every earlier tile, V stage j-1 is free
                if (!__all_sync(0xffffffffu, wait_bar(&buf_free[(j - 1) % C::NSB], ((j - 1) / C::NSB) & 1, abort_flag,
                                                      p.err, p.wait_ns)))
                    return false;
                tc::fence_after_sync();
                if (warp == 4 && lane == 0) mbar_arrive(&v_empty[(j - 1) % C::VS]);
                if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
                    for (int cc = 0; cc < C::DP / 64; ++cc) {
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
            // P overwrites the first 32 columns of the S it came from (this thread's own cells)
            tc::st_16x128b_x8(s_addr, pk);
            tc::wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[j % C::NSB]);
            return true;
        };

        bool ok = true;
        for (int j = 0; ok && j < n_tiles; ++j) ok = step(j);
        if (ok && __all_sync(0xffffffffu, wait_bar(&buf_free[(n_tiles - 1) % C::NSB], ((n_tiles - 1) / C::NSB) & 1,
                                                   abort_flag, p.err, p.wait_ns))) {
            tc::fence_after_sync();
            float inv[2];
            T* orow[2];
            bool valid[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float l = l_r[q];
                l += __shfl_xor_sync(0xffffffffu, l, 1);
                l += __shfl_xor_sync(0xffffffffu, l, 2);
                inv[q] = l > 0.f ? 1.f / l : 0.f;
                const int r = lb + gid + 8 * q;
                const int64_t rho = tile_rho(r);
                valid[q] = row_live(r);
                const int i = (int)(rho / p.G), g = (int)(rho - (int64_t)i * p.G);
                const int64_t t = q0 + i;
                const int h = hk * p.G + g;
                orow[q] = out + t * p.o_s0 + (int64_t)h * p.o_s1;
                if (valid[q] && tig == 0)
                    p.lse[(int64_t)h * p.lse_s0 + t + (int64_t)b * p.lse_sb] =
                        l > 0.f ? (m_r[q] + log2f(l)) * 0.69314718055994531f : -INFINITY;
            }
#pragma unroll 1
            for (int cc = 0; cc < C::DP / 64; ++cc) {
                float o[32];
                tc::ld_16x256b_x8(o_addr + cc * 64, o);
                tc::wait_ld();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int d = cc * 64 + 8 * k + 2 * tig;
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        if (valid[q] && d < p.D)
                            *reinterpret_cast<uint32_t*>(orow[q] + d) =
                                pack2<T>(o[4 * k + 2 * q] * inv[q], o[4 * k + 2 * q + 1] * inv[q]);
                }
            }
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

template <typename T, bool ALIBI>
int run_prefill256(const Args& a, const PrefillParams& pp, cudaStream_t stream, char* msg, size_t msg_len) {
    using C = P2Cfg;
    CUtensorMap tq, tk, tv;
    {  // q as (D, H, total_q, 1), box (64, G, 128 / G, 1), as in the head-dim-128 kernel
        const uint64_t dims[4] = {(uint64_t)a.D, (uint64_t)a.H, (uint64_t)a.total_q, 1};
        const uint64_t strides[3] = {(uint64_t)a.q_s1 * 2, (uint64_t)a.q_s0 * 2, (uint64_t)a.q_s0 * 2 * a.total_q};
        const uint32_t box[4] = {64u, (uint32_t)pp.G, (uint32_t)(128 / pp.G), 1u};
        int rc = encode_tmap_4d(&tq, a.dtype, a.q, dims, strides, box, 1, msg, msg_len);
        if (rc != PA_OK) return rc;
    }
    {
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
        int rc = encode_tmap_4d(&tk, a.dtype, a.k, dims, strides, box, 1, msg, msg_len);
        if (rc != PA_OK) return rc;
        rc = encode_tmap_4d(&tv, a.dtype, a.v, dims, strides, box, 1, msg, msg_len);
        if (rc != PA_OK) return rc;
    }
    auto kern = prefill256_kernel<T, ALIBI>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) {
            snprintf(msg, msg_len, "cudaFuncSetAttribute(prefill256, %d bytes): %s", C::SMEM, cudaGetErrorString(e));
            return PA_ERR_CUDA;
        }
        configured = true;
    }
    dim3 grid(pp.pairs, a.Hkv, 1);
    NvtxRange nv("pa::prefill256_kernel");
    timer_begin(PA_KC_PREFILL, stream);
    kern<<<grid, kPrefillThreads, C::SMEM, stream>>>(tq, tk, tv, pp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "prefill256 launch: %s", cudaGetErrorString(e));
        return PA_ERR_CUDA;
    }
    timer_end(PA_KC_PREFILL, stream);
    count_launches(1);
    return PA_OK;
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

int launch_prefill(const Args& a, unsigned int* err, char* msg, size_t msg_len) {
    PrefillParams pp{};
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
    if (a.paged) {
        pp.box_rows = (a.page % 128 == 0) ? 128 : (a.page % 64 == 0) ? 64 : 32;
    } else {
        pp.box_rows = 128;
    }
    pp.boxes_per_tile = 128 / pp.box_rows;
    pp.max_sq = a.max_sq;
    pp.max_sk = a.max_sk;
    pp.scale_log2 = a.scale * 1.4426950408889634f;
    pp.alibi = a.alibi;
    pp.wl = a.wl;
    pp.wr = a.wr;
    pp.rows_cap = prefill_rows_threshold();
    // upper bound of the number of tile pairs (2 qpt queries each, qpt = floor(128 / G)):
    // sum_b ceil(sq_b / (2 qpt)) <= ceil(total_q / (2 qpt)) + batch
    const int64_t pq = 2 * (128 / pp.G);
    pp.pairs = (int)std::min<int64_t>(((int64_t)a.total_q + pq - 1) / pq + a.batch,
                                      (int64_t)a.batch * (((int64_t)a.max_sq + pq - 1) / pq));
    pp.err = err;
    pp.wait_ns = a.wait_ns;
    pp.withhold = a.withhold_loads;
    const bool alibi = a.alibi != nullptr;
    if (a.D > 128) {  // one 128-row query tile per CTA, 64-key K/V tiles
        pp.box_rows = a.paged ? (a.page % 64 == 0 ? 64 : 32) : 64;
        pp.boxes_per_tile = 64 / pp.box_rows;
        // upper bound of the number of tiles: sum_b ceil(sq_b / qpt) <= ceil(total_q / qpt) + batch
        const int64_t qpt = 128 / pp.G;
        pp.pairs = (int)std::min<int64_t>(((int64_t)a.total_q + qpt - 1) / qpt + a.batch,
                                          (int64_t)a.batch * (((int64_t)a.max_sq + qpt - 1) / qpt));
        if (a.dtype == PA_BF16)
            return alibi ? run_prefill256<__nv_bfloat16, true>(a, pp, a.stream, msg, msg_len)
                         : run_prefill256<__nv_bfloat16, false>(a, pp, a.stream, msg, msg_len);
        return alibi ? run_prefill256<__half, true>(a, pp, a.stream, msg, msg_len)
                     : run_prefill256<__half, false>(a, pp, a.stream, msg, msg_len);
    }
    const int dp = a.D <= 64 ? 64 : 128;
    if (a.dtype == PA_BF16) {
        if (alibi)
            return dp == 64 ? run_prefill<__nv_bfloat16, 64, true>(a, pp, a.stream, msg, msg_len)
                            : run_prefill<__nv_bfloat16, 128, true>(a, pp, a.stream, msg, msg_len);
        return dp == 64 ? run_prefill<__nv_bfloat16, 64, false>(a, pp, a.stream, msg, msg_len)
                        : run_prefill<__nv_bfloat16, 128, false>(a, pp, a.stream, msg, msg_len);
    }
    if (alibi)
        return dp == 64 ? run_prefill<__half, 64, true>(a, pp, a.stream, msg, msg_len)
                        : run_prefill<__half, 128, true>(a, pp, a.stream, msg, msg_len);
    return dp == 64 ? run_prefill<__half, 64, false>(a, pp, a.stream, msg, msg_len)
                    : run_prefill<__half, 128, false>(a, pp, a.stream, msg, msg_len);
}

}  // namespace pa
