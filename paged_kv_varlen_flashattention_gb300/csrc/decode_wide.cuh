// Decode-class paged attention kernel for the widest heads (head dim 257..512).
//
// One CTA owns one (sequence, kv head, key split) with at most 32 query rows (the
// (query, head) pairs of the GQA group, ordered i * G + g), like the warp-sliced decode
// kernel.  At head dim 512 a warp cannot hold the output of 16 rows over the whole head
// dim in registers (256 fp32 a thread), so the eight consumer warps split the head dim in
// quarters of 128 columns instead: warp w takes quarter w % 4 of the rows and keys of its
// group w / 4 (the two 16-row groups of a 32-row tile, or the two 16-key halves of every
// tile when the CTA has 16 rows).  Per key tile of 32 keys:
//   * each warp forms the partial scores of its rows and keys over its 128 columns
//     (Q fragments held in registers, K fragments from the TMA-swizzled stage);
//   * the four quarter warps of a group exchange their fp32 partials through a
//     double-buffered shared-memory slot and a 128-thread named barrier.  With 32 rows (one
//     group per 16 rows, all 32 keys) the exchange is a reduce-scatter: warp dq sums the
//     partials of the 8 keys 8 dq .. 8 dq + 7 only, runs the softmax of those keys and posts
//     their probabilities (in the precision of V) and its row maxima; after a second barrier
//     every warp reads the whole P tile.  The four warps share one running reference per
//     row, raised (and O rescaled) only when some key exceeds it by more than 2^8, a
//     decision all four take from the same posted maxima.  With 16 rows (two key halves)
//     every warp sums all four partials of its 16 keys in quarter order;
//   * each accumulates P.V for its 128 output columns, then releases the stage.
// Four producer warps feed a three-stage ring of 64 KB K/V tiles with TMA: warp p issues
// the 64-column chunks 2p and 2p + 1 of K and V and posts its own bytes on the stage's
// full barrier before issuing them (one TMA issuing thread per warp keeps the per-thread
// issue rate from bounding the load rate).  At the end every warp normalises and stores its
// own rows and columns from registers; the two key halves of a 16-row CTA are first merged
// through one lane-matched shared-memory exchange.
#pragma once

#include <limits.h>

#include "decode_kernel.cuh"

namespace pa {

template <int MG, int STAGES>
struct WideCfg {
    static constexpr int DP = 512, NT = 32, CH = DP / 64;
    static constexpr int M = 16 * MG;             // rows per CTA
    static constexpr int KW = 2 / MG;             // key slices per row group
    static constexpr int KPW = NT / KW;           // keys per warp per tile
    static constexpr int NSC = KPW / 8;           // n8 score tiles per warp
    static constexpr int CONS = 8, PROD = 4;
    static constexpr int THREADS = (CONS + PROD) * 32;
    static constexpr int QW = 128;                // output columns per warp
    static constexpr int TILE_BYTES = CH * NT * 128;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    // Score exchange per tile (two buffers, alternating by tile).  Two key slices (16 rows):
    // one float4 per (warp, score tile, lane).  One slice (32 rows): a reduce-scatter, where
    // warp dq owns score tile dq (keys 8 dq .. 8 dq + 7) and receives the other three quarters'
    // partials of it (one float4 per (warp, slot, lane)), then posts its probabilities in the
    // precision of V (one pair of words per (warp, lane)) and its rows' maxima.
    static constexpr int XS_BYTES = CONS * 3 * 32 * 16;
    static constexpr int XP_OFF = XS_BYTES;
    static constexpr int XM_OFF = XP_OFF + CONS * 32 * 8;
    static constexpr int XBUF_BYTES = KW == 2 ? CONS * NSC * 32 * 16 : XM_OFF + 2 * 16 * 4 * 4;
    static constexpr int Q_BYTES = CH * M * 128;
    static constexpr int X_BYTES = 2 * XBUF_BYTES > Q_BYTES ? 2 * XBUF_BYTES : Q_BYTES;
    static_assert(KW == 2 || NSC == 4, "one score tile per quarter warp");
    static constexpr int OFF_X = STAGES * STAGE_BYTES;        // Q staging, then the score exchange
    static constexpr int OFF_ROW = OFF_X + X_BYTES;           // row_lo[M], row_hi[M], row_dg[M], row_ab[M]
    static constexpr int OFF_BAR = OFF_ROW + 4 * M * 4;
    static constexpr int OFF_FLAG = OFF_BAR + 2 * STAGES * 8;
    static constexpr int SMEM = OFF_FLAG + 16 + 1024;         // + slack for 1024-byte alignment
    static constexpr int MERGE_BYTES = 4 * (QW / 8) * 32 * 16 + 4 * 32 * 16;  // second key half's O, m, l
    static_assert(KPW % 16 == 0, "keys per warp");
    static_assert(MERGE_BYTES <= STAGES * STAGE_BYTES, "merge scratch");
    static_assert(SMEM + (kRankInCta + 1) * 4 <= 227 * 1024, "shared memory per CTA");
};

template <typename T, int MG, int STAGES>
__global__ void __launch_bounds__(WideCfg<MG, STAGES>::THREADS, 1)
    decode512_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const SplitParams p) {
    using C = WideCfg<MG, STAGES>;
    constexpr int M = C::M, NT = C::NT, DP = C::DP;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    allow_dependent_launch();
    if (tid == C::CONS * 32) {  // the first producer lane: descriptors on their way at once
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    // sequences longest first, as in the warp-sliced decode kernel
    __shared__ int rank_len[kRankInCta];
    __shared__ int rank_pick;
    int b = (int)blockIdx.z;
    if (p.order) {
        b = p.order[blockIdx.z];
    } else if (p.rank_in_cta) {
        if (tid < p.batch) rank_len[tid] = p.cu_k[tid + 1] - p.cu_k[tid];
        if (tid == 0) rank_pick = (int)blockIdx.z;
        __syncthreads();
        if (tid < p.batch) {
            const int ls = rank_len[tid];
            int rank = 0;
            for (int t = 0; t < p.batch; ++t) {
                const int lt = rank_len[t];
                rank += (lt > ls) || (lt == ls && t < tid);
            }
            if (rank == (int)blockIdx.z) rank_pick = tid;
        }
        __syncthreads();
        b = rank_pick;
    }
    const int hk = blockIdx.y % p.Hkv, split = blockIdx.x;
    if (warp == C::CONS) prefetch_split_pages<NT>(p, b, split, lane);  // overlaps tile_view's loads

    TileView tv;
    if (!tile_view<M, NT>(p, b, 0, tv, split == 0)) return;
    if (split >= max(tv.nsplit, 1)) return;
    const bool single = tv.nsplit <= 1;
    const int t_begin = split * p.split_tiles;
    const int n_iter = max(0, min(tv.ntiles, t_begin + p.split_tiles) - t_begin);

    int* row_lo = reinterpret_cast<int*>(smem + C::OFF_ROW);
    int* row_hi = row_lo + M;
    int* row_dg = row_hi + M;
    float* row_ab = reinterpret_cast<float*>(row_dg + M);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* empty = full + STAGES;
    volatile uint32_t* abort_flag = reinterpret_cast<uint32_t*>(smem + C::OFF_FLAG);

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
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], C::PROD);
            mbar_init(&empty[s], C::CONS);
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    // rows and barriers visible to every role; the producers start their loads at once, the
    // consumers stage q meanwhile
    __syncthreads();

    if (warp >= C::CONS) {
        // ---------------- producers: warp pw issues chunks 2 pw and 2 pw + 1 ----------------
        const int pw = warp - C::CONS;
        if (lane == 0 && !p.withhold) {
            const uint64_t policy = l2_policy_evict_first();
            const int c_a = 2 * pw, c_b = 2 * pw + 1;
            const bool has_a = c_a * 64 < p.D, has_b = c_b * 64 < p.D;
            const uint32_t mine = 2u * ((has_a ? 1u : 0u) + (has_b ? 1u : 0u)) * NT * 128u;
            const int kbeg = tv.kt0 + t_begin * NT;
            const int32_t* bt_row = p.paged ? p.bt + (int64_t)b * p.bt_s0 : nullptr;
            auto block_of = [&](int key) {
                return p.paged ? box_block(bt_row, p.bt_cols, p.num_blocks, p.P, key, tv.sk, p.err)
                               : (key < tv.sk ? 0 : -1);
            };
            int blk_next = n_iter > 0 ? block_of(kbeg) : -1;
            for (int it = 0; it < n_iter; ++it) {
                const int stage = it % STAGES;
                const int key = kbeg + it * NT;
                const int blk = blk_next;
                if (it + 1 < n_iter) blk_next = block_of(key + NT);  // looked up while the stage drains
                if (it >= STAGES && !dec_wait(&empty[stage], ((it / STAGES) - 1) & 1, abort_flag, p.err, p.wait_ns))
                    break;
                uint8_t* kst = smem + stage * C::STAGE_BYTES;
                uint8_t* vst = kst + C::TILE_BYTES;
                mbar_arrive_expect_tx(&full[stage], blk >= 0 ? mine : 0u);
                if (blk >= 0 && (has_a || has_b)) {
                    const int c2 = p.paged ? key - (key / p.P) * p.P : p.cu_k[b] + key;
                    const int c3 = p.paged ? blk : 0;
                    if (has_a) {
                        tma_load_4d(kst + c_a * NT * 128, &tm_k, &full[stage], c_a * 64, hk, c2, c3, policy);
                        tma_load_4d(vst + c_a * NT * 128, &tm_v, &full[stage], c_a * 64, hk, c2, c3, policy);
                    }
                    if (has_b) {
                        tma_load_4d(kst + c_b * NT * 128, &tm_k, &full[stage], c_b * 64, hk, c2, c3, policy);
                        tma_load_4d(vst + c_b * NT * 128, &tm_v, &full[stage], c_b * 64, hk, c2, c3, policy);
                    }
                }
            }
        }
        return;  // the consumers synchronise among themselves with named barriers 1..3
    }

    {  // q rows -> the exchange area (128-byte swizzled rows, zero padded), read once below, by
       // the consumer threads, each issuing its loads in batches ahead of their stores
        const T* q = static_cast<const T*>(p.q);
        constexpr int UNITS = DP / 8;
        constexpr int QI = (M * UNITS + C::CONS * 32 - 1) / (C::CONS * 32);
        uint8_t* qs = smem + C::OFF_X;
        constexpr int QB = QI < 4 ? QI : 4;  // loads in flight per batch
#pragma unroll
        for (int j0 = 0; j0 < QI; j0 += QB) {
            int4 val[QB];
#pragma unroll
            for (int j = 0; j < QB; ++j) {
                const int idx = tid + (j0 + j) * (C::CONS * 32);
                const int r = idx / UNITS, u = idx - r * UNITS;
                val[j] = make_int4(0, 0, 0, 0);
                if (idx < M * UNITS && r < tv.rows && u * 8 < p.D) {
                    const int rho = tv.row0 + r;
                    const int i = rho / p.G, g = rho - i * p.G;
                    val[j] = __ldg(reinterpret_cast<const int4*>(q + (int64_t)(tv.q0 + i) * p.q_s0 +
                                                                 (int64_t)(hk * p.G + g) * p.q_s1 + u * 8));
                }
            }
#pragma unroll
            for (int j = 0; j < QB; ++j) {
                const int idx = tid + (j0 + j) * (C::CONS * 32);
                const int r = idx / UNITS, u = idx - r * UNITS;
                if (idx < M * UNITS) *reinterpret_cast<int4*>(qs + (u >> 3) * (M * 128) + swz128(r, u & 7)) = val[j];
            }
        }
    }
    named_barrier_sync(1, C::CONS * 32);  // q staged

    // ---------------- consumers ----------------
    const int dq = warp & 3, grp = warp >> 2;
    const int rg = grp / C::KW, kq = grp % C::KW;
    const int gq = lane >> 2, tq = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;
    const int r0 = rg * 16 + gq, r1 = r0 + 8;  // the two rows this lane holds
    // Key interval every real row of this warp attends: tiles inside it need no mask (the
    // rows' own bounds are read from shared memory only for the tiles that do).  Padding
    // rows (past the tile's rows) are never written and do not restrict it.
    int wlo = INT_MIN, whi = INT_MAX;
    if (r0 < tv.rows) {
        wlo = max(wlo, row_lo[r0]);
        whi = min(whi, row_hi[r0]);
    }
    if (r1 < tv.rows) {
        wlo = max(wlo, row_lo[r1]);
        whi = min(whi, row_hi[r1]);
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        wlo = max(wlo, __shfl_xor_sync(0xffffffffu, wlo, off));
        whi = min(whi, __shfl_xor_sync(0xffffffffu, whi, off));
    }
    if (rg * 16 >= tv.rows) {  // nothing but padding: always masked
        wlo = INT_MAX;
        whi = INT_MIN;
    }

    uint32_t qf[8][4];
    {
        const uint32_t q_base = smem_addr(smem + C::OFF_X);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int row = rg * 16 + rr + ((mi & 1) << 3);
            ldsm_x4(q_base + (dq * 2 + (ks >> 2)) * (M * 128) + swz128(row, (ks & 3) * 2 + (mi >> 1)), qf[ks][0],
                    qf[ks][1], qf[ks][2], qf[ks][3]);
        }
    }
    named_barrier_sync(1, C::CONS * 32);  // Q read by every consumer: the area now holds the exchange

    float o[C::QW / 8][4];
#pragma unroll
    for (int n = 0; n < C::QW / 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    bool stopped = false;
    const int key0 = kq * C::KPW;
    const int kstep_end = min(8, (p.D - dq * C::QW + 15) / 16);  // 16-column steps of this quarter with data

    for (int it = 0; it < n_iter; ++it) {
        const int stage = it % STAGES;
        const bool ok = __all_sync(0xffffffffu, dec_wait(&full[stage], (it / STAGES) & 1, abort_flag, p.err, p.wait_ns));
        const int kt = tv.kt0 + (t_begin + it) * NT;
        uint8_t* kst = smem + stage * C::STAGE_BYTES;
        uint8_t* vst = kst + C::TILE_BYTES;
        const uint32_t xb = smem_addr(smem + C::OFF_X + (it & 1) * C::XBUF_BYTES);
        float pr[4];  // one-slice layout: this warp's probabilities (keys 8 dq + 2 tq, + 1; rows r0, r1)
        float s[C::NSC][4];
#pragma unroll
        for (int n = 0; n < C::NSC; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
        const int valid = tv.sk - kt;
        const bool zeroed = valid < key0 + C::KPW;
        if (ok) {
            // V rows of this warp's keys and columns at or past sk -> 0 (NaN-safe P.V)
            if (zeroed) {
                const int z0 = max(valid, key0), zr = key0 + C::KPW - z0;
                for (int idx = lane; idx < 2 * zr * 8; idx += 32) {
                    const int c = dq * 2 + idx / (zr * 8), rem = idx % (zr * 8);
                    *reinterpret_cast<int4*>(vst + (c * NT + z0 + (rem >> 3)) * 128 + ((rem & 7) << 4)) =
                        make_int4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            // partial scores of this warp's rows and keys over its 128 columns
            const uint32_t k_base = smem_addr(kst);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                if (ks < kstep_end) {
                    const int chunk = dq * 2 + (ks >> 2);
#pragma unroll
                    for (int np = 0; np < C::KPW / 16; ++np) {
                        const int key = key0 + np * 16 + rr + ((mi >> 1) << 3);
                        uint32_t b00, b01, b10, b11;
                        ldsm_x4(k_base + chunk * NT * 128 + swz128(key, (ks & 3) * 2 + (mi & 1)), b00, b01, b10, b11);
                        MmaOp<T>::run(s[2 * np], qf[ks], b00, b01);
                        MmaOp<T>::run(s[2 * np + 1], qf[ks], b10, b11);
                    }
                }
            }
            if constexpr (C::KW == 1) {
                // the partials of the three score tiles other quarters own
#pragma unroll
                for (int n = 0; n < C::NSC; ++n)
                    if (n != dq)
                        st_shared_f4(xb + ((warp * 3 + (n < dq ? n : n - 1)) * 32 + lane) * 16,
                                     make_float4(s[n][0], s[n][1], s[n][2], s[n][3]));
            } else {
#pragma unroll
                for (int n = 0; n < C::NSC; ++n)
                    st_shared_f4(xb + ((warp * C::NSC + n) * 32 + lane) * 16,
                                 make_float4(s[n][0], s[n][1], s[n][2], s[n][3]));
            }
        }
        // every quarter of the group has posted its partial (or one of them gave up)
        if (named_barrier_or(2 + grp, 128, !ok)) {
            stopped = true;
            break;
        }
        if constexpr (C::KW == 1) {
            // score tile dq: the four quarters' partials in quarter order
            float t4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
                float v[4];
                if (w4 == dq) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        v[e] = dq == 0 ? s[0][e] : dq == 1 ? s[1][e] : dq == 2 ? s[2][e] : s[3][e];
                } else {
                    const float4 x = ld_shared_f4(xb + (((grp * 4 + w4) * 3 + (dq < w4 ? dq : dq - 1)) * 32 + lane) * 16);
                    v[0] = x.x;
                    v[1] = x.y;
                    v[2] = x.z;
                    v[3] = x.w;
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) t4[e] += v[e];
            }
            const bool inside = !p.alibi && kt >= wlo && kt + NT - 1 <= whi;
            if (inside) {
#pragma unroll
                for (int e = 0; e < 4; ++e) t4[e] *= p.scale_log2;
            } else {
                const int lo0 = row_lo[r0], hi0 = row_hi[r0], lo1 = row_lo[r1], hi1 = row_hi[r1];
                const int dg0 = row_dg[r0], dg1 = row_dg[r1];
                const float ab0 = row_ab[r0], ab1 = row_ab[r1];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const bool up = e < 2;
                    const int key = kt + dq * 8 + tq * 2 + (e & 1);
                    const bool in = up ? (key >= lo0 && key <= hi0) : (key >= lo1 && key <= hi1);
                    t4[e] = in ? biased_log2(t4[e], p.scale_log2, up ? ab0 : ab1, up ? dg0 : dg1, key) : -INFINITY;
                }
            }
            float mx0 = fmaxf(t4[0], t4[1]), mx1 = fmaxf(t4[2], t4[3]);
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            // probabilities against the current reference, posted with the rows' maxima
            const uint32_t xp = xb + C::XP_OFF + (warp * 32 + lane) * 8;
            const uint32_t xm = xb + C::XM_OFF + (grp * 16 + gq) * 16;
            {
                const float u0 = m0 == -INFINITY ? 0.f : m0, u1 = m1 == -INFINITY ? 0.f : m1;
                pr[0] = fast_exp2(t4[0] - u0);
                pr[1] = fast_exp2(t4[1] - u0);
                pr[2] = fast_exp2(t4[2] - u1);
                pr[3] = fast_exp2(t4[3] - u1);
                st_shared_u2(xp, pack2<T>(pr[0], pr[1]), pack2<T>(pr[2], pr[3]));
                if (tq == 0) {
                    st_shared_f(xm + dq * 4, mx0);
                    st_shared_f(xm + 8 * 16 + dq * 4, mx1);
                }
            }
            named_barrier_sync(2 + grp, 128);
            // every row's maximum over the tile; above the reference by more than 2^8 (or a
            // first finite score): all four quarters raise it, rescale and post P again
            const float4 g0 = ld_shared_f4(xm), g1 = ld_shared_f4(xm + 8 * 16);
            const float n0 = fmaxf(m0, fmaxf(fmaxf(g0.x, g0.y), fmaxf(g0.z, g0.w)));
            const float n1 = fmaxf(m1, fmaxf(fmaxf(g1.x, g1.y), fmaxf(g1.z, g1.w)));
            const bool raise0 = m0 == -INFINITY ? n0 > m0 : n0 > m0 + 8.f;
            const bool raise1 = m1 == -INFINITY ? n1 > m1 : n1 > m1 + 8.f;
            if (__any_sync(0xffffffffu, raise0 || raise1)) {  // the same decision in all four warps
                const float a0 = (n0 == -INFINITY) ? 1.f : fast_exp2(m0 - n0);
                const float a1 = (n1 == -INFINITY) ? 1.f : fast_exp2(m1 - n1);
#pragma unroll
                for (int n = 0; n < C::QW / 8; ++n) {
                    o[n][0] *= a0;
                    o[n][1] *= a0;
                    o[n][2] *= a1;
                    o[n][3] *= a1;
                }
                l0 *= a0;
                l1 *= a1;
                m0 = n0;
                m1 = n1;
                const float u0 = m0 == -INFINITY ? 0.f : m0, u1 = m1 == -INFINITY ? 0.f : m1;
                pr[0] = fast_exp2(t4[0] - u0);
                pr[1] = fast_exp2(t4[1] - u0);
                pr[2] = fast_exp2(t4[2] - u1);
                pr[3] = fast_exp2(t4[3] - u1);
                st_shared_u2(xp, pack2<T>(pr[0], pr[1]), pack2<T>(pr[2], pr[3]));  // no quarter reads P yet
                named_barrier_sync(2 + grp, 128);
            }
            l0 += pr[0] + pr[1];  // this quarter's keys; the quarters' sums are added at the end
            l1 += pr[2] + pr[3];
        } else {
        // full scores: the four partials in quarter order (identical in all four warps)
#pragma unroll
        for (int n = 0; n < C::NSC; ++n) {
            float4 a = ld_shared_f4(xb + (((grp * 4) * C::NSC + n) * 32 + lane) * 16);
#pragma unroll
            for (int w4 = 1; w4 < 4; ++w4) {
                const float4 v = ld_shared_f4(xb + (((grp * 4 + w4) * C::NSC + n) * 32 + lane) * 16);
                a.x += v.x;
                a.y += v.y;
                a.z += v.z;
                a.w += v.w;
            }
            s[n][0] = a.x;
            s[n][1] = a.y;
            s[n][2] = a.z;
            s[n][3] = a.w;
        }
        // scale into the log2 domain, mask by select (unless the tile is inside every row's
        // interval and there is no position bias), and take the row maxima
        const bool inside = !p.alibi && kt + key0 >= wlo && kt + key0 + C::KPW - 1 <= whi;
        if (inside) {
#pragma unroll
            for (int n = 0; n < C::NSC; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[n][e] *= p.scale_log2;
        } else {
            const int lo0 = row_lo[r0], hi0 = row_hi[r0], lo1 = row_lo[r1], hi1 = row_hi[r1];
            const int dg0 = row_dg[r0], dg1 = row_dg[r1];
            const float ab0 = row_ab[r0], ab1 = row_ab[r1];
#pragma unroll
            for (int n = 0; n < C::NSC; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const bool up = e < 2;
                    const int key = kt + key0 + n * 8 + tq * 2 + (e & 1);
                    const bool in = up ? (key >= lo0 && key <= hi0) : (key >= lo1 && key <= hi1);
                    s[n][e] = in ? biased_log2(s[n][e], p.scale_log2, up ? ab0 : ab1, up ? dg0 : dg1, key) : -INFINITY;
                }
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int n = 0; n < C::NSC; ++n) {
            mx0 = max3f(mx0, s[n][0], s[n][1]);
            mx1 = max3f(mx1, s[n][2], s[n][3]);
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
        if (__any_sync(0xffffffffu, n0 > m0 || n1 > m1)) {  // a running max grew: rescale O and l
            const float a0 = (n0 == -INFINITY) ? 1.f : fast_exp2(m0 - n0);
            const float a1 = (n1 == -INFINITY) ? 1.f : fast_exp2(m1 - n1);
#pragma unroll
            for (int n = 0; n < C::QW / 8; ++n) {
                o[n][0] *= a0;
                o[n][1] *= a0;
                o[n][2] *= a1;
                o[n][3] *= a1;
            }
            l0 *= a0;
            l1 *= a1;
            m0 = n0;
            m1 = n1;
        }
        const float u0 = m0 == -INFINITY ? 0.f : m0, u1 = m1 == -INFINITY ? 0.f : m1;
#pragma unroll
        for (int n = 0; n < C::NSC; ++n) {
            s[n][0] = fast_exp2(s[n][0] - u0);
            s[n][1] = fast_exp2(s[n][1] - u0);
            s[n][2] = fast_exp2(s[n][2] - u1);
            s[n][3] = fast_exp2(s[n][3] - u1);
            l0 += s[n][0] + s[n][1];
            l1 += s[n][2] + s[n][3];
        }
        }
        // O += P V over this warp's 128 columns; the score fragments of two n8 tiles are
        // the A fragment of one k16 step
        const uint32_t v_base = smem_addr(vst);
#pragma unroll
        for (int kc = 0; kc < C::KPW / 16; ++kc) {
            uint32_t pa[4];
            if constexpr (C::KW == 1) {  // score tiles 2 kc and 2 kc + 1, as their quarters posted them
                const uint2 x = ld_shared_u2(xb + C::XP_OFF + ((grp * 4 + 2 * kc) * 32 + lane) * 8);
                const uint2 y = ld_shared_u2(xb + C::XP_OFF + ((grp * 4 + 2 * kc + 1) * 32 + lane) * 8);
                pa[0] = x.x;
                pa[1] = x.y;
                pa[2] = y.x;
                pa[3] = y.y;
            } else {
                pa[0] = pack2<T>(s[2 * kc][0], s[2 * kc][1]);
                pa[1] = pack2<T>(s[2 * kc][2], s[2 * kc][3]);
                pa[2] = pack2<T>(s[2 * kc + 1][0], s[2 * kc + 1][1]);
                pa[3] = pack2<T>(s[2 * kc + 1][2], s[2 * kc + 1][3]);
            }
            const int key = key0 + kc * 16 + rr + ((mi & 1) << 3);
#pragma unroll
            for (int np = 0; np < C::QW / 16; ++np) {
                const int d0 = dq * C::QW + np * 16;
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(v_base + (d0 >> 6) * NT * 128 + swz128(key, ((d0 & 63) >> 3) + (mi >> 1)), b0, b1, b2, b3);
                MmaOp<T>::run(o[2 * np], pa, b0, b1);
                MmaOp<T>::run(o[2 * np + 1], pa, b2, b3);
            }
        }
        if (zeroed) fence_proxy_async_smem();  // the stage is rewritten by TMA later
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
    }

    // ---- normalise and write: each warp its own rows and 128 columns, from registers ----
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    // every consumer is done with the stages (reused below); stop together if any role gave up
    if (named_barrier_or(1, C::CONS * 32, stopped || *abort_flag != 0u)) return;
    if constexpr (C::KW == 1) {
        // each quarter summed its own keys' probabilities: the four sums in quarter order
        const uint32_t xl = smem_addr(smem + C::OFF_X) + (grp * 16 + gq) * 16;  // [group][row][quarter]
        if (tq == 0) {
            st_shared_f(xl + dq * 4, l0);
            st_shared_f(xl + 8 * 16 + dq * 4, l1);
        }
        named_barrier_sync(1, C::CONS * 32);
        const float4 a = ld_shared_f4(xl), c = ld_shared_f4(xl + 8 * 16);
        l0 = (a.x + a.y) + (a.z + a.w);
        l1 = (c.x + c.y) + (c.z + c.w);
    }
    if constexpr (C::KW == 2) {
        // 16-row CTA: the warp of the second key half hands its (O, m, l) to the warp of the
        // first, lane for lane (both hold the same rows and columns)
        float4* xo = reinterpret_cast<float4*>(smem);  // [quarter][n8 tile][lane], then [quarter][lane]
        float4* xml = xo + 4 * (C::QW / 8) * 32;
        if (kq == 1) {
#pragma unroll
            for (int n = 0; n < C::QW / 8; ++n)
                xo[(dq * (C::QW / 8) + n) * 32 + lane] = make_float4(o[n][0], o[n][1], o[n][2], o[n][3]);
            xml[dq * 32 + lane] = make_float4(m0, m1, l0, l1);
        }
        named_barrier_sync(1, C::CONS * 32);
        if (kq == 1) return;
        const float4 ml = xml[dq * 32 + lane];
        const float mm0 = fmaxf(m0, ml.x), mm1 = fmaxf(m1, ml.y);
        const float u0 = mm0 == -INFINITY ? 0.f : mm0, u1 = mm1 == -INFINITY ? 0.f : mm1;
        const float fa0 = fast_exp2(m0 - u0), fb0 = fast_exp2(ml.x - u0);
        const float fa1 = fast_exp2(m1 - u1), fb1 = fast_exp2(ml.y - u1);
        l0 = fa0 * l0 + fb0 * ml.z;
        l1 = fa1 * l1 + fb1 * ml.w;
#pragma unroll
        for (int n = 0; n < C::QW / 8; ++n) {
            const float4 ob = xo[(dq * (C::QW / 8) + n) * 32 + lane];
            o[n][0] = fa0 * o[n][0] + fb0 * ob.x;
            o[n][1] = fa0 * o[n][1] + fb0 * ob.y;
            o[n][2] = fa1 * o[n][2] + fb1 * ob.z;
            o[n][3] = fa1 * o[n][3] + fb1 * ob.w;
        }
        m0 = mm0;
        m1 = mm1;
    }
    T* out = static_cast<T*>(p.out);
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int row = hr ? r1 : r0;
        if (row >= tv.rows) continue;
        const float L = hr ? l1 : l0, mm = hr ? m1 : m0;
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const int rho = tv.row0 + row;
        const int i = rho / p.G, g = rho - i * p.G;
        const int64_t t = tv.q0 + i;
        const int h = hk * p.G + g;
        T* orow = out + t * p.o_s0 + (int64_t)h * p.o_s1;
        float* prow = p.part_o + ((int64_t)split * p.part_stride + t * p.H + h) * p.D;
#pragma unroll
        for (int n = 0; n < C::QW / 8; ++n) {
            const int d = dq * C::QW + n * 8 + tq * 2;
            if (d >= p.D) continue;
            const float x0 = o[n][hr * 2] * inv, x1 = o[n][hr * 2 + 1] * inv;
            if (single)
                *reinterpret_cast<uint32_t*>(orow + d) = pack2<T>(x0, x1);
            else
                *reinterpret_cast<float2*>(prow + d) = make_float2(x0, x1);
        }
        if (dq == 0 && tq == 0) {
            const float lse = L > 0.f ? (mm + log2f(L)) * 0.69314718055994531f : -INFINITY;
            if (single)
                p.lse[(int64_t)h * p.lse_s0 + t + (int64_t)b * p.lse_sb] = lse;
            else
                p.part_lse[(int64_t)split * p.part_stride + t * p.H + h] = lse;
        }
    }
}

}  // namespace pa
