// Decode-class paged attention kernel with warp-private key slices.
//
// One CTA owns one (sequence, kv head, key split) with at most 32 query rows (the
// (query, head) pairs of the GQA group, ordered i * G + g).  Warp 4 is the producer:
// it walks the block table and issues TMA loads of K/V tiles into a ring of
// shared-memory stages (full/empty mbarriers).  Warps 0..3 consume: warp w takes row
// group w / KW and the w % KW-th slice of every tile's keys, computes its scores with
// mma.sync, runs the online softmax inside the warp (quad shuffles only), feeds P from
// registers straight into the P.V mma, and releases the stage.  No CTA-wide barrier
// runs inside the key loop; the per-warp (max, sum, O) triples are merged once at the
// end through shared memory, each warp of a row group merging and storing a share of the
// columns.
#pragma once

#include "splitkv_kernel.cuh"

namespace pa {

constexpr int kDecodeThreads = 160;  // 4 consumer warps + 1 producer warp

// ML: the row groups the shared-memory layout is sized for (>= MG).  A kernel built for two
// row groups runs units of at most 16 rows with the one-group body (MG = 1) in its own
// layout (ML = 2), so that the barriers and the ring it set up stay where they are.
template <int DP, int MG, int NT, int STAGES, int ML = MG>
struct DecCfg {
    static constexpr int M = 16 * MG;        // rows per CTA
    static constexpr int KW = 4 / MG;        // warps sharing one row group (key-slice ways)
    static constexpr int KPW = NT / KW;      // keys per warp per tile
    static constexpr int CH = DP / 64;
    static constexpr int TILE_BYTES = CH * NT * 128;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int Q_BYTES = CH * 16 * ML * 128;
    static constexpr int OFF_Q = STAGES * STAGE_BYTES;
    static constexpr int OFF_ROW = OFF_Q + Q_BYTES;            // row_lo[M], row_hi[M], row_dg[M], row_ab[M]
    static constexpr int OFF_BAR = (OFF_ROW + 4 * (16 * ML) * 4 + 15) & ~15;
    static constexpr int OFF_FLAG = OFF_BAR + 2 * STAGES * 8;
    static constexpr int OFF_IDS = OFF_FLAG + 16;              // block id of every TMA box of the split
    static constexpr int MAX_BOXES = 512;
    static constexpr int SMEM = OFF_IDS + MAX_BOXES * 4 + 1024;
    static constexpr int MERGE_BYTES = 4 * (DP / 8) * 32 * 16 + 4 * 32 * 16;  // O, m, l of every warp, in the stages
    static constexpr bool Q_IN_REGS = DP <= 128;
    static_assert(KPW % 16 == 0, "keys per warp");
    static_assert(MERGE_BYTES <= STAGES * STAGE_BYTES, "merge scratch");
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

__device__ __forceinline__ bool dec_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
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

// The work of one (sequence b, kv head hk, key split) on a CTA: its rows' bounds and q into
// shared memory, then the producer warp and the four consumer warps.  `g0` is the number of
// key tiles the CTA's ring has carried before (ring stage and phase continue from it);
// `n_done` returns the tiles of this unit (the same in every thread).  Every thread returns
// from here: early (no work, uniformly), when its role ends, or after the epilogue.
template <typename T, int DP, int MG, int NT, int STAGES, int ML = MG>
__device__ __forceinline__ void decode_unit(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const SplitParams& p,
                                            uint8_t* smem, int b, int hk, int split, int g0, int& n_done) {
    using C = DecCfg<DP, MG, NT, STAGES, ML>;
    constexpr int M = C::M;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    TileView tv;
    n_done = 0;
    if (!tile_view<M, NT>(p, b, 0, tv, split == 0)) return;
    if (split >= max(tv.nsplit, 1)) return;
    const bool single = tv.nsplit <= 1;
    const int t_begin = split * p.split_tiles;
    const int n_iter = max(0, min(tv.ntiles, t_begin + p.split_tiles) - t_begin);
    n_done = n_iter;

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
    // rows (and, for a CTA's first unit, the barrier set-up) visible to every role; the
    // producer starts its loads at once, the consumers stage q meanwhile
    __syncthreads();

    if (warp == 4) {
        // ---------------- producer ----------------
        // physical block of every box of this split's key range, looked up once
        int* ids = reinterpret_cast<int*>(smem + C::OFF_IDS);
        const int kbeg = tv.kt0 + t_begin * NT;
        const int n_boxes = min(n_iter * p.boxes_per_tile, C::MAX_BOXES);
        const int32_t* bt_row = p.paged ? p.bt + (int64_t)b * p.bt_s0 : nullptr;
        for (int bi = lane; bi < n_boxes; bi += 32) {
            const int key = kbeg + bi * p.box_rows;
            ids[bi] = p.paged ? box_block(bt_row, p.bt_cols, p.num_blocks, p.P, key, tv.sk, p.err)
                              : (key < tv.sk ? 0 : -1);
        }
        __syncwarp();
        if (lane == 0 && !p.withhold) {
            const uint64_t policy = l2_policy_evict_first();
            for (int it = 0; it < n_iter; ++it) {
                const int gi = g0 + it;  // position in the CTA's stream of tiles
                const int stage = gi % STAGES;
                if (gi >= STAGES && !dec_wait(&empty[stage], ((gi / STAGES) - 1) & 1, abort_flag, p.err, p.wait_ns)) break;
                const int kt = kbeg + it * NT;
                uint8_t* kst = smem + stage * C::STAGE_BYTES;
                uint8_t* vst = kst + C::TILE_BYTES;
                int blk[2];  // a 64-key tile is at most two 32-row boxes
                uint32_t bytes = 0;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int bi = it * p.boxes_per_tile + j;
                    const int key = kt + j * p.box_rows;
                    blk[j] = j >= p.boxes_per_tile ? -1
                             : bi < C::MAX_BOXES ? ids[bi]
                             : (p.paged ? box_block(bt_row, p.bt_cols, p.num_blocks, p.P, key, tv.sk, p.err)
                                        : (key < tv.sk ? 0 : -1));
                    if (blk[j] >= 0) bytes += 2u * C::CH * p.box_rows * 128u;
                }
                mbar_arrive_expect_tx(&full[stage], bytes);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    if (blk[j] < 0) continue;
                    const int key = kt + j * p.box_rows;
                    const int c2 = p.paged ? key - (key / p.P) * p.P : p.cu_k[b] + key;
                    const int c3 = p.paged ? blk[j] : 0;
                    for (int c = 0; c < C::CH; ++c) {
                        const int off = (c * NT + j * p.box_rows) * 128;
                        tma_load_4d(kst + off, &tm_k, &full[stage], c * 64, hk, c2, c3, policy);
                        tma_load_4d(vst + off, &tm_v, &full[stage], c * 64, hk, c2, c3, policy);
                    }
                }
            }
        }
        return;  // the consumers synchronise among themselves with named barrier 1
    }

    {  // q rows -> shared memory (128-byte swizzled rows, zero padded), by the 128 consumer
       // threads, each issuing its loads in batches ahead of their stores
        const T* q = static_cast<const T*>(p.q);
        constexpr int UNITS = DP / 8;
        constexpr int QI = (M * UNITS + 127) / 128;
        constexpr int QB = QI < 4 ? QI : 4;
        uint8_t* qs = smem + C::OFF_Q;
#pragma unroll
        for (int j0 = 0; j0 < QI; j0 += QB) {
            int4 val[QB];
#pragma unroll
            for (int j = 0; j < QB; ++j) {
                const int idx = tid + (j0 + j) * 128;
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
                const int idx = tid + (j0 + j) * 128;
                const int r = idx / UNITS, u = idx - r * UNITS;
                if (idx < M * UNITS) *reinterpret_cast<int4*>(qs + (u >> 3) * (M * 128) + swz128(r, u & 7)) = val[j];
            }
        }
    }
    named_barrier_sync(1, 128);  // q staged

    // ---------------- consumers ----------------
    const int rg = warp / C::KW, kq = warp % C::KW;
    const int gq = lane >> 2, tq = lane & 3;
    const int mi = lane >> 3, rr = lane & 7;
    const int r0 = rg * 16 + gq, r1 = r0 + 8;  // the two rows this lane holds
    const int lo0 = row_lo[r0], hi0 = row_hi[r0], lo1 = row_lo[r1], hi1 = row_hi[r1];
    const int dg0 = row_dg[r0], dg1 = row_dg[r1];
    const float ab0 = row_ab[r0], ab1 = row_ab[r1];
    const uint32_t q_base = smem_addr(smem + C::OFF_Q);

    uint32_t qf[C::Q_IN_REGS ? DP / 16 : 1][4];
    if constexpr (C::Q_IN_REGS) {
#pragma unroll
        for (int ks = 0; ks < DP / 16; ++ks) {
            const int row = rg * 16 + rr + ((mi & 1) << 3);
            ldsm_x4(q_base + (ks >> 2) * (M * 128) + swz128(row, (ks & 3) * 2 + (mi >> 1)), qf[ks][0], qf[ks][1],
                    qf[ks][2], qf[ks][3]);
        }
    }

    float o[DP / 8][4];
#pragma unroll
    for (int n = 0; n < DP / 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    bool ok = true;

    for (int it = 0; it < n_iter; ++it) {
        const int gi = g0 + it;
        const int stage = gi % STAGES;
        ok = __all_sync(0xffffffffu, dec_wait(&full[stage], (gi / STAGES) & 1, abort_flag, p.err, p.wait_ns));
        if (!ok) break;
        const int kt = tv.kt0 + (t_begin + it) * NT;
        uint8_t* kst = smem + stage * C::STAGE_BYTES;
        uint8_t* vst = kst + C::TILE_BYTES;
        const int key0 = kq * C::KPW;
        // V rows of this warp's slice at or past sk -> 0 (NaN-safe P.V)
        const int valid = tv.sk - kt;
        const bool zeroed = valid < key0 + C::KPW;
        if (zeroed) {
            const int z0 = max(valid, key0), zr = key0 + C::KPW - z0;
            for (int idx = lane; idx < C::CH * zr * 8; idx += 32) {
                const int c = idx / (zr * 8), rem = idx - c * zr * 8;
                *reinterpret_cast<int4*>(vst + (c * NT + z0 + (rem >> 3)) * 128 + ((rem & 7) << 4)) =
                    make_int4(0, 0, 0, 0);
            }
            __syncwarp();
        }
        const uint32_t k_base = smem_addr(kst), v_base = smem_addr(vst);
#pragma unroll
        for (int kc = 0; kc < C::KPW / 16; ++kc) {
            const int kk0 = key0 + kc * 16;
            float s[2][4];
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < DP / 16; ++ks) {
                uint32_t b00, b01, b10, b11;
                const int key = kk0 + rr + ((mi >> 1) << 3);
                ldsm_x4(k_base + (ks >> 2) * NT * 128 + swz128(key, (ks & 3) * 2 + (mi & 1)), b00, b01, b10, b11);
                uint32_t af[4];
                if constexpr (C::Q_IN_REGS) {
                    af[0] = qf[ks][0];
                    af[1] = qf[ks][1];
                    af[2] = qf[ks][2];
                    af[3] = qf[ks][3];
                } else {
                    const int row = rg * 16 + rr + ((mi & 1) << 3);
                    ldsm_x4(q_base + (ks >> 2) * (M * 128) + swz128(row, (ks & 3) * 2 + (mi >> 1)), af[0], af[1], af[2],
                            af[3]);
                }
                MmaOp<T>::run(s[0], af, b00, b01);
                MmaOp<T>::run(s[1], af, b10, b11);
            }
            // scale into the log2 domain, mask by select, and take the row maxima
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = kt + kk0 + n * 8 + tq * 2 + (e & 1);
                    const bool up = e < 2;
                    const bool in = up ? (key >= lo0 && key <= hi0) : (key >= lo1 && key <= hi1);
                    s[n][e] = in ? biased_log2(s[n][e], p.scale_log2, up ? ab0 : ab1, up ? dg0 : dg1, key) : -INFINITY;
                    if (up)
                        mx0 = fmaxf(mx0, s[n][e]);
                    else
                        mx1 = fmaxf(mx1, s[n][e]);
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
                for (int n = 0; n < DP / 8; ++n) {
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
            float pv[2][4];
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                pv[n][0] = fast_exp2(s[n][0] - u0);
                pv[n][1] = fast_exp2(s[n][1] - u0);
                pv[n][2] = fast_exp2(s[n][2] - u1);
                pv[n][3] = fast_exp2(s[n][3] - u1);
                l0 += pv[n][0] + pv[n][1];
                l1 += pv[n][2] + pv[n][3];
            }
            // the score fragment of two n8 tiles is the A fragment of a k16 step
            uint32_t pa[4];
            pa[0] = pack2<T>(pv[0][0], pv[0][1]);
            pa[1] = pack2<T>(pv[0][2], pv[0][3]);
            pa[2] = pack2<T>(pv[1][0], pv[1][1]);
            pa[3] = pack2<T>(pv[1][2], pv[1][3]);
#pragma unroll
            for (int np = 0; np < DP / 16; ++np) {
                const int d0 = np * 16;
                const int key = kk0 + rr + ((mi & 1) << 3);
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

    // ---- merge the KW key slices of each row group, then write ----
    // Every warp leaves its (O, m, l) in shared memory lane for lane; warp kq of a row group
    // then merges the KW slices of the kq-th share of the columns and stores them.
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    // every consumer is done with the stages (reused below); stop together if any role gave up
    if (named_barrier_or(1, 128, !ok || *abort_flag != 0u)) return;
    float4* xo = reinterpret_cast<float4*>(smem);  // [warp][n8 tile][lane]
    float4* xml = xo + 4 * (DP / 8) * 32;          // [warp][lane]: m0, m1, l0, l1
#pragma unroll
    for (int n = 0; n < DP / 8; ++n) xo[(warp * (DP / 8) + n) * 32 + lane] = make_float4(o[n][0], o[n][1], o[n][2], o[n][3]);
    xml[warp * 32 + lane] = make_float4(m0, m1, l0, l1);
    named_barrier_sync(1, 128);

    float f0[C::KW], f1[C::KW];
    float L0 = 0.f, L1 = 0.f, mm0 = -INFINITY, mm1 = -INFINITY;
#pragma unroll
    for (int k = 0; k < C::KW; ++k) {
        const float4 ml = xml[(rg * C::KW + k) * 32 + lane];
        mm0 = fmaxf(mm0, ml.x);
        mm1 = fmaxf(mm1, ml.y);
    }
    {
        const float u0 = mm0 == -INFINITY ? 0.f : mm0, u1 = mm1 == -INFINITY ? 0.f : mm1;
#pragma unroll
        for (int k = 0; k < C::KW; ++k) {
            const float4 ml = xml[(rg * C::KW + k) * 32 + lane];
            f0[k] = fast_exp2(ml.x - u0);
            f1[k] = fast_exp2(ml.y - u1);
            L0 += f0[k] * ml.z;
            L1 += f1[k] * ml.w;
        }
    }
    const float inv0 = L0 > 0.f ? 1.f / L0 : 0.f, inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
    constexpr int NPW = (DP / 8) / C::KW;  // n8 column tiles this warp stores
    T* out = static_cast<T*>(p.out);
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int row = hr ? r1 : r0;
        if (row >= tv.rows) continue;
        const int rho = tv.row0 + row;
        const int i = rho / p.G, g = rho - i * p.G;
        const int64_t t = tv.q0 + i;
        const int h = hk * p.G + g;
        T* orow = out + t * p.o_s0 + (int64_t)h * p.o_s1;
        float* prow = p.part_o + ((int64_t)split * p.part_stride + t * p.H + h) * p.D;
        const float inv = hr ? inv1 : inv0;
#pragma unroll
        for (int nn = 0; nn < NPW; ++nn) {
            const int n = kq * NPW + nn;
            const int d = n * 8 + tq * 2;
            if (d >= p.D) continue;
            float x0 = 0.f, x1 = 0.f;
#pragma unroll
            for (int k = 0; k < C::KW; ++k) {
                const float4 ov = xo[((rg * C::KW + k) * (DP / 8) + n) * 32 + lane];
                const float f = hr ? f1[k] : f0[k];
                x0 += f * (hr ? ov.z : ov.x);
                x1 += f * (hr ? ov.w : ov.y);
            }
            if (single)
                *reinterpret_cast<uint32_t*>(orow + d) = pack2<T>(x0 * inv, x1 * inv);
            else
                *reinterpret_cast<float2*>(prow + d) = make_float2(x0 * inv, x1 * inv);
        }
        if (kq == 0 && tq == 0) {
            const float L = hr ? L1 : L0, mm = hr ? mm1 : mm0;
            const float lse = L > 0.f ? (mm + log2f(L)) * 0.69314718055994531f : -INFINITY;
            if (single)
                p.lse[(int64_t)h * p.lse_s0 + t + (int64_t)b * p.lse_sb] = lse;
            else
                p.part_lse[(int64_t)split * p.part_stride + t * p.H + h] = lse;
        }
    }
}

// Resident CTAs per SM the register bound keeps possible: three at head dim 64, two at 128
// (as many as the shared memory allows), one at 256.
template <typename T, int DP, int MG, int NT, int STAGES>
__global__ void __launch_bounds__(kDecodeThreads, DP <= 64 ? 3 : DP <= 128 ? 2 : 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                     const __grid_constant__ CUtensorMap tm_v,
                                                     const SplitParams p) {
    using C = DecCfg<DP, MG, NT, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x;
    allow_dependent_launch();
    if (tid == 128) {  // the producer lane: descriptors on their way at once
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* empty = full + STAGES;
    volatile uint32_t* abort_flag = reinterpret_cast<uint32_t*>(smem + C::OFF_FLAG);
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 4);
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    // A two-group kernel (the plan's bound on rows was above 16) runs the units of sequences
    // with at most 16 rows on the one-group body: its four warps split each tile's keys in
    // quarters instead of leaving two warps on padding rows (decode rows of the mixed batch:
    // 321 -> 293 us).  Both bodies see the same key interval and split count for such a unit.
    auto run_unit = [&](int b, int hk, int split, int g0, int& n_done) {
        if constexpr (MG == 2) {
            // the one-group body must find the barriers, flag and ids where this kernel put them
            using L1 = DecCfg<DP, 1, NT, STAGES, 2>;
            static_assert(L1::OFF_Q == C::OFF_Q && L1::OFF_ROW == C::OFF_ROW && L1::OFF_BAR == C::OFF_BAR &&
                              L1::OFF_FLAG == C::OFF_FLAG && L1::OFF_IDS == C::OFF_IDS && L1::SMEM == C::SMEM,
                          "both bodies share one shared-memory layout");
            if (b >= 0 && b < p.batch && (int64_t)(p.cu_q[b + 1] - p.cu_q[b]) * p.G <= 16) {
                decode_unit<T, DP, 1, NT, STAGES, 2>(tm_k, tm_v, p, smem, b, hk, split, g0, n_done);
                return;
            }
        }
        decode_unit<T, DP, MG, NT, STAGES, MG>(tm_k, tm_v, p, smem, b, hk, split, g0, n_done);
    };
    if (p.work) {
        // Persistent: the CTA takes (sequence, split) x kv head items in list order (longest
        // sequences first) until none is left; the stage ring carries on from item to item.
        __shared__ int s_item;
        const int total = p.work[1] * p.Hkv;
        int g0 = 0;
        for (;;) {
            if (tid == 0) s_item = atomicAdd(p.work, 1);
            __syncthreads();  // also orders the barrier set-up before the first item
            const int w = s_item;
            if (w >= total) break;
            const int pair = w / p.Hkv;
            int n_done = 0;
            run_unit(p.work[2 + 2 * pair], w - pair * p.Hkv, p.work[3 + 2 * pair], g0, n_done);
            // every role is done with the item (its stages, q and rows); the epilogue's
            // shared-memory writes are ordered before the next item's TMA writes to the stages
            fence_proxy_async_smem();
            __syncthreads();
            if (*abort_flag) break;
            g0 += n_done;
        }
        return;
    }
    // Sequences longest first (ties by index): their CTAs start first and the short ones
    // fill the tail of the grid.  Small batches are ranked here, one sequence per thread;
    // larger ones come with an order from a ranking pass.
    __shared__ int rank_len[kDecodeThreads];
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
    if (tid >= 128) prefetch_split_pages<NT>(p, b, (int)blockIdx.x, tid - 128);  // overlaps tile_view's loads
    int n_done = 0;
    run_unit(b, (int)blockIdx.y % p.Hkv, (int)blockIdx.x, 0, n_done);
}

}  // namespace pa
