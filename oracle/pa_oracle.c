/*
 * Oracle for paged-KV varlen attention (forward) -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may load
 * this file's library.  It is a plain, slow, fp64 CPU restatement of what the
 * attention path computes, written so a reader can check it by eye against the
 * definitions below.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * Sources (the candle error-explanation pages, huggingface/candle@d5fee525bf):
 *  - "flash-attn-varlen expects input tensors of rank 3", Source: q is the
 *    packed varlen tensor (total_q, num_heads, head_dim); non-paged k/v are
 *    (total_k, num_heads_k, head_dim).
 *  - "flash-attn-varlen paged expects k/v tensors of rank 4", What it means:
 *    paged k/v are (num_blocks, page_block_size, num_heads_k, head_dim), and a
 *    block_table maps each sequence's logical pages to physical blocks.
 *  - "paged flash-attn requires page_block_size", Source: the page size is the
 *    second dimension of the rank-4 cache.
 *  The pages do not write out the attention arithmetic or the mask; this file
 *  takes the plain definitions stated at each function below.
 *
 * Readings taken where the pages are silent:
 *  - seqlens are cumulative int32 offsets of length batch+1 (cu[0] = 0); in
 *    paged mode only sk_b = cu_k[b+1] - cu_k[b] is used and the keys of
 *    sequence b are logical positions 0 .. sk_b-1 of block_table row b.
 *  - query head h reads kv head h / (num_heads / num_heads_k).
 *  - the mask is bottom-right aligned with inclusive window bounds; a negative
 *    window side is unbounded; causal is (window_left, window_right) = (-1, 0).
 *  - a row with no attended key gives out = 0 and lse = -inf.
 *  - lse is the natural log of sum_j exp(s_j) over the attended keys.
 *  - alibi_slopes: the pages name the argument only through its shape check
 *    ("shape mismatch alibi_slopes {:?}, expected {:?}" among the related errors of
 *    "paged flash-attn requires page_block_size to be a multiple of 32" and of "flash-attn-
 *    varlen paged expects k/v tensors of rank 4").  The reading taken is the usual
 *    linear-bias definition: one fp32 slope per query head, and the score of query i
 *    and key j is shifted by -slope_h * |i + sk - sq - j|, the distance to the query's
 *    bottom-right aligned diagonal.
 *
 * All arithmetic is IEEE binary64 on the exact fp16 / bf16 input values, in two
 * passes (scores and their maximum first, then the exponentials), with no
 * blocking, online rescaling or reordering.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1 };

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Written from the format's definition. */
static double decode_f16(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24);          /* subnormal: frac * 2^-14 * 2^-10 */
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp((double)(frac | 0x400), expo - 25); /* (1.frac) * 2^(expo-15) */
    }
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE 754 binary32 word. */
static double decode_bf16(uint16_t bits) {
    uint32_t word = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

static double decode(int dtype, uint16_t bits) {
    return dtype == ORACLE_F16 ? decode_f16(bits) : decode_bf16(bits);
}

/* Mask definition (bottom-right aligned): with c = sk - sq, query i of a
 * sequence attends key j iff 0 <= j < sk, and j >= i + c - wl when wl >= 0,
 * and j <= i + c + wr when wr >= 0.  Causal attention is (wl, wr) = (-1, 0). */
static int attends(int64_t i, int64_t j, int64_t sq, int64_t sk, int wl, int wr) {
    int64_t c = sk - sq;
    if (j < 0 || j >= sk) return 0;
    if (wl >= 0 && j < i + c - wl) return 0;
    if (wr >= 0 && j > i + c + wr) return 0;
    return 1;
}

/* Linear position bias (the reading above): -slope * |i + sk - sq - j|. */
static double alibi_bias(double slope, int64_t i, int64_t j, int64_t sq, int64_t sk) {
    int64_t c = sk - sq;
    return -slope * fabs((double)(i + c - j));
}

/* Address of key (or value) row j of sequence b, kv head hk.
 * Paged: logical page j / P of row b of the block table names the physical
 * block; the row sits at slot j mod P of that block.
 * Non-paged: the row is token cu_k[b] + j of the packed (total_k, Hkv, D) tensor. */
static const uint16_t* kv_row(const uint16_t* base, const int64_t* s, int paged,
                              const int32_t* block_table, int64_t bt_row_stride,
                              int page_block_size, const int32_t* cu_k,
                              int64_t b, int64_t j, int64_t hk) {
    if (paged) {
        int64_t block = block_table[b * bt_row_stride + j / page_block_size];
        return base + block * s[0] + (j % page_block_size) * s[1] + hk * s[2];
    }
    return base + ((int64_t)cu_k[b] + j) * s[0] + hk * s[1];
}

int pa_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * out[r, :] and lse[r] for each requested (token, head) row r:
 *   J    = { j : attends(i, j) }                      (i = token - cu_q[b])
 *   s_j  = softmax_scale * sum_d q[token, h, d] * K_j[d]  (+ alibi_bias(slope_h, i, j) when
 *          alibi_slopes is given)
 *   m    = max_{j in J} s_j,   l = sum_{j in J} exp(s_j - m)
 *   out  = sum_{j in J} exp(s_j - m) * V_j / l,   lse = m + ln(l)
 *
 * Arguments (element strides; the last dimension of every tensor is contiguous):
 *   q, q_stride[2]        (total_q, H, D) token and head strides
 *   k, v, kv_stride[3]    paged: (block, slot, head) strides of (NB, P, Hkv, D)
 *                         non-paged: (token, head) strides of (total_k, Hkv, D)
 *   cu_q, cu_k            int32 [batch + 1]
 *   block_table           int32 [batch, bt_row_stride-spaced rows], NULL = non-paged
 *   alibi_slopes          double [H] (one slope per query head), or NULL for no bias
 *   rows                  int64 [n_rows] of token * H + head, or NULL for all rows
 *   out                   double [n_rows, D] (or [total_q * H, D])
 *   lse                   double [n_rows]
 * Returns 0, or -1 on an argument it cannot use.
 */
int pa_oracle_fwd(int dtype,
                  const uint16_t* q, const int64_t* q_stride,
                  const uint16_t* k, const uint16_t* v, const int64_t* kv_stride,
                  const int32_t* cu_q, const int32_t* cu_k, int64_t batch,
                  const int32_t* block_table, int64_t bt_row_stride, int page_block_size,
                  int64_t num_heads, int64_t num_heads_k, int64_t head_dim,
                  double softmax_scale, int window_left, int window_right,
                  const double* alibi_slopes,
                  const int64_t* rows, int64_t n_rows,
                  double* out, double* lse) {
    if (dtype != ORACLE_F16 && dtype != ORACLE_BF16) return -1;
    if (num_heads_k <= 0 || num_heads % num_heads_k != 0 || head_dim <= 0) return -1;
    int paged = block_table != NULL;
    if (paged && page_block_size <= 0) return -1;
    int64_t total_q = cu_q[batch];
    int64_t all_rows = total_q * num_heads;
    int64_t n = rows ? n_rows : all_rows;
    int64_t group = num_heads / num_heads_k;

    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t r = 0; r < n; ++r) {
        int64_t row = rows ? rows[r] : r;
        if (row < 0 || row >= all_rows) { bad = 1; continue; }
        int64_t token = row / num_heads, h = row % num_heads, hk = h / group;
        int64_t b = 0;
        while (!(cu_q[b] <= token && token < cu_q[b + 1])) ++b; /* the sequence holding token */
        int64_t i = token - cu_q[b];
        int64_t sq = cu_q[b + 1] - cu_q[b];
        int64_t sk = (int64_t)cu_k[b + 1] - cu_k[b];
        const uint16_t* qrow = q + token * q_stride[0] + h * q_stride[1];
        double* o = out + r * head_dim;

        double* score = (double*)malloc(sizeof(double) * (size_t)(sk > 0 ? sk : 1));
        /* pass 1: scores of attended keys and their maximum */
        double m = -INFINITY;
        int64_t attended = 0;
        for (int64_t j = 0; j < sk; ++j) {
            if (!attends(i, j, sq, sk, window_left, window_right)) continue;
            const uint16_t* krow = kv_row(k, kv_stride, paged, block_table, bt_row_stride,
                                          page_block_size, cu_k, b, j, hk);
            double dot = 0.0;
            for (int64_t d = 0; d < head_dim; ++d) dot += decode(dtype, qrow[d]) * decode(dtype, krow[d]);
            score[j] = softmax_scale * dot;
            if (alibi_slopes) score[j] += alibi_bias(alibi_slopes[h], i, j, sq, sk);
            if (score[j] > m) m = score[j];
            ++attended;
        }
        for (int64_t d = 0; d < head_dim; ++d) o[d] = 0.0;
        if (attended == 0) {
            lse[r] = -INFINITY;
            free(score);
            continue;
        }
        /* pass 2: exponentials, their sum, and the weighted sum of value rows */
        double l = 0.0;
        for (int64_t j = 0; j < sk; ++j) {
            if (!attends(i, j, sq, sk, window_left, window_right)) continue;
            const uint16_t* vrow = kv_row(v, kv_stride, paged, block_table, bt_row_stride,
                                          page_block_size, cu_k, b, j, hk);
            double w = exp(score[j] - m);
            l += w;
            for (int64_t d = 0; d < head_dim; ++d) o[d] += w * decode(dtype, vrow[d]);
        }
        for (int64_t d = 0; d < head_dim; ++d) o[d] /= l;
        lse[r] = m + log(l);
        free(score);
    }
    return bad ? -1 : 0;
}

/* Exposed so the tests can compare the format decoders against numpy / torch. */
double pa_oracle_decode(int dtype, uint16_t bits) { return decode(dtype, bits); }
