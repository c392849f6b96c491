/*
 * pa_varlen.h -- C ABI of the GB300 (sm_103a) paged-KV varlen flash-attention
 * forward library (libpa_varlen.so).
 *
 * The operation is the forward pass of variable-length attention over a paged
 * KV cache, as validated by candle-flash-attn's varlen wrapper
 * (huggingface/candle@d5fee525bf, as explained by the pages
 * "flash-attn-varlen expects input tensors of rank 3",
 * "flash-attn-varlen paged expects k/v tensors of rank 4",
 * "paged flash-attn requires page_block_size",
 * "page_block_size ... does not match k shape" and
 * "paged flash-attn requires page_block_size to be a multiple of 32").
 *
 * For every sequence b, query head h (kv head hk = h / (num_heads/num_heads_k))
 * and query i < sq_b, with sq_b = cu_seqlens_q[b+1]-cu_seqlens_q[b],
 * sk_b = cu_seqlens_k[b+1]-cu_seqlens_k[b] and c_b = sk_b - sq_b:
 *   J      = { j in [0, sk_b) : (wl < 0 or j >= i+c_b-wl) and (wr < 0 or j <= i+c_b+wr) }
 *   s_j    = softmax_scale * q[cu_q[b]+i, h, :] . K_j,
 *            K_j = k_cache[block_table[b, j / P], j mod P, hk, :] (paged)
 *   out    = sum_{j in J} softmax(s)_j V_j   (rounded to the input dtype)
 *   lse    = ln sum_{j in J} exp(s_j)          (fp32; -inf and out = 0 when J is empty)
 * Causal attention is (window_left, window_right) = (-1, 0), aligned to the
 * bottom-right corner of each sequence's (sq_b x sk_b) score matrix.
 *
 * Everything runs asynchronously on the caller's CUDA stream; no call reads
 * device memory on the host or synchronises, except pa_device_status().
 */
#ifndef PA_VARLEN_H
#define PA_VARLEN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types of a tensor descriptor. */
typedef enum pa_dtype { PA_F16 = 0, PA_BF16 = 1, PA_F32 = 2, PA_I32 = 3 } pa_dtype;

/* A borrowed strided tensor: `data` is a device address (the caller owns it and
 * keeps it alive until the stream has finished the call); `shape` and `stride`
 * hold `ndim` (1..4) entries; strides are in elements, not bytes. */
typedef struct pa_tensor {
    void* data;
    int32_t dtype;  /* pa_dtype */
    int32_t ndim;
    int64_t shape[4];
    int64_t stride[4];
} pa_tensor;

/* Status codes.  The messages (pa_last_error) word the page conditions the
 * way candle's wrapper words them. */
enum {
    PA_OK = 0,
    PA_ERR_RANK = 1,            /* q not rank 3, or non-paged k/v not rank 3
                                   ("flash-attn-varlen expects input tensors of rank 3", Source) */
    PA_ERR_RANK_PAGED = 2,      /* paged and k/v not rank 4
                                   ("flash-attn-varlen paged expects k/v tensors of rank 4", Source) */
    PA_ERR_NONCONTIG = 3,       /* last dim of q/k/v (or an index tensor) not contiguous
                                   (same Source; "Related errors" of the page-size pages) */
    PA_ERR_SHAPE = 4,           /* k vs v shape, or k head size vs q head size
                                   ("paged flash-attn requires page_block_size", Source) */
    PA_ERR_PAGE_UNSET = 5,      /* paged and page_block_size <= 0
                                   ("paged flash-attn requires page_block_size") */
    PA_ERR_PAGE_MISMATCH = 6,   /* page_block_size != k_cache.shape[1]
                                   ("page_block_size ... does not match k shape") */
    PA_ERR_PAGE_MULT32 = 7,     /* page_block_size % 32 != 0
                                   ("paged flash-attn requires page_block_size to be a multiple of 32") */
    PA_ERR_HEADDIM = 8,         /* head_dim > 512 (same Source: "supports head sizes up to 512") */
    PA_ERR_NOT_DEVICE = 9,      /* a tensor is not in device memory ("block_table must be a cuda
                                   tensor", "seqlens_k must be a cuda tensor": Related errors) */
    PA_ERR_ARG = 10,            /* a scalar disagrees with a descriptor, dtype mismatch, H % Hkv != 0,
                                   bad out/lse/index shapes, block table too narrow for max_seqlen_k */
    PA_ERR_UNSUPPORTED = 11,    /* an implementation limit, not a page condition: head_dim not a
                                   multiple of 8, a stride or address not 16-byte aligned */
    PA_ERR_CUDA = 12,           /* a CUDA runtime call or launch failed */
    PA_ERR_DEVICE_TIMEOUT = 13, /* (pa_device_status) a kernel gave up a bounded wait */
    PA_ERR_DEVICE_BOUNDS = 14,  /* (pa_device_status) a kernel saw a block id outside [0, num_blocks),
                                   a page past the block table, non-monotone cu_seqlens, or a
                                   sequence longer than max_seqlen_q / max_seqlen_k; the offending
                                   work was skipped, its output is undefined */
    PA_ERR_WORKSPACE = 15       /* the scratch must grow while the stream is capturing (or, for
                                   pa_varlen_fwd_noalloc, exceeds its fixed array) */
};

/*
 * pa_varlen_fwd -- forward paged (or non-paged) varlen attention.
 *
 *  q             (total_q, num_heads, head_dim), f16 or bf16, last dim contiguous.
 *  k_cache,
 *  v_cache       paged:     (num_blocks, page_block_size, num_heads_k, head_dim), same dtype
 *                non-paged: (total_k, num_heads_k, head_dim) when block_table is NULL
 *                last dim contiguous; other strides free (multiples of 8 elements).
 *  cu_seqlens_q,
 *  cu_seqlens_k  int32 (batch + 1), contiguous, cumulative offsets starting at 0.  In paged
 *                mode only the differences sk_b are used: the keys of sequence b are the
 *                logical positions 0..sk_b-1 of row b of the block table.
 *  block_table   int32 (batch, max_pages), last dim contiguous; entry [b, p] is the
 *                physical block of logical page p of sequence b.  Entries at or past
 *                ceil(sk_b / page_block_size) are never read.  NULL selects non-paged mode.
 *  max_seqlen_q,
 *  max_seqlen_k  upper bounds of sq_b and sk_b (grid sizing; a kernel that sees a longer
 *                sequence flags PA_ERR_DEVICE_BOUNDS and skips the excess).
 *  num_heads, num_heads_k, head_dim
 *                must equal the descriptors' sizes; num_heads % num_heads_k == 0.
 *  page_block_size  paged mode: the cache's page size (0 = not set -> PA_ERR_PAGE_UNSET).
 *  softmax_scale    multiplies q.k before the softmax.
 *  window_left, window_right   window sides in keys; a negative side is unbounded.
 *  out           (total_q, num_heads, head_dim), dtype of q, last dim contiguous.
 *  softmax_lse   f32 (num_heads, total_q), last dim contiguous.
 *  stream        a cudaStream_t (NULL = the legacy default stream).
 *
 * Checks run in the pages' order: ranks, last-dim contiguity, k/v shapes, page size set,
 * page size == k shape, page size % 32, head size <= 512; then device residency, then the
 * library's own argument checks.  Returns PA_OK or a status (message: pa_last_error()).
 * Memory: the library keeps one grow-only scratch per (device, stream) for the split-KV
 * partial results, the decode kernel's launch order or work list (longest sequence first;
 * the list, with its take counter, is rewritten on the device by every call) and the
 * prefill kernels' item counter (256 bytes, zeroed on the device by every call that runs
 * them); it is allocated on first need with cudaMalloc and never while `stream` is capturing
 * (PA_ERR_WORKSPACE): before capturing a call into a CUDA graph, make one call of the
 * largest shape on the capture stream.
 * Streams: a batch that holds prefill-class sequences (more than 32 rows of q_len x the
 * GQA group) runs the tensor-core prefill kernel on a second stream forked from `stream`
 * and joined back to it with events, beside the decode-class pass on `stream`.  The
 * library keeps one such side stream (with its two events) per (device, caller stream),
 * created by the first such call on that stream: make it before capturing `stream` into a
 * graph.  Two caller streams never share a side stream, so their prefill work can overlap.
 * Thread safety: calls from several host threads are safe.
 */
int pa_varlen_fwd(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                  const pa_tensor* cu_seqlens_q, const pa_tensor* cu_seqlens_k,
                  const pa_tensor* block_table, int32_t max_seqlen_q, int32_t max_seqlen_k,
                  int32_t num_heads, int32_t num_heads_k, int32_t head_dim,
                  int32_t page_block_size, float softmax_scale, int32_t window_left,
                  int32_t window_right, const pa_tensor* out, const pa_tensor* softmax_lse,
                  void* stream);

/*
 * pa_varlen_fwd_noalloc -- pa_varlen_fwd without any device allocation.  (The pages have
 * no counterpart: this is a deployment variant of the same call.)
 *
 * For callers that cannot call cudaMalloc: inference runtimes that hand all device memory
 * to their own arena at start-up, code that runs where an allocation could synchronise the
 * device or fail at the worst moment (latency-critical serving loops), and hosts that only
 * let a plug-in use the buffers they pass in.  Same arguments, checks and results as
 * pa_varlen_fwd; the caller still provides every input and output.
 *
 * Scratch: split-KV partial results (and the decode launch order of batches of more than
 * 160 sequences whose grid takes more than one wave of resident CTAs, or the work list of
 * batches of 16 or more that the plan splits, and the prefill kernels' item counter) go
 * to one fixed 32 MiB array compiled into the library
 * (a static device array: every GPU that loads the library holds it until the process
 * exits) instead of the library's growable workspace.  A call whose split plan needs more
 * than 32 MiB is rejected with PA_ERR_WORKSPACE and a message giving both sizes.  The
 * array keeps the last call's contents; nothing in it needs to start at zero (the work
 * list's and the prefill kernels' take counters are zeroed on the device by the call that
 * uses them).  All calls,
 * on every stream and host thread, share this one array: calls that overlap on the GPU
 * race and give undefined results, so serialise them (one stream, or events).
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, which allocates nothing); make that first call before any stream
 * capture.  It calls no cudaMalloc, cudaFree or allocating library routine, and creates no
 * stream or event: a batch with prefill-class sequences runs its prefill kernel and its
 * decode-class pass one after the other on `stream` (pa_varlen_fwd overlaps them).
 */
int pa_varlen_fwd_noalloc(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                          const pa_tensor* cu_seqlens_q, const pa_tensor* cu_seqlens_k,
                          const pa_tensor* block_table, int32_t max_seqlen_q, int32_t max_seqlen_k,
                          int32_t num_heads, int32_t num_heads_k, int32_t head_dim,
                          int32_t page_block_size, float softmax_scale, int32_t window_left,
                          int32_t window_right, const pa_tensor* out, const pa_tensor* softmax_lse,
                          void* stream);

/*
 * pa_varlen_check -- the host-side checks of pa_varlen_fwd alone: no device-residency
 * check, no CUDA call, no launch.  Same arguments (no stream), same status codes.
 * Lets a caller (or a test without a GPU) validate descriptors ahead of time.
 */
int pa_varlen_check(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                    const pa_tensor* cu_seqlens_q, const pa_tensor* cu_seqlens_k,
                    const pa_tensor* block_table, int32_t max_seqlen_q, int32_t max_seqlen_k,
                    int32_t num_heads, int32_t num_heads_k, int32_t head_dim,
                    int32_t page_block_size, float softmax_scale, int32_t window_left,
                    int32_t window_right, const pa_tensor* out, const pa_tensor* softmax_lse);

/*
 * pa_varlen_fwd_alibi -- pa_varlen_fwd with a linear position bias.  The pages name
 * alibi_slopes only through the condition "shape mismatch alibi_slopes {:?}, expected
 * {:?}" (a related error of "paged flash-attn requires page_block_size to be a multiple of
 * 32" and of "flash-attn-varlen paged expects k/v tensors of rank 4"); the bias taken is
 * the usual one: the score of query i and key j of a sequence with sq queries and sk
 * keys, for query head h, becomes
 *     softmax_scale * q.k_j - alibi_slopes[h] * |i + sk - sq - j|,
 * before the mask and the softmax (lse includes the bias).
 *
 *  alibi_slopes  (num_heads,) f32, contiguous, device memory, borrowed for the call;
 *                NULL gives exactly pa_varlen_fwd.
 * Extra status codes, checked after the q/k/v shape conditions: PA_ERR_SHAPE "shape
 * mismatch alibi_slopes [n], expected [num_heads]" (rank other than 1 or a wrong
 * length), PA_ERR_NONCONTIG (stride != 1), PA_ERR_NOT_DEVICE, PA_ERR_ARG (dtype not f32).
 * Everything else is as for pa_varlen_fwd.
 */
int pa_varlen_fwd_alibi(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                        const pa_tensor* cu_seqlens_q, const pa_tensor* cu_seqlens_k,
                        const pa_tensor* block_table, int32_t max_seqlen_q, int32_t max_seqlen_k,
                        int32_t num_heads, int32_t num_heads_k, int32_t head_dim,
                        int32_t page_block_size, float softmax_scale, int32_t window_left,
                        int32_t window_right, const pa_tensor* alibi_slopes, const pa_tensor* out,
                        const pa_tensor* softmax_lse, void* stream);

/* pa_varlen_check with alibi_slopes (host-side checks only, as pa_varlen_check). */
int pa_varlen_check_alibi(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                          const pa_tensor* cu_seqlens_q, const pa_tensor* cu_seqlens_k,
                          const pa_tensor* block_table, int32_t max_seqlen_q, int32_t max_seqlen_k,
                          int32_t num_heads, int32_t num_heads_k, int32_t head_dim,
                          int32_t page_block_size, float softmax_scale, int32_t window_left,
                          int32_t window_right, const pa_tensor* alibi_slopes, const pa_tensor* out,
                          const pa_tensor* softmax_lse);

/*
 * pa_kv_append -- writes new key/value tokens into the paged caches, the step that comes
 * before pa_varlen_fwd in a serving loop.  The pages give no append operation; they say
 * that a sequence's occupancy of its pages is tracked through the block table ("paged
 * flash-attn requires page_block_size to be a multiple of 32", Solutions) and that the
 * table maps a sequence's logical pages to physical blocks ("flash-attn-varlen paged
 * expects k/v tensors of rank 4", What it means).  The placement taken is the one the
 * bottom-right aligned mask implies: sequence b has sk_b = cu_seqlens_k[b+1] -
 * cu_seqlens_k[b] keys after the append, and its n_b = cu_seqlens_new[b+1] -
 * cu_seqlens_new[b] new tokens are the last n_b of them.  New token t (0-based) goes to
 * logical key pos = sk_b - n_b + t, i.e. slot pos % P of block block_table[b, pos / P].
 * For a chunked-prefill or decode step, cu_seqlens_new is the step's cu_seqlens_q and the
 * attention call that follows uses the same cu_seqlens_k and block_table.
 *
 *  k_new, v_new    (total_new, num_heads_k, head_dim), the caches' dtype (f16 or bf16),
 *                  last dim contiguous, other strides multiples of 8 elements
 *  cu_seqlens_new  int32 [batch + 1], contiguous
 *  cu_seqlens_k    int32 [batch + 1], contiguous: lengths after the append
 *  block_table     int32 [batch, max_pages], last dim contiguous
 *  k_cache,
 *  v_cache         (num_blocks, page_block_size, num_heads_k, head_dim), same shape and
 *                  strides; written in place (only the new tokens' slots)
 *  stream          cudaStream_t the copy is ordered on; the call is asynchronous and
 *                  every tensor is borrowed until it completes.
 * Host checks, in the pages' order where they apply, with pa_varlen_fwd's codes and texts:
 * ranks (k_new/v_new 3: PA_ERR_RANK; caches 4: PA_ERR_RANK_PAGED), last-dim contiguity
 * (PA_ERR_NONCONTIG), shapes (PA_ERR_SHAPE), page size (PA_ERR_PAGE_UNSET / _MISMATCH /
 * _MULT32), head_dim > 512 (PA_ERR_HEADDIM), index tensors, device residency
 * (PA_ERR_NOT_DEVICE), dtypes and batch sizes (PA_ERR_ARG), alignment (PA_ERR_UNSUPPORTED).
 * On the device, a sequence with n_b > sk_b, a position past its block-table row or a
 * block id outside [0, num_blocks) is skipped and reported by pa_device_status() as
 * PA_ERR_DEVICE_BOUNDS.  Tokens of other sequences are still written.
 */
int pa_kv_append(const pa_tensor* k_new, const pa_tensor* v_new, const pa_tensor* cu_seqlens_new,
                 const pa_tensor* cu_seqlens_k, const pa_tensor* block_table, const pa_tensor* k_cache,
                 const pa_tensor* v_cache, int32_t page_block_size, void* stream);

/* The host-side checks of pa_kv_append alone: no device-residency check, no CUDA call. */
int pa_kv_append_check(const pa_tensor* k_new, const pa_tensor* v_new, const pa_tensor* cu_seqlens_new,
                       const pa_tensor* cu_seqlens_k, const pa_tensor* block_table, const pa_tensor* k_cache,
                       const pa_tensor* v_cache, int32_t page_block_size);

/*
 * pa_fwd_padded -- attention over a padded batch (every sequence of the batch has seqlen_q
 * queries and seqlen_k keys), the non-varlen API the pages point to for padded batches
 * ("flash-attn-varlen expects input tensors of rank 3", Solutions: use FlashAttention
 * (non-varlen) for padded batch attention).  Same arithmetic, mask (bottom-right
 * aligned: causal = (-1, 0)), GQA mapping and optional linear position bias as
 * pa_varlen_fwd_alibi; no paging.
 *
 *  q             (batch, seqlen_q, num_heads, head_dim), f16 or bf16, last dim contiguous
 *  k, v          (batch, seqlen_k, num_heads_k, head_dim), same dtype, same shape
 *  alibi_slopes  (num_heads,) f32 or NULL
 *  out           (batch, seqlen_q, num_heads, head_dim), q's dtype, written
 *  softmax_lse   (batch, num_heads, seqlen_q) f32, last dim contiguous, written
 *  stream        cudaStream_t; asynchronous, tensors borrowed until it completes.
 * The batch and sequence dimensions of q, k, v and out must be mergeable (batch stride =
 * seqlen * sequence stride, as for contiguous tensors), else PA_ERR_UNSUPPORTED.  Status
 * codes: PA_ERR_RANK for a rank other than 4, PA_ERR_NONCONTIG, PA_ERR_SHAPE (k vs v, q vs
 * k, alibi_slopes), then the checks of pa_varlen_fwd on the packed view.  The library
 * keeps a small per-(device, stream) device buffer for the uniform cumulative lengths
 * (grown outside stream capture only, PA_ERR_WORKSPACE otherwise).
 */
int pa_fwd_padded(const pa_tensor* q, const pa_tensor* k, const pa_tensor* v, int32_t num_heads,
                  int32_t num_heads_k, int32_t head_dim, float softmax_scale, int32_t window_left,
                  int32_t window_right, const pa_tensor* alibi_slopes, const pa_tensor* out,
                  const pa_tensor* softmax_lse, void* stream);

/* The host-side checks of pa_fwd_padded alone: no device-residency check, no CUDA call. */
int pa_check_padded(const pa_tensor* q, const pa_tensor* k, const pa_tensor* v, int32_t num_heads,
                    int32_t num_heads_k, int32_t head_dim, float softmax_scale, int32_t window_left,
                    int32_t window_right, const pa_tensor* alibi_slopes, const pa_tensor* out,
                    const pa_tensor* softmax_lse);

/* Message of the calling thread's last failed call ("" after a success).  The string
 * stays valid until that thread's next call into the library. */
const char* pa_last_error(void);

/* Synchronises `stream`, then reads and clears the current device's error word set by
 * the kernels (bounded-wait timeouts, out-of-range metadata).  Returns PA_OK,
 * PA_ERR_DEVICE_TIMEOUT, PA_ERR_DEVICE_BOUNDS or PA_ERR_CUDA. */
int pa_device_status(void* stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int pa_version(void);

/* Upper bound, in nanoseconds of wall time, on every wait inside the kernels (for
 * pipeline stages that never complete).  Default 2e9; 0 restores the default.  A wait
 * that runs out makes its CTA leave and pa_device_status() report PA_ERR_DEVICE_TIMEOUT;
 * the CUDA context stays usable.  Applies to calls made after it. */
void pa_set_wait_limit_ns(uint64_t ns);

/* Fault injection for tests of the bounded waits: while enabled (non-zero), the kernels'
 * load producers issue no loads, so every consumer wait runs out after the wait limit
 * and the call reports PA_ERR_DEVICE_TIMEOUT through pa_device_status().  Outputs of
 * such calls are undefined.  No GPU fault is involved.  Applies to calls made after it. */
void pa_set_withhold_loads(int enable);

/* Number of kernels this library has launched in this process (all threads, all
 * devices), for profiling: a caller reads it before and after a region. */
uint64_t pa_kernel_launches(void);

/* Per-kernel device timing, for profiling.  After pa_kernel_timing(1), every kernel this
 * library launches (any thread, any device) is bracketed by two CUDA events recorded on
 * the stream it is launched on; launches into a stream that is being captured are not
 * timed, and at most 65,536 launches are kept between two reads.  pa_kernel_timing(0)
 * stops recording; what was recorded stays until it is read.
 * pa_kernel_times waits for the recorded events, writes to ms[c] the summed elapsed
 * milliseconds and to launches[c] the number of timed launches of kernel class c, and
 * clears the record.  Classes: PA_KC_PREFILL (the tensor-core prefill kernels),
 * PA_KC_SPLITKV (the split-KV pass: decode_kernel, decode512_kernel, decode_tc_kernel or
 * splitkv_kernel), PA_KC_COMBINE (the split-KV combine), PA_KC_APPEND (pa_kv_append's
 * kernel).  ms and launches are caller-owned host arrays of PA_KERNEL_CLASSES entries.  Returns PA_OK, PA_ERR_ARG for a null array, or PA_ERR_CUDA if an event
 * query failed (message in pa_last_error; the record is cleared either way). */
#define PA_KC_PREFILL 0
#define PA_KC_SPLITKV 1
#define PA_KC_COMBINE 2
#define PA_KC_APPEND 3
#define PA_KERNEL_CLASSES 4
void pa_kernel_timing(int enable);
int pa_kernel_times(double* ms, uint64_t* launches);

#ifdef __cplusplus
}
#endif

#endif /* PA_VARLEN_H */
