// C-ABI front end of libpa_varlen: argument validation in the order candle's
// varlen wrapper checks (ranks, last-dim contiguity, k/v shapes, page size set,
// page size matches k, page size multiple of 32, head size <= 512 -- the Source
// excerpts of "flash-attn-varlen expects input tensors of rank 3" and
// "paged flash-attn requires page_block_size"), device residency of the index
// tensors (their "Related errors"), then this library's own limits; workspace
// management; and dispatch to the kernels.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "pa_internal.h"

namespace {

thread_local char g_msg[1024] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return code;
}

std::string dims(const pa_tensor* t) {
    std::string s = "[";
    for (int i = 0; i < t->ndim && i < 4; ++i) {
        if (i) s += ", ";
        s += std::to_string(t->shape[i]);
    }
    return s + "]";
}

std::string strides(const pa_tensor* t) {
    std::string s = "[";
    for (int i = 0; i < t->ndim && i < 4; ++i) {
        if (i) s += ", ";
        s += std::to_string(t->stride[i]);
    }
    return s + "]";
}

bool same_shape(const pa_tensor* a, const pa_tensor* b) {
    if (a->ndim != b->ndim) return false;
    for (int i = 0; i < a->ndim; ++i)
        if (a->shape[i] != b->shape[i]) return false;
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t numel(const pa_tensor* t) {
    int64_t n = 1;
    for (int i = 0; i < t->ndim && i < 4; ++i) n *= t->shape[i];
    return n;
}

bool is_device_memory(const void* p) {
    cudaPointerAttributes attr{};
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged;
}

int validate(const pa_tensor* q, const pa_tensor* k, const pa_tensor* v, const pa_tensor* cu_q,
             const pa_tensor* cu_k, const pa_tensor* bt, int32_t max_sq, int32_t max_sk, int32_t num_heads,
             int32_t num_heads_k, int32_t head_dim, int32_t page_block_size, float softmax_scale, int32_t wl,
             int32_t wr, const pa_tensor* alibi, const pa_tensor* out, const pa_tensor* lse, bool check_device,
             pa::Args* a) {
    if (!q || !k || !v || !cu_q || !cu_k || !out || !lse)
        return fail(PA_ERR_ARG, "a tensor descriptor is NULL (only block_table may be NULL)");
    const bool paged = bt != nullptr;
    const int q_rank = q->ndim, k_rank = k->ndim, v_rank = v->ndim;

    // -- ranks
    if (q_rank != 3 || (!paged && k_rank != 3) || (!paged && v_rank != 3))
        return fail(PA_ERR_RANK, "flash-attn-varlen expects input tensors of rank 3 (q: %d, k: %d, v: %d)", q_rank,
                    k_rank, v_rank);
    if (paged && (k_rank != 4 || v_rank != 4))
        return fail(PA_ERR_RANK_PAGED, "flash-attn-varlen paged expects k/v tensors of rank 4 (k: %d, v: %d)",
                    k_rank, v_rank);
    // -- last-dim contiguity
    if (q->stride[q_rank - 1] != 1)
        return fail(PA_ERR_NONCONTIG, "the last dim of q must be contiguous %s", strides(q).c_str());
    if (k->stride[k_rank - 1] != 1)
        return fail(PA_ERR_NONCONTIG, "the last dim of k must be contiguous %s", strides(k).c_str());
    if (v->stride[v_rank - 1] != 1)
        return fail(PA_ERR_NONCONTIG, "the last dim of v must be contiguous %s", strides(v).c_str());

    const int64_t total_q = q->shape[0], hq = q->shape[1], head_size = q->shape[2];
    int64_t hkv = 0, num_blocks = 0, page = 0;
    if (paged) {
        // -- paged shape branch
        page = k->shape[1];
        hkv = k->shape[2];
        num_blocks = k->shape[0];
        if (!same_shape(k, v))
            return fail(PA_ERR_SHAPE, "shape mismatch k %s and v %s", dims(k).c_str(), dims(v).c_str());
        if (k->shape[3] != head_size)
            return fail(PA_ERR_SHAPE, "shape mismatch q %s and k %s", dims(q).c_str(), dims(k).c_str());
        if (page_block_size <= 0) return fail(PA_ERR_PAGE_UNSET, "paged flash-attn requires page_block_size");
        if (page_block_size != page)
            return fail(PA_ERR_PAGE_MISMATCH, "page_block_size %d does not match k shape %s", page_block_size,
                        dims(k).c_str());
        if (page % 32 != 0)
            return fail(PA_ERR_PAGE_MULT32,
                        "paged flash-attn requires page_block_size to be a multiple of 32 (got %lld)",
                        (long long)page);
        if (head_size > 512)
            return fail(PA_ERR_HEADDIM, "paged flash-attn supports head sizes up to 512 (got %lld)",
                        (long long)head_size);
    } else {
        // -- non-paged branch: k and v are (total_k, num_heads_k, head_size)
        hkv = k->shape[1];
        num_blocks = k->shape[0];
        if (!(k->shape[0] == num_blocks && k->shape[1] == hkv && k->shape[2] == head_size))
            return fail(PA_ERR_SHAPE, "shape mismatch q %s and k %s", dims(q).c_str(), dims(k).c_str());
        if (!(v->shape[0] == num_blocks && v->shape[1] == hkv && v->shape[2] == head_size))
            return fail(PA_ERR_SHAPE, "shape mismatch q %s and v %s", dims(q).c_str(), dims(v).c_str());
    }
    // -- alibi_slopes (optional): one slope per query head (the "shape mismatch alibi_slopes"
    // condition the pages list beside the k/v shape checks)
    if (alibi && (alibi->ndim != 1 || alibi->shape[0] != hq))
        return fail(PA_ERR_SHAPE, "shape mismatch alibi_slopes %s, expected [%lld]", dims(alibi).c_str(),
                    (long long)hq);

    // -- index tensors
    if (cu_q->ndim != 1) return fail(PA_ERR_ARG, "seqlens_q must be rank 1, got rank %d", cu_q->ndim);
    if (cu_k->ndim != 1) return fail(PA_ERR_ARG, "seqlens_k must be rank 1, got rank %d", cu_k->ndim);
    if (cu_q->stride[0] != 1) return fail(PA_ERR_NONCONTIG, "seqlens_q has to be contiguous");
    if (cu_k->stride[0] != 1) return fail(PA_ERR_NONCONTIG, "seqlens_k has to be contiguous");
    if (paged) {
        if (bt->ndim != 2) return fail(PA_ERR_ARG, "block_table must be rank 2, got rank %d", bt->ndim);
        if (bt->stride[1] != 1) return fail(PA_ERR_NONCONTIG, "block_table last dimension must be contiguous");
    }
    if (alibi && alibi->stride[0] != 1) return fail(PA_ERR_NONCONTIG, "alibi_slopes has to be contiguous");
    if (check_device) {  // tensors with no elements are never read or written
        auto on_device = [](const pa_tensor* t) { return numel(t) == 0 || is_device_memory(t->data); };
        if (paged && !on_device(bt)) return fail(PA_ERR_NOT_DEVICE, "block_table must be a cuda tensor");
        if (!on_device(cu_q)) return fail(PA_ERR_NOT_DEVICE, "seqlens_q must be a cuda tensor");
        if (!on_device(cu_k)) return fail(PA_ERR_NOT_DEVICE, "seqlens_k must be a cuda tensor");
        if (!on_device(q)) return fail(PA_ERR_NOT_DEVICE, "q must be a cuda tensor");
        if (!on_device(k)) return fail(PA_ERR_NOT_DEVICE, "k must be a cuda tensor");
        if (!on_device(v)) return fail(PA_ERR_NOT_DEVICE, "v must be a cuda tensor");
        if (!on_device(out)) return fail(PA_ERR_NOT_DEVICE, "out must be a cuda tensor");
        if (!on_device(lse)) return fail(PA_ERR_NOT_DEVICE, "softmax_lse must be a cuda tensor");
        if (alibi && !on_device(alibi)) return fail(PA_ERR_NOT_DEVICE, "alibi_slopes must be a cuda tensor");
    }

    // -- this library's own argument checks
    if (q->dtype != PA_F16 && q->dtype != PA_BF16)
        return fail(PA_ERR_UNSUPPORTED, "q dtype %d: only f16 and bf16 are supported", q->dtype);
    if (k->dtype != q->dtype || v->dtype != q->dtype || out->dtype != q->dtype)
        return fail(PA_ERR_ARG, "q, k, v and out must share one dtype (q %d, k %d, v %d, out %d)", q->dtype,
                    k->dtype, v->dtype, out->dtype);
    if (lse->dtype != PA_F32) return fail(PA_ERR_ARG, "softmax_lse must be f32");
    if (alibi && alibi->dtype != PA_F32) return fail(PA_ERR_ARG, "alibi_slopes must be f32");
    if (cu_q->dtype != PA_I32 || cu_k->dtype != PA_I32 || (paged && bt->dtype != PA_I32))
        return fail(PA_ERR_ARG, "cu_seqlens and block_table must be int32");
    if (num_heads != hq || head_dim != head_size || num_heads_k != hkv)
        return fail(PA_ERR_ARG,
                    "scalars disagree with the tensors: num_heads %d vs %lld, num_heads_k %d vs %lld, head_dim %d "
                    "vs %lld",
                    num_heads, (long long)hq, num_heads_k, (long long)hkv, head_dim, (long long)head_size);
    if (hkv <= 0 || hq <= 0 || hq % hkv != 0)
        return fail(PA_ERR_ARG, "num_heads (%lld) must be a positive multiple of num_heads_k (%lld)", (long long)hq,
                    (long long)hkv);
    if (head_size <= 0) return fail(PA_ERR_ARG, "head_dim must be positive");
    if (out->ndim != 3 || out->shape[0] != total_q || out->shape[1] != hq || out->shape[2] != head_size)
        return fail(PA_ERR_ARG, "out must have q's shape %s, got %s", dims(q).c_str(), dims(out).c_str());
    if (out->stride[2] != 1)
        return fail(PA_ERR_NONCONTIG, "the last dim of out must be contiguous %s", strides(out).c_str());
    if (lse->ndim != 2 || lse->shape[0] != hq || lse->shape[1] != total_q || lse->stride[1] != 1)
        return fail(PA_ERR_ARG, "softmax_lse must be (num_heads, total_q) = (%lld, %lld) with a contiguous last dim",
                    (long long)hq, (long long)total_q);
    if (cu_q->shape[0] < 1 || cu_q->shape[0] != cu_k->shape[0])
        return fail(PA_ERR_ARG, "cu_seqlens_q and cu_seqlens_k must both have batch + 1 >= 1 entries (%lld, %lld)",
                    (long long)cu_q->shape[0], (long long)cu_k->shape[0]);
    const int64_t batch = cu_q->shape[0] - 1;
    if (paged && bt->shape[0] != batch)
        return fail(PA_ERR_ARG, "block_table has %lld rows for a batch of %lld", (long long)bt->shape[0],
                    (long long)batch);
    if (max_sq < 0 || max_sk < 0) return fail(PA_ERR_ARG, "max_seqlen_q and max_seqlen_k must be >= 0");
    if (paged && (int64_t)max_sk > bt->shape[1] * page)
        return fail(PA_ERR_ARG, "block_table holds %lld pages of %lld slots, too few for max_seqlen_k %d",
                    (long long)bt->shape[1], (long long)page, max_sk);
    if (!std::isfinite(softmax_scale)) return fail(PA_ERR_ARG, "softmax_scale must be finite");

    // -- implementation limits (not page conditions)
    if (head_size % 8 != 0)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %lld: kernels need a multiple of 8", (long long)head_size);
    if (!paged && head_size > 512)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %lld: kernels support up to 512", (long long)head_size);
    if (batch > 65535) return fail(PA_ERR_UNSUPPORTED, "batch %lld exceeds 65535", (long long)batch);
    if (total_q >= (1ll << 31) || num_blocks >= (1ll << 31) || hq * total_q >= (1ll << 40))
        return fail(PA_ERR_UNSUPPORTED, "sizes beyond 2^31 rows are not supported");
    for (const pa_tensor* t : {q, k, v, out}) {
        if (numel(t) == 0) continue;
        if (!aligned16(t->data))
            return fail(PA_ERR_UNSUPPORTED, "q/k/v/out base addresses must be 16-byte aligned");
        for (int d = 0; d < t->ndim - 1; ++d)
            if (t->stride[d] % 8 != 0 || t->stride[d] <= 0)
                return fail(PA_ERR_UNSUPPORTED, "strides %s: all but the last must be positive multiples of 8 elements",
                            strides(t).c_str());
    }

    a->dtype = q->dtype;
    a->q = q->data;
    a->q_s0 = q->stride[0];
    a->q_s1 = q->stride[1];
    a->k = k->data;
    a->v = v->data;
    if (paged) {
        if (k->stride[0] != v->stride[0] || k->stride[1] != v->stride[1] || k->stride[2] != v->stride[2])
            return fail(PA_ERR_UNSUPPORTED, "k and v caches must share strides (k %s, v %s)", strides(k).c_str(),
                        strides(v).c_str());
        a->kv_s0 = k->stride[0];
        a->kv_s1 = k->stride[1];
        a->kv_s2 = k->stride[2];
    } else {
        if (k->stride[0] != v->stride[0] || k->stride[1] != v->stride[1])
            return fail(PA_ERR_UNSUPPORTED, "k and v must share strides (k %s, v %s)", strides(k).c_str(),
                        strides(v).c_str());
        a->kv_s0 = k->stride[0];
        a->kv_s1 = 0;
        a->kv_s2 = k->stride[1];
    }
    a->paged = paged;
    a->num_blocks = num_blocks;
    a->page = paged ? (int)page : 0;
    a->cu_q = static_cast<const int32_t*>(cu_q->data);
    a->cu_k = static_cast<const int32_t*>(cu_k->data);
    a->batch = (int)batch;
    a->block_table = paged ? static_cast<const int32_t*>(bt->data) : nullptr;
    a->bt_s0 = paged ? bt->stride[0] : 0;
    a->bt_cols = paged ? (int)bt->shape[1] : 0;
    a->max_sq = max_sq;
    a->max_sk = max_sk;
    a->H = (int)hq;
    a->Hkv = (int)hkv;
    a->D = (int)head_size;
    a->scale = softmax_scale;
    a->wl = wl < 0 ? -1 : wl;
    a->wr = wr < 0 ? -1 : wr;
    a->out = out->data;
    a->o_s0 = out->stride[0];
    a->o_s1 = out->stride[1];
    a->lse = static_cast<float*>(lse->data);
    a->lse_s0 = lse->stride[0];
    a->total_q = total_q;
    a->alibi = alibi ? static_cast<const float*>(alibi->data) : nullptr;
    // grid limits of the launches: the split-KV pass puts (kv head, row tile) in grid.y.
    // Long rows go to the tensor-core prefill kernel when it takes the call (one row tile
    // left for the split-KV pass); otherwise every 32 rows of the longest sequence are a tile.
    if (hkv > 65535) return fail(PA_ERR_UNSUPPORTED, "num_heads_k %lld exceeds 65535", (long long)hkv);
    if (!pa::prefill_supported(*a)) {
        const int64_t rows = std::max<int64_t>(1, (int64_t)max_sq * (hq / hkv));
        const int64_t row_tiles = rows <= 16 ? 1 : (rows + 31) / 32;
        if (hkv * row_tiles > 65535)
            return fail(PA_ERR_UNSUPPORTED,
                        "num_heads_k (%lld) x row tiles of max_seqlen_q x group (%lld) exceeds 65535 CTAs per "
                        "sequence for this head_dim / group size; split the call into shorter query chunks",
                        (long long)hkv, (long long)row_tiles);
    }
    g_msg[0] = '\0';
    return PA_OK;
}

// ---- KV append: host checks ----------------------------------------------------------------
int validate_append(const pa_tensor* kn, const pa_tensor* vn, const pa_tensor* cu_new, const pa_tensor* cu_k,
                    const pa_tensor* bt, const pa_tensor* kc, const pa_tensor* vc, int32_t page_block_size,
                    bool check_device, pa::AppendArgs* a) {
    if (!kn || !vn || !cu_new || !cu_k || !bt || !kc || !vc)
        return fail(PA_ERR_ARG, "a tensor descriptor is NULL");
    // -- ranks: new tokens are packed like non-paged k/v, the caches are paged
    if (kn->ndim != 3 || vn->ndim != 3)
        return fail(PA_ERR_RANK, "kv append expects k_new/v_new tensors of rank 3 (k_new: %d, v_new: %d)", kn->ndim,
                    vn->ndim);
    if (kc->ndim != 4 || vc->ndim != 4)
        return fail(PA_ERR_RANK_PAGED, "flash-attn-varlen paged expects k/v tensors of rank 4 (k: %d, v: %d)",
                    kc->ndim, vc->ndim);
    // -- last-dim contiguity
    for (const pa_tensor* t : {kn, vn, kc, vc})
        if (t->stride[t->ndim - 1] != 1)
            return fail(PA_ERR_NONCONTIG, "the last dim of %s must be contiguous %s",
                        t == kn ? "k_new" : t == vn ? "v_new" : t == kc ? "k" : "v", strides(t).c_str());
    // -- shapes
    if (!same_shape(kc, vc)) return fail(PA_ERR_SHAPE, "shape mismatch k %s and v %s", dims(kc).c_str(), dims(vc).c_str());
    if (!same_shape(kn, vn))
        return fail(PA_ERR_SHAPE, "shape mismatch k_new %s and v_new %s", dims(kn).c_str(), dims(vn).c_str());
    if (kn->shape[1] != kc->shape[2] || kn->shape[2] != kc->shape[3])
        return fail(PA_ERR_SHAPE, "shape mismatch k_new %s and k %s", dims(kn).c_str(), dims(kc).c_str());
    const int64_t page = kc->shape[1], head_size = kc->shape[3];
    // -- page size and head size, as for the paged forward call
    if (page_block_size <= 0) return fail(PA_ERR_PAGE_UNSET, "paged flash-attn requires page_block_size");
    if (page_block_size != page)
        return fail(PA_ERR_PAGE_MISMATCH, "page_block_size %d does not match k shape %s", page_block_size,
                    dims(kc).c_str());
    if (page % 32 != 0)
        return fail(PA_ERR_PAGE_MULT32, "paged flash-attn requires page_block_size to be a multiple of 32 (got %lld)",
                    (long long)page);
    if (head_size > 512)
        return fail(PA_ERR_HEADDIM, "paged flash-attn supports head sizes up to 512 (got %lld)", (long long)head_size);
    // -- index tensors
    if (cu_new->ndim != 1 || cu_k->ndim != 1) return fail(PA_ERR_ARG, "cu_seqlens_new and cu_seqlens_k must be rank 1");
    if (cu_new->stride[0] != 1) return fail(PA_ERR_NONCONTIG, "seqlens_new has to be contiguous");
    if (cu_k->stride[0] != 1) return fail(PA_ERR_NONCONTIG, "seqlens_k has to be contiguous");
    if (bt->ndim != 2) return fail(PA_ERR_ARG, "block_table must be rank 2, got rank %d", bt->ndim);
    if (bt->stride[1] != 1) return fail(PA_ERR_NONCONTIG, "block_table last dimension must be contiguous");
    if (check_device) {
        auto on_device = [](const pa_tensor* t) { return numel(t) == 0 || is_device_memory(t->data); };
        if (!on_device(bt)) return fail(PA_ERR_NOT_DEVICE, "block_table must be a cuda tensor");
        if (!on_device(cu_new)) return fail(PA_ERR_NOT_DEVICE, "seqlens_new must be a cuda tensor");
        if (!on_device(cu_k)) return fail(PA_ERR_NOT_DEVICE, "seqlens_k must be a cuda tensor");
        if (!on_device(kn) || !on_device(vn)) return fail(PA_ERR_NOT_DEVICE, "k_new and v_new must be cuda tensors");
        if (!on_device(kc) || !on_device(vc)) return fail(PA_ERR_NOT_DEVICE, "k and v must be cuda tensors");
    }
    // -- this library's own argument checks
    if (kc->dtype != PA_F16 && kc->dtype != PA_BF16)
        return fail(PA_ERR_UNSUPPORTED, "cache dtype %d: only f16 and bf16 are supported", kc->dtype);
    if (vc->dtype != kc->dtype || kn->dtype != kc->dtype || vn->dtype != kc->dtype)
        return fail(PA_ERR_ARG, "k_new, v_new and the caches must share one dtype");
    if (cu_new->dtype != PA_I32 || cu_k->dtype != PA_I32 || bt->dtype != PA_I32)
        return fail(PA_ERR_ARG, "cu_seqlens and block_table must be int32");
    if (cu_new->shape[0] < 1 || cu_new->shape[0] != cu_k->shape[0])
        return fail(PA_ERR_ARG, "cu_seqlens_new and cu_seqlens_k must both have batch + 1 >= 1 entries (%lld, %lld)",
                    (long long)cu_new->shape[0], (long long)cu_k->shape[0]);
    const int64_t batch = cu_new->shape[0] - 1;
    if (bt->shape[0] != batch)
        return fail(PA_ERR_ARG, "block_table has %lld rows for a batch of %lld", (long long)bt->shape[0],
                    (long long)batch);
    if (kc->stride[0] != vc->stride[0] || kc->stride[1] != vc->stride[1] || kc->stride[2] != vc->stride[2])
        return fail(PA_ERR_UNSUPPORTED, "k and v caches must share strides (k %s, v %s)", strides(kc).c_str(),
                    strides(vc).c_str());
    if (head_size % 8 != 0)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %lld: the copy needs a multiple of 8", (long long)head_size);
    if (batch > (1ll << 30) || kn->shape[0] >= (1ll << 31) || kc->shape[0] >= (1ll << 31))
        return fail(PA_ERR_UNSUPPORTED, "sizes beyond 2^31 rows are not supported");
    for (const pa_tensor* t : {kn, vn, kc, vc}) {
        if (numel(t) == 0) continue;
        if (!aligned16(t->data)) return fail(PA_ERR_UNSUPPORTED, "k_new/v_new/cache base addresses must be 16-byte aligned");
        for (int d = 0; d < t->ndim - 1; ++d)
            if (t->stride[d] % 8 != 0 || t->stride[d] <= 0)
                return fail(PA_ERR_UNSUPPORTED, "strides %s: all but the last must be positive multiples of 8 elements",
                            strides(t).c_str());
    }
    a->k_new = kn->data;
    a->v_new = vn->data;
    a->kn_s0 = kn->stride[0];
    a->kn_s1 = kn->stride[1];
    a->vn_s0 = vn->stride[0];
    a->vn_s1 = vn->stride[1];
    a->k_cache = kc->data;
    a->v_cache = vc->data;
    a->c_s0 = kc->stride[0];
    a->c_s1 = kc->stride[1];
    a->c_s2 = kc->stride[2];
    a->cu_new = static_cast<const int32_t*>(cu_new->data);
    a->cu_k = static_cast<const int32_t*>(cu_k->data);
    a->bt = static_cast<const int32_t*>(bt->data);
    a->bt_s0 = bt->stride[0];
    a->bt_cols = (int)bt->shape[1];
    a->batch = (int)batch;
    a->total_new = kn->shape[0];
    a->num_blocks = kc->shape[0];
    a->P = (int)page;
    a->Hkv = (int)kc->shape[2];
    a->D = (int)head_size;
    g_msg[0] = '\0';
    return PA_OK;
}

// ---- per-(device, stream) split-KV workspace ------------------------------------------------
std::mutex g_ws_mu;
std::map<std::pair<int, cudaStream_t>, pa::Workspace> g_ws;
// uniform cu_seqlens of the padded entry point, per (device, stream) like the workspace
std::map<std::pair<int, cudaStream_t>, pa::Workspace> g_cu;

int grow_buffer(std::map<std::pair<int, cudaStream_t>, pa::Workspace>& buffers, cudaStream_t stream, size_t bytes,
                void** ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    std::lock_guard<std::mutex> lock(g_ws_mu);
    pa::Workspace& w = buffers[{dev, stream}];
    if (w.bytes < bytes) {
        cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
        e = cudaStreamIsCapturing(stream, &st);
        if (e != cudaSuccess) return fail(PA_ERR_CUDA, "cudaStreamIsCapturing: %s", cudaGetErrorString(e));
        if (st != cudaStreamCaptureStatusNone)
            return fail(PA_ERR_WORKSPACE,
                        "a library buffer must grow to %zu bytes while the stream is capturing; run one call "
                        "of the largest shape before capture",
                        bytes);
        if (w.ptr) {
            e = cudaFree(w.ptr);  // synchronises the device: earlier calls are done with it
            w.ptr = nullptr;
            w.bytes = 0;
            if (e != cudaSuccess) return fail(PA_ERR_CUDA, "cudaFree(workspace): %s", cudaGetErrorString(e));
        }
        size_t want = std::max(bytes + bytes / 4, (size_t)1 << 20);
        e = cudaMalloc(&w.ptr, want);
        if (e != cudaSuccess) {
            w.ptr = nullptr;
            return fail(PA_ERR_CUDA, "cudaMalloc(workspace, %zu): %s", want, cudaGetErrorString(e));
        }
        w.bytes = want;
    }
    *ptr = w.ptr;
    return PA_OK;
}

int workspace_for(cudaStream_t stream, size_t bytes, void** ptr) { return grow_buffer(g_ws, stream, bytes, ptr); }

// A second stream per (device, caller stream) on which the tensor-core prefill kernel runs
// beside the split-KV kernel (forked from and joined back to the caller's stream with
// events, so stream ordering and graph capture behave as for a single launch).  Each caller
// stream has its own, so the prefill work of two serving streams does not queue behind one
// another; the entry's mutex orders the fork/launch/join of callers sharing one stream.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    std::mutex mu;
};
std::mutex g_side_mu;  // guards the map only
std::map<std::pair<int, cudaStream_t>, SideStream> g_side;

int side_stream(cudaStream_t caller, SideStream** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    std::lock_guard<std::mutex> lock(g_side_mu);
    SideStream& ss = g_side[{dev, caller}];  // std::map: the entry's address never changes
    if (!ss.stream) {
        if ((e = cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming)) != cudaSuccess)
            return fail(PA_ERR_CUDA, "creating the prefill side stream: %s", cudaGetErrorString(e));
    }
    *out = &ss;
    return PA_OK;
}

// Scratch provider of pa_varlen_fwd: the library's own grow-only workspace.
int library_workspace(void*, cudaStream_t stream, size_t bytes, void** ptr, char*, size_t) {
    return workspace_for(stream, bytes, ptr);
}

int sm_count() {
    static int cached[256] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return 148;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qres;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qres) ==
                cudaSuccess &&
            qres == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

namespace pa {

static std::atomic<uint64_t> g_launches{0};
static std::atomic<uint64_t> g_wait_ns{PA_WAIT_LIMIT_NS};
static std::atomic<int> g_withhold{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

// ---- per-kernel timing ----------------------------------------------------------------------
namespace {
struct TimedLaunch {
    int cls, dev;
    cudaEvent_t begin, end;
};
constexpr size_t kMaxTimed = 65536;
std::atomic<int> g_timing{0};
std::mutex g_timer_mu;
std::vector<TimedLaunch> g_timed;                       // guarded by g_timer_mu
std::vector<std::pair<int, cudaEvent_t>> g_event_pool;  // (device, event), guarded by g_timer_mu
thread_local cudaEvent_t t_pending = nullptr;           // begin event of this thread's launch
thread_local int t_pending_dev = -1;

// An event of device `dev` from the pool, or a new one (nullptr on failure).  Caller holds
// g_timer_mu and has `dev` current.
cudaEvent_t pooled_event(int dev) {
    for (size_t i = g_event_pool.size(); i-- > 0;) {
        if (g_event_pool[i].first == dev) {
            cudaEvent_t e = g_event_pool[i].second;
            g_event_pool.erase(g_event_pool.begin() + (long)i);
            return e;
        }
    }
    cudaEvent_t e = nullptr;
    return cudaEventCreate(&e) == cudaSuccess ? e : nullptr;
}
}  // namespace

void timer_begin(int, cudaStream_t stream) {
    if (!g_timing.load(std::memory_order_relaxed)) return;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
        (void)cudaGetLastError();
        return;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return;
    std::lock_guard<std::mutex> lock(g_timer_mu);
    if (t_pending) {  // the previous launch of this thread failed: recycle its event
        g_event_pool.emplace_back(t_pending_dev, t_pending);
        t_pending = nullptr;
    }
    if (g_timed.size() >= kMaxTimed) return;
    cudaEvent_t e = pooled_event(dev);
    if (!e) return;
    if (cudaEventRecord(e, stream) != cudaSuccess) {
        g_event_pool.emplace_back(dev, e);
        return;
    }
    t_pending = e;
    t_pending_dev = dev;
}

void timer_end(int cls, cudaStream_t stream) {
    if (!t_pending) return;
    std::lock_guard<std::mutex> lock(g_timer_mu);
    cudaEvent_t e = pooled_event(t_pending_dev);
    if (e && cudaEventRecord(e, stream) == cudaSuccess) {
        g_timed.push_back({cls, t_pending_dev, t_pending, e});
    } else {
        if (e) g_event_pool.emplace_back(t_pending_dev, e);
        g_event_pool.emplace_back(t_pending_dev, t_pending);
    }
    t_pending = nullptr;
}

int encode_tmap_4d(void* map, int dtype, const void* base, const uint64_t dims_[4], const uint64_t strides_bytes[3],
                   const uint32_t box[4], int swizzle128, char* msg, size_t msg_len) {
    auto fn = encode_fn();
    if (!fn) {
        snprintf(msg, msg_len, "cuTensorMapEncodeTiled is not available from the driver");
        return PA_ERR_CUDA;
    }
    cuuint64_t gdim[4] = {dims_[0], dims_[1], dims_[2], dims_[3]};
    cuuint64_t gstride[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
    cuuint32_t bdim[4] = {box[0], box[1], box[2], box[3]};
    cuuint32_t estride[4] = {1, 1, 1, 1};
    CUresult r = fn(reinterpret_cast<CUtensorMap*>(map),
                    dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                    const_cast<void*>(base), gdim, gstride, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(msg, msg_len,
                 "cuTensorMapEncodeTiled failed (%d): dims [%llu %llu %llu %llu], strides [%llu %llu %llu] bytes", (int)r,
                 (unsigned long long)gdim[0], (unsigned long long)gdim[1], (unsigned long long)gdim[2],
                 (unsigned long long)gdim[3], (unsigned long long)gstride[0], (unsigned long long)gstride[1],
                 (unsigned long long)gstride[2]);
        return PA_ERR_UNSUPPORTED;
    }
    return PA_OK;
}

bool decode_tc_wanted(int dp) {
    // Opt-in (PA_DECODE_TC=1, read per call): on GB300 it measured below the warp-sliced
    // kernel at head dims 128 and 256 (0.50 / 0.73 of the copy peak against 0.93 / 0.91) and
    // below the quarter-column kernel at 512 (0.30 against 0.54).
    const char* env = std::getenv("PA_DECODE_TC");
    return dp >= 128 && env && env[0] == '1';
}

SplitPlan plan_splitkv(const Args& a, bool prefill_takes_long_rows, int prefill_sms, int num_sms) {
    SplitPlan pl{};
    pl.dp = a.D <= 64 ? 64 : a.D <= 128 ? 128 : a.D <= 256 ? 256 : 512;
    pl.nt = pl.dp == 512 ? 32 : 64;
    const int G = a.H / a.Hkv;
    const int64_t rows_max = (int64_t)a.max_sq * G;
    pl.rows_cap = prefill_takes_long_rows ? prefill_rows_threshold() : (1 << 30);
    const int64_t rows_here = std::max<int64_t>(1, std::min<int64_t>(rows_max, pl.rows_cap));
    pl.mt = rows_here <= 16 ? 1 : 2;
    const int M = 16 * pl.mt;
    pl.row_tiles = (int)((rows_here + M - 1) / M);
    pl.tile_rows = (int)std::min<int64_t>(M, rows_here);
    static const bool force_generic = std::getenv("PA_FORCE_GENERIC") != nullptr;
    pl.tc = pl.row_tiles == 1 && !force_generic && decode_tc_wanted(pl.dp);
    if (pl.tc) pl.nt = 128;
    // keys one row tile can touch: its queries span at most M / G + 1 positions
    int64_t kspan = a.max_sk;
    if (a.wl >= 0) kspan = std::min<int64_t>(kspan, (int64_t)a.wl + M / G + 1 + std::max(a.wr, 0) + 1);
    const int64_t tiles_max = std::max<int64_t>(1, kspan / pl.nt + 2);
    int64_t split_tiles = tiles_max;
    const int64_t units = (int64_t)a.batch * a.Hkv * pl.row_tiles;
    const char* env_tiles = std::getenv("PA_SPLIT_TILES");
    if (pl.row_tiles == 1)
        pl.slots = num_sms * (pl.tc ? decode_tc_occupancy(a.dtype, pl.dp, M)
                              : a.dtype == PA_BF16 ? splitkv_occupancy_bf16(pl) : splitkv_occupancy_f16(pl));
    if (env_tiles) {
        split_tiles = std::max<int64_t>(1, std::atoll(env_tiles));
    } else if (pl.row_tiles == 1) {
        // Fewer (sequence, kv head) units than resident CTA slots: one wave, every unit's keys
        // split evenly over slots / units CTAs (each further wave would add a pipeline ramp,
        // a merge and a partial result per CTA).  Otherwise one CTA per unit, no split and no
        // combine: launched longest first, the units themselves even out the waves (on 64
        // decode sequences of U[512, 4096] keys, 512 units over 304 slots: 6.37 TB/s, against
        // 5.72 with two splits per unit and 5.61 with three).  A split is never shorter than
        // 4 tiles, nor than 8 M keys: its fp32 partial result (M rows x D x 4 bytes, written
        // and read back) then costs at most ~1/8 of the K/V bytes it reads.  When this pass runs
        // beside a prefill kernel whose persistent grid may take every SM (its item bound,
        // from the sizes alone, reaches the SM count), there are no free slots to fill: one
        // CTA per unit (the key cap below still spreads a very long sequence) and no combine
        // grid, whose CTAs, empty when the batch is all prefill, would hold the SMs the
        // prefill CTAs wait for (causal batch: prefill CTAs starting ~6.5 us into the call
        // behind 4,096 empty combine CTAs).  A smaller prefill grid leaves the plan as it is
        // (the bound counts every sequence as prefill-class, so it overstates such a grid:
        // one 64-query prompt beside four 8,000-key decode sequences measured 5 % slower
        // when the split was sized to the SMs the bound left).
        const int64_t slots = prefill_sms >= num_sms ? 0 : pl.slots;
        int64_t splits = units < slots ? slots / units : 1;
        splits = std::max<int64_t>(1, std::min(splits, tiles_max));
        const int64_t min_tiles = std::max<int64_t>(4, (8ll * M + pl.nt - 1) / pl.nt);
        split_tiles = std::max<int64_t>(min_tiles, (tiles_max + splits - 1) / splits);
        // Nor does a split hold more than kMaxSplitKeys keys.  The host does not read the
        // lengths, so a batch where one sequence is far longer than the rest (a 131,072-key
        // sequence among 4,096-key ones) would otherwise leave that sequence's one CTA per kv
        // head as the tail of the grid; with the cap its keys spread over many CTAs, while
        // sequences below the cap keep one CTA (their further split indices exit at once, or,
        // in the persistent mode below, are never listed).
        split_tiles = std::min(split_tiles, std::max(min_tiles, kMaxSplitKeys / pl.nt));
    }
    split_tiles = std::min(split_tiles, tiles_max);
    pl.split_tiles = (int)split_tiles;
    pl.max_splits = (int)((tiles_max + split_tiles - 1) / split_tiles);
    if (pl.max_splits > 1024) {  // the combine keeps at most 1024 split weights per row
        pl.split_tiles = (int)((tiles_max + 1023) / 1024);
        pl.max_splits = (int)((tiles_max + pl.split_tiles - 1) / pl.split_tiles);
    }
    // Persistent mode of the warp-sliced decode kernel: when a batch of many sequences has
    // some sequence split, the split indices of every shorter sequence would be CTAs without
    // work (about 1.5 us of an SM slot each: 40 us of a 223 us call on a 64-sequence batch
    // with one 131,072-key sequence).  A one-CTA pass then lists the (sequence, split) items
    // on the device and one CTA per resident slot takes them in turn (that batch: 180 us;
    // shorter splits measured no faster: 4,096 keys 179 us, 2,048 keys 184 us).
    pl.work = !pl.tc && pl.row_tiles == 1 && pl.dp <= 256 && !force_generic && a.batch >= kWorkMinBatch &&
              a.batch <= kMaxOrderBatch && pl.max_splits > 1 && pl.slots > 0;
    // Otherwise the decode kernels launch sequences longest first (a one-CTA ranking pass)
    // for batches they can rank; the order sits at the start of the scratch.  A grid that
    // fits the resident slots runs as one wave, where the order is moot: its CTAs skip the
    // ranking and its dependent memory round trip
    const bool decode_kernel = pl.tc || (pl.row_tiles == 1 && !force_generic);
    const bool one_wave = pl.slots > 0 && units * pl.max_splits <= pl.slots;
    const bool ranked = !pl.work && decode_kernel && !one_wave;
    pl.rank_in_cta = ranked && a.batch >= 2 && a.batch <= kRankInCta;
    pl.order_bytes = ranked && a.batch > kRankInCta && a.batch <= kMaxOrderBatch
                         ? ((size_t)a.batch * sizeof(int) + 255) / 256 * 256
                         : 0;
    pl.work_bytes = pl.work ? ((2 + 2 * (size_t)a.batch * pl.max_splits) * sizeof(int) + 255) / 256 * 256 : 0;
    pl.ws_bytes = pl.order_bytes + pl.work_bytes;
    if (pl.max_splits > 1) {
        const size_t rows = (size_t)a.total_q * a.H;
        pl.ws_bytes += (size_t)pl.max_splits * rows * ((size_t)a.D + 1) * sizeof(float) + 256;
    }
    return pl;
}

int launch_splitkv(const Args& a, const SplitPlan& plan, void* workspace, unsigned int* err, char* msg,
                   size_t msg_len) {
    if (a.dtype == PA_BF16) return launch_splitkv_bf16(a, plan, workspace, err, msg, msg_len);
    return launch_splitkv_f16(a, plan, workspace, err, msg, msg_len);
}

}  // namespace pa

namespace pa {

int forward_impl(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                 const pa_tensor* cu_seqlens_q, const pa_tensor* cu_seqlens_k, const pa_tensor* block_table,
                 int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_heads, int32_t num_heads_k,
                 int32_t head_dim, int32_t page_block_size, float softmax_scale, int32_t window_left,
                 int32_t window_right, const pa_tensor* alibi_slopes, const pa_tensor* out,
                 const pa_tensor* softmax_lse, void* stream, ScratchFn scratch, void* scratch_ctx,
                 bool side_stream_ok) {
    NvtxRange range("pa_varlen_fwd");
    pa::Args a{};
    int rc = validate(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_table, max_seqlen_q, max_seqlen_k,
                      num_heads, num_heads_k, head_dim, page_block_size, softmax_scale, window_left, window_right,
                      alibi_slopes, out, softmax_lse, true, &a);
    if (rc != PA_OK) return rc;
    return launch_forward(a, stream, scratch, scratch_ctx, side_stream_ok);
}

// Everything after the host checks: split plan, scratch, and the launches (prefill on the
// caller stream's side stream beside the split-KV pass on the caller's stream, or both on
// the caller's stream one after the other when `side_stream_ok` is false).
int launch_forward(pa::Args& a, void* stream, ScratchFn scratch, void* scratch_ctx, bool side_stream_ok) {
    int rc = PA_OK;
    a.stream = static_cast<cudaStream_t>(stream);
    a.wait_ns = pa::g_wait_ns.load(std::memory_order_relaxed);
    a.withhold_loads = pa::g_withhold.load(std::memory_order_relaxed);
    if (a.total_q == 0 || a.batch == 0) return PA_OK;

    unsigned int* err = nullptr;
    int ce = pa::error_word(&err);
    if (ce != cudaSuccess) return fail(PA_ERR_CUDA, "error word: %s", cudaGetErrorString((cudaError_t)ce));

    const bool use_prefill = pa::prefill_supported(a);
    // SMs the persistent prefill grid may hold beside the decode-class pass (it runs before
    // that pass, not beside it, when there is no side stream)
    const int prefill_sms =
        use_prefill && side_stream_ok ? (int)std::min<int64_t>(sm_count(), pa::prefill_items_bound(a)) : 0;
    const pa::SplitPlan plan = pa::plan_splitkv(a, use_prefill, prefill_sms, sm_count());
    // the prefill kernels' item counter follows the split-KV scratch
    const size_t counter_at = (plan.ws_bytes + 255) / 256 * 256;
    const size_t ws_bytes = use_prefill ? counter_at + pa::kPrefillCounterBytes : plan.ws_bytes;
    void* ws = nullptr;
    if (ws_bytes) {
        rc = scratch(scratch_ctx, a.stream, ws_bytes, &ws, g_msg, sizeof g_msg);
        if (rc != PA_OK) return rc;
    }
    int* counter = use_prefill ? reinterpret_cast<int*>(static_cast<char*>(ws) + counter_at) : nullptr;
    if (!use_prefill || !side_stream_ok) {
        if (use_prefill && (rc = pa::launch_prefill(a, counter, err, g_msg, sizeof g_msg)) != PA_OK) return rc;
        rc = pa::launch_splitkv(a, plan, ws, err, g_msg, sizeof g_msg);
        if (rc != PA_OK) return rc;
        g_msg[0] = '\0';
        return PA_OK;
    }
    // prefill-class sequences on the side stream, decode-class ones on the caller's stream
    SideStream* ss = nullptr;
    if ((rc = side_stream(a.stream, &ss)) != PA_OK) return rc;
    std::lock_guard<std::mutex> lock(ss->mu);
    cudaError_t e = cudaEventRecord(ss->fork, a.stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ss->stream, ss->fork, 0);
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "forking the prefill stream: %s", cudaGetErrorString(e));
    pa::Args ap = a;
    ap.stream = ss->stream;
    rc = pa::launch_prefill(ap, counter, err, g_msg, sizeof g_msg);
    if (rc == PA_OK) rc = pa::launch_splitkv(a, plan, ws, err, g_msg, sizeof g_msg);
    // join even after a failed launch, so the caller's stream never runs ahead of the side stream
    e = cudaEventRecord(ss->join, ss->stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(a.stream, ss->join, 0);
    if (rc != PA_OK) return rc;
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "joining the prefill stream: %s", cudaGetErrorString(e));
    g_msg[0] = '\0';
    return PA_OK;
}

}  // namespace pa

// ---- padded (non-varlen) entry point ---------------------------------------------------------
namespace {

// A rank-3 descriptor of a rank-4 (batch, seq, heads, dim) tensor whose batch and sequence
// dimensions can be merged (batch stride = seq * seq stride).
pa_tensor merged(const pa_tensor* t) {
    pa_tensor m = *t;
    m.ndim = 3;
    m.shape[0] = t->shape[0] * t->shape[1];
    m.shape[1] = t->shape[2];
    m.shape[2] = t->shape[3];
    m.stride[0] = t->stride[1];
    m.stride[1] = t->stride[2];
    m.stride[2] = t->stride[3];
    m.shape[3] = m.stride[3] = 0;
    return m;
}

bool mergeable(const pa_tensor* t) { return t->shape[0] <= 1 || t->shape[1] <= 1 || t->stride[0] == t->shape[1] * t->stride[1]; }

int padded_common(const pa_tensor* q, const pa_tensor* k, const pa_tensor* v, int32_t num_heads, int32_t num_heads_k,
                  int32_t head_dim, float softmax_scale, int32_t wl, int32_t wr, const pa_tensor* alibi,
                  const pa_tensor* out, const pa_tensor* lse, bool check_device, void* cu_storage, pa::Args* a) {
    if (!q || !k || !v || !out || !lse) return fail(PA_ERR_ARG, "a tensor descriptor is NULL (only alibi_slopes may be)");
    if (q->ndim != 4 || k->ndim != 4 || v->ndim != 4)
        return fail(PA_ERR_RANK, "flash-attn expects input tensors of rank 4 (q: %d, k: %d, v: %d)", q->ndim, k->ndim,
                    v->ndim);
    for (const pa_tensor* t : {q, k, v})
        if (t->stride[3] != 1)
            return fail(PA_ERR_NONCONTIG, "the last dim of %s must be contiguous %s", t == q ? "q" : t == k ? "k" : "v",
                        strides(t).c_str());
    if (!same_shape(k, v)) return fail(PA_ERR_SHAPE, "shape mismatch k %s and v %s", dims(k).c_str(), dims(v).c_str());
    if (k->shape[0] != q->shape[0] || k->shape[3] != q->shape[3])
        return fail(PA_ERR_SHAPE, "shape mismatch q %s and k %s", dims(q).c_str(), dims(k).c_str());
    if (out->ndim != 4 || !same_shape(out, q))
        return fail(PA_ERR_ARG, "out must have q's shape %s, got %s", dims(q).c_str(), dims(out).c_str());
    const int64_t B = q->shape[0], Sq = q->shape[1], Sk = k->shape[1], H = q->shape[2];
    if (lse->ndim != 3 || lse->shape[0] != B || lse->shape[1] != H || lse->shape[2] != Sq || lse->stride[2] != 1)
        return fail(PA_ERR_ARG, "softmax_lse must be (batch, num_heads, seqlen_q) = (%lld, %lld, %lld) with a contiguous "
                    "last dim", (long long)B, (long long)H, (long long)Sq);
    for (const pa_tensor* t : {q, k, v, out})
        if (!mergeable(t))
            return fail(PA_ERR_UNSUPPORTED, "batch stride must equal seqlen * sequence stride %s", strides(t).c_str());
    if (Sq > INT32_MAX / (B > 0 ? B : 1) || Sk > INT32_MAX / (B > 0 ? B : 1))
        return fail(PA_ERR_UNSUPPORTED, "batch * seqlen beyond 2^31 is not supported");
    const pa_tensor q3 = merged(q), k3 = merged(k), v3 = merged(v), o3 = merged(out);
    pa_tensor l2 = *lse;  // (H, B Sq) view for the shared checks; the batch offset is set below
    l2.ndim = 2;
    l2.shape[0] = H;
    l2.shape[1] = B * Sq;
    l2.stride[0] = lse->stride[1];
    l2.stride[1] = 1;
    pa_tensor cq{}, ck{};
    cq.data = cu_storage;
    ck.data = cu_storage ? static_cast<int32_t*>(cu_storage) + (B + 1) : nullptr;
    cq.dtype = ck.dtype = PA_I32;
    cq.ndim = ck.ndim = 1;
    cq.shape[0] = ck.shape[0] = B + 1;
    cq.stride[0] = ck.stride[0] = 1;
    int rc = validate(&q3, &k3, &v3, &cq, &ck, nullptr, (int32_t)Sq, (int32_t)Sk, num_heads, num_heads_k, head_dim, 0,
                      softmax_scale, wl, wr, alibi, &o3, &l2, check_device, a);
    if (rc != PA_OK) return rc;
    // token t = b Sq + i of head h lands at b lse.stride[0] + h lse.stride[1] + i
    a->lse_sb = lse->stride[0] - Sq;
    return PA_OK;
}

}  // namespace

extern "C" {

int pa_varlen_check(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                    const pa_tensor* cu_seqlens_q, const pa_tensor* cu_seqlens_k, const pa_tensor* block_table,
                    int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_heads, int32_t num_heads_k,
                    int32_t head_dim, int32_t page_block_size, float softmax_scale, int32_t window_left,
                    int32_t window_right, const pa_tensor* out, const pa_tensor* softmax_lse) {
    return pa_varlen_check_alibi(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_table, max_seqlen_q,
                                 max_seqlen_k, num_heads, num_heads_k, head_dim, page_block_size, softmax_scale,
                                 window_left, window_right, nullptr, out, softmax_lse);
}

int pa_varlen_check_alibi(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                          const pa_tensor* cu_seqlens_q, const pa_tensor* cu_seqlens_k, const pa_tensor* block_table,
                          int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_heads, int32_t num_heads_k,
                          int32_t head_dim, int32_t page_block_size, float softmax_scale, int32_t window_left,
                          int32_t window_right, const pa_tensor* alibi_slopes, const pa_tensor* out,
                          const pa_tensor* softmax_lse) {
    pa::Args a{};
    return validate(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_table, max_seqlen_q, max_seqlen_k,
                    num_heads, num_heads_k, head_dim, page_block_size, softmax_scale, window_left, window_right,
                    alibi_slopes, out, softmax_lse, false, &a);
}

int pa_varlen_fwd(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                  const pa_tensor* cu_seqlens_q, const pa_tensor* cu_seqlens_k, const pa_tensor* block_table,
                  int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_heads, int32_t num_heads_k,
                  int32_t head_dim, int32_t page_block_size, float softmax_scale, int32_t window_left,
                  int32_t window_right, const pa_tensor* out, const pa_tensor* softmax_lse, void* stream) {
    return pa::forward_impl(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_table, max_seqlen_q,
                            max_seqlen_k, num_heads, num_heads_k, head_dim, page_block_size, softmax_scale,
                            window_left, window_right, nullptr, out, softmax_lse, stream, library_workspace,
                            nullptr, true);
}

int pa_varlen_fwd_alibi(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                        const pa_tensor* cu_seqlens_q, const pa_tensor* cu_seqlens_k, const pa_tensor* block_table,
                        int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_heads, int32_t num_heads_k,
                        int32_t head_dim, int32_t page_block_size, float softmax_scale, int32_t window_left,
                        int32_t window_right, const pa_tensor* alibi_slopes, const pa_tensor* out,
                        const pa_tensor* softmax_lse, void* stream) {
    return pa::forward_impl(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_table, max_seqlen_q,
                            max_seqlen_k, num_heads, num_heads_k, head_dim, page_block_size, softmax_scale,
                            window_left, window_right, alibi_slopes, out, softmax_lse, stream, library_workspace,
                            nullptr, true);
}

// ---- padded (non-varlen) entry points ----
int pa_check_padded(const pa_tensor* q, const pa_tensor* k, const pa_tensor* v, int32_t num_heads, int32_t num_heads_k,
                    int32_t head_dim, float softmax_scale, int32_t window_left, int32_t window_right,
                    const pa_tensor* alibi_slopes, const pa_tensor* out, const pa_tensor* softmax_lse) {
    pa::Args a{};
    static int32_t fake_cu[1];  // never dereferenced by the host checks
    return padded_common(q, k, v, num_heads, num_heads_k, head_dim, softmax_scale, window_left, window_right,
                         alibi_slopes, out, softmax_lse, false, fake_cu, &a);
}

int pa_fwd_padded(const pa_tensor* q, const pa_tensor* k, const pa_tensor* v, int32_t num_heads, int32_t num_heads_k,
                  int32_t head_dim, float softmax_scale, int32_t window_left, int32_t window_right,
                  const pa_tensor* alibi_slopes, const pa_tensor* out, const pa_tensor* softmax_lse, void* stream) {
    if (!q || q->ndim != 4)
        return pa_check_padded(q, k, v, num_heads, num_heads_k, head_dim, softmax_scale, window_left, window_right,
                               alibi_slopes, out, softmax_lse);
    pa::NvtxRange range("pa_fwd_padded");
    const int64_t B = q->shape[0];
    void* cu = nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the host checks first, so that a bad call allocates nothing
    int rc = pa_check_padded(q, k, v, num_heads, num_heads_k, head_dim, softmax_scale, window_left, window_right,
                             alibi_slopes, out, softmax_lse);
    if (rc != PA_OK) return rc;
    if ((rc = grow_buffer(g_cu, s, (size_t)(2 * (B + 1)) * sizeof(int32_t), &cu)) != PA_OK) return rc;
    pa::Args a{};
    rc = padded_common(q, k, v, num_heads, num_heads_k, head_dim, softmax_scale, window_left, window_right,
                       alibi_slopes, out, softmax_lse, true, cu, &a);
    if (rc != PA_OK) return rc;
    if (a.total_q == 0 || a.batch == 0) return PA_OK;
    rc = pa::launch_uniform_cu(static_cast<int32_t*>(cu), static_cast<int32_t*>(cu) + (B + 1), (int)B,
                               (int)q->shape[1], (int)k->shape[1], s, g_msg, sizeof g_msg);
    if (rc != PA_OK) return rc;
    return pa::launch_forward(a, stream, library_workspace, nullptr, true);
}

int pa_kv_append_check(const pa_tensor* k_new, const pa_tensor* v_new, const pa_tensor* cu_seqlens_new,
                       const pa_tensor* cu_seqlens_k, const pa_tensor* block_table, const pa_tensor* k_cache,
                       const pa_tensor* v_cache, int32_t page_block_size) {
    pa::AppendArgs a{};
    return validate_append(k_new, v_new, cu_seqlens_new, cu_seqlens_k, block_table, k_cache, v_cache,
                           page_block_size, false, &a);
}

int pa_kv_append(const pa_tensor* k_new, const pa_tensor* v_new, const pa_tensor* cu_seqlens_new,
                 const pa_tensor* cu_seqlens_k, const pa_tensor* block_table, const pa_tensor* k_cache,
                 const pa_tensor* v_cache, int32_t page_block_size, void* stream) {
    pa::NvtxRange range("pa_kv_append");
    pa::AppendArgs a{};
    int rc = validate_append(k_new, v_new, cu_seqlens_new, cu_seqlens_k, block_table, k_cache, v_cache,
                             page_block_size, true, &a);
    if (rc != PA_OK) return rc;
    a.stream = static_cast<cudaStream_t>(stream);
    unsigned int* err = nullptr;
    int ce = pa::error_word(&err);
    if (ce != cudaSuccess) return fail(PA_ERR_CUDA, "error word: %s", cudaGetErrorString((cudaError_t)ce));
    rc = pa::launch_kv_append(a, err, g_msg, sizeof g_msg);
    if (rc == PA_OK) g_msg[0] = '\0';
    return rc;
}

const char* pa_last_error(void) { return g_msg; }

int pa_device_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
    unsigned int* word = nullptr;
    int ce = pa::error_word(&word);
    if (ce != cudaSuccess) return fail(PA_ERR_CUDA, "error word: %s", cudaGetErrorString((cudaError_t)ce));
    unsigned int v = 0;
    e = cudaMemcpy(&v, word, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "reading the error word: %s", cudaGetErrorString(e));
    if (!v) {
        g_msg[0] = '\0';
        return PA_OK;
    }
    e = cudaMemset(word, 0, sizeof v);
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "clearing the error word: %s", cudaGetErrorString(e));
    const int code = (int)(v & 0xffu);
    if (code == PA_ERR_DEVICE_TIMEOUT)
        return fail(code, "a kernel gave up a bounded wait (its output is undefined)");
    return fail(code, "a kernel met out-of-range metadata (block id, page, cu_seqlens or max_seqlen); "
                      "that work was skipped and its output is undefined");
}

int pa_version(void) { return 100; }

void pa_set_wait_limit_ns(uint64_t ns) { pa::g_wait_ns.store(ns ? ns : PA_WAIT_LIMIT_NS); }

void pa_set_withhold_loads(int enable) { pa::g_withhold.store(enable ? 1 : 0); }

uint64_t pa_kernel_launches(void) { return pa::g_launches.load(std::memory_order_relaxed); }

void pa_kernel_timing(int enable) { pa::g_timing.store(enable ? 1 : 0, std::memory_order_relaxed); }

int pa_kernel_times(double* ms, uint64_t* launches) {
    if (!ms || !launches) return fail(PA_ERR_ARG, "pa_kernel_times: null output array");
    for (int c = 0; c < PA_KERNEL_CLASSES; ++c) {
        ms[c] = 0.0;
        launches[c] = 0;
    }
    std::lock_guard<std::mutex> lock(pa::g_timer_mu);
    if (pa::g_timed.empty()) return PA_OK;
    int prev = 0;
    cudaGetDevice(&prev);
    int rc = PA_OK;
    for (const auto& t : pa::g_timed) {
        float el = 0.f;
        cudaError_t e = cudaSetDevice(t.dev);
        if (e == cudaSuccess) e = cudaEventSynchronize(t.end);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&el, t.begin, t.end);
        if (e != cudaSuccess && rc == PA_OK)
            rc = fail(PA_ERR_CUDA, "pa_kernel_times: %s", cudaGetErrorString(e));
        if (e == cudaSuccess && t.cls >= 0 && t.cls < PA_KERNEL_CLASSES) {
            ms[t.cls] += el;
            launches[t.cls] += 1;
        }
        pa::g_event_pool.emplace_back(t.dev, t.begin);
        pa::g_event_pool.emplace_back(t.dev, t.end);
    }
    pa::g_timed.clear();
    cudaSetDevice(prev);
    return rc;
}

}  // extern "C"
