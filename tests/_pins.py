"""Pins that tie the oracle to something other than itself.

Each pin takes an ``attn`` callable with the signature of ``oracle.attention``
(optionally bound to a mutated build) and raises AssertionError on a mismatch.
The expected values come from library routines (numpy masks built with
``tril``/``triu``, torch SDPA in float64, numpy gathers and means), closed forms,
or invariances of the definition -- never from the CUDA path.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --- small input builders ---------------------------------------------------------------

def f16(rng, shape, std=1.0):
    return (rng.standard_normal(shape) * std).astype(np.float16)


def cu(lengths):
    c = np.zeros(len(lengths) + 1, dtype=np.int32)
    c[1:] = np.cumsum(lengths)
    return c


def pack_paged(k_tok, seqlens_k, P, rng, spare=3):
    """Lay packed (total_k, Hkv, D) key rows into a shuffled pool of P-slot pages.
    Unowned slots hold NaN.  Returns (pool, block_table)."""
    Hkv, D = k_tok.shape[1:]
    pages = [(s + P - 1) // P for s in seqlens_k]
    nb = sum(pages) + spare
    perm = rng.permutation(nb)
    pool = np.full((nb, P, Hkv, D), np.nan, dtype=k_tok.dtype)
    bt = np.full((len(seqlens_k), max(max(pages), 1)), -1, dtype=np.int32)
    cur, off = 0, 0
    for b, s in enumerate(seqlens_k):
        for p in range(pages[b]):
            blk = perm[cur]
            cur += 1
            bt[b, p] = blk
            n = min(P, s - p * P)
            pool[blk, :n] = k_tok[off + p * P: off + p * P + n]
        off += s
    return pool, bt


def mask_by_library(sq, sk, wl, wr):
    """The bottom-right aligned window mask built from numpy's triangle routines:
    the right bound is a lower triangle at diagonal offset (sk - sq) + wr, the left
    bound an upper triangle at offset (sk - sq) - wl."""
    m = np.ones((sq, sk), dtype=bool)
    c = sk - sq
    if wr >= 0:
        m &= np.tril(np.ones((sq, sk), dtype=bool), k=c + wr)
    if wl >= 0:
        m &= np.triu(np.ones((sq, sk), dtype=bool), k=c - wl)
    return m


def dense_reference(q, k, v, mask, scale):
    """Masked softmax for one head: q (sq, D), k/v (sk, D) float64, mask (sq, sk)."""
    s = scale * (q @ k.T)
    out = np.zeros((q.shape[0], v.shape[1]))
    lse = np.full(q.shape[0], -np.inf)
    for i in range(q.shape[0]):
        if not mask[i].any():
            continue
        si = s[i][mask[i]]
        m = si.max()
        w = np.exp(si - m)
        out[i] = (w[:, None] * v[mask[i]]).sum(0) / w.sum()
        lse[i] = m + math.log(w.sum())
    return out, lse


# --- pins -------------------------------------------------------------------------------

def pin_decoders(decode):
    """Every fp16 bit pattern decodes as numpy's float16; every bf16 pattern as torch's."""
    import torch
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    want16 = bits.view(np.float16).astype(np.float64)
    got16 = np.array([decode("f16", int(b)) for b in bits])
    assert np.array_equal(np.isnan(want16), np.isnan(got16))
    ok = ~np.isnan(want16)
    assert np.array_equal(want16[ok], got16[ok]), "fp16 decoder"
    wantbf = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    gotbf = np.array([decode("bf16", int(b)) for b in bits])
    assert np.array_equal(np.isnan(wantbf), np.isnan(gotbf))
    ok = ~np.isnan(wantbf)
    assert np.array_equal(wantbf[ok], gotbf[ok]), "bf16 decoder"


def pin_mask_bruteforce(attn, paged=False):
    """All sq <= 12, sk <= 12 and wl, wr in {-1, 0, 1, 3}: the oracle equals a dense
    softmax under the numpy-triangle mask (fully masked rows: out 0, lse -inf)."""
    rng = np.random.default_rng(100)
    pairs = [(sq, sk) for sq in range(1, 13) for sk in range(0, 13)]
    sq_list = [p[0] for p in pairs]
    sk_list = [p[1] for p in pairs]
    D, scale = 8, 0.7
    q = f16(rng, (sum(sq_list), 1, D))
    k = f16(rng, (sum(sk_list), 1, D))
    v = f16(rng, (sum(sk_list), 1, D))
    cq, ck = cu(sq_list), cu(sk_list)
    if paged:
        kp, bt = pack_paged(k, sk_list, 32, np.random.default_rng(5))
        vp, _ = pack_paged(v, sk_list, 32, np.random.default_rng(5))
    for wl in (-1, 0, 1, 3):
        for wr in (-1, 0, 1, 3):
            if paged:
                out, lse = attn("f16", q, kp, vp, cq, ck, bt, scale, wl, wr)
            else:
                out, lse = attn("f16", q, k, v, cq, ck, None, scale, wl, wr)
            for b, (sq, sk) in enumerate(pairs):
                m = mask_by_library(sq, sk, wl, wr)
                qq = q[cq[b]:cq[b + 1], 0].astype(np.float64)
                kk = k[ck[b]:ck[b + 1], 0].astype(np.float64)
                vv = v[ck[b]:ck[b + 1], 0].astype(np.float64)
                o_ref, l_ref = dense_reference(qq, kk, vv, m, scale)
                o = out[cq[b]:cq[b + 1]]
                l = lse[cq[b]:cq[b + 1]]
                assert np.allclose(o, o_ref, rtol=1e-12, atol=1e-12), (sq, sk, wl, wr)
                assert np.array_equal(np.isinf(l), np.isinf(l_ref)), (sq, sk, wl, wr)
                fin = np.isfinite(l_ref)
                assert np.allclose(l[fin], l_ref[fin], rtol=1e-12, atol=1e-12), (sq, sk, wl, wr)


def pin_sdpa(attn):
    """One sequence, no paging: the oracle equals torch's scaled_dot_product_attention
    in float64 (full, causal with sq == sk, and grouped-query heads); lse equals
    torch.logsumexp of the scaled scores."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(101)
    for H, Hkv, causal in ((3, 3, False), (3, 3, True), (4, 2, False), (6, 2, True)):
        S, D, scale = 37, 16, 0.3
        q = f16(rng, (S, H, D))
        k = f16(rng, (S, Hkv, D))
        v = f16(rng, (S, Hkv, D))
        wl, wr = (-1, 0) if causal else (-1, -1)
        out, lse = attn("f16", q, k, v, cu([S]), cu([S]), None, scale, wl, wr)
        tq = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)[None]
        tk = torch.from_numpy(k.astype(np.float64)).permute(1, 0, 2)[None]
        tv = torch.from_numpy(v.astype(np.float64)).permute(1, 0, 2)[None]
        ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale,
                                             enable_gqa=(H != Hkv))
        ref = ref[0].permute(1, 0, 2).reshape(S * H, D).numpy()
        assert np.allclose(out, ref, rtol=1e-10, atol=1e-12), (H, Hkv, causal)
        if not causal:
            G = H // Hkv
            tk_rep = tk.repeat_interleave(G, dim=1)
            sc = scale * (tq @ tk_rep.transpose(-1, -2))
            lref = torch.logsumexp(sc, dim=-1)[0].permute(1, 0).reshape(-1).numpy()
            assert np.allclose(lse, lref, rtol=1e-12, atol=1e-12)


def _multi_seq(rng, Hkv=2, H=4, D=16, dtype=np.float16):
    sq = [1, 5, 9, 1, 12]
    sk = [1, 40, 70, 97, 12]
    q = f16(rng, (sum(sq), H, D))
    k = f16(rng, (sum(sk), Hkv, D))
    v = f16(rng, (sum(sk), Hkv, D))
    return sq, sk, q, k, v


def pin_paging_identity(attn):
    """Paged mode through any block table equals the packed rank-3 (non-paged) result,
    bit for bit, for several page sizes and windows."""
    rng = np.random.default_rng(102)
    sq, sk, q, k, v = _multi_seq(rng)
    for P in (32, 64):
        kp, bt = pack_paged(k, sk, P, np.random.default_rng(P))
        vp, _ = pack_paged(v, sk, P, np.random.default_rng(P))
        for wl, wr in ((-1, 0), (-1, -1), (5, 2)):
            o1, l1 = attn("f16", q, k, v, cu(sq), cu(sk), None, 0.25, wl, wr)
            o2, l2 = attn("f16", q, kp, vp, cu(sq), cu(sk), bt, 0.25, wl, wr)
            assert np.array_equal(o1, o2) and np.array_equal(l1, l2), (P, wl, wr)


def pin_block_permutation(attn):
    """Permuting the physical blocks, with the table rewritten to match, leaves out and lse
    bit-identical."""
    rng = np.random.default_rng(103)
    sq, sk, q, k, v = _multi_seq(rng)
    kp, bt = pack_paged(k, sk, 32, np.random.default_rng(7))
    vp, _ = pack_paged(v, sk, 32, np.random.default_rng(7))
    perm = np.random.default_rng(8).permutation(kp.shape[0])
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    bt2 = bt.copy()
    bt2[bt >= 0] = perm[bt[bt >= 0]]
    o1, l1 = attn("f16", q, kp, vp, cu(sq), cu(sk), bt, 0.25, -1, 0)
    o2, l2 = attn("f16", q, kp[inv], vp[inv], cu(sq), cu(sk), bt2, 0.25, -1, 0)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def pin_rows_sum_to_one(attn):
    """V = 1 everywhere gives out = 1 in every row with an attended key (softmax rows sum to 1)."""
    rng = np.random.default_rng(104)
    sq, sk, q, k, v = _multi_seq(rng)
    ones = np.ones_like(v)
    for wl, wr in ((-1, 0), (3, 0), (-1, -1)):
        out, lse = attn("f16", q, k, ones, cu(sq), cu(sk), None, 0.25, wl, wr)
        live = np.isfinite(lse)
        assert live.any()
        assert np.allclose(out[live], 1.0, rtol=0, atol=1e-14)
        assert np.all(out[~live] == 0.0)


def pin_zero_query(attn):
    """q = 0 makes every attended score 0: out is the plain mean of the attended value rows
    (numpy gather + mean) and lse = ln |J|."""
    rng = np.random.default_rng(105)
    sq, sk, q, k, v = _multi_seq(rng)
    q0 = np.zeros_like(q)
    H, Hkv = q.shape[1], k.shape[1]
    G = H // Hkv
    for wl, wr in ((-1, 0), (4, 1)):
        out, lse = attn("f16", q0, k, v, cu(sq), cu(sk), None, 0.25, wl, wr)
        out = out.reshape(len(q), H, -1)
        lse = lse.reshape(len(q), H)
        cq, ck = cu(sq), cu(sk)
        for b in range(len(sq)):
            m = mask_by_library(sq[b], sk[b], wl, wr)
            for i in range(sq[b]):
                for h in range(H):
                    rows = v[ck[b]:ck[b + 1], h // G][m[i]].astype(np.float64)
                    t = cq[b] + i
                    if len(rows) == 0:
                        assert lse[t, h] == -np.inf
                        continue
                    assert np.allclose(out[t, h], rows.mean(0), rtol=1e-12, atol=1e-13)
                    assert abs(lse[t, h] - math.log(len(rows))) < 1e-12


def pin_single_key(attn):
    """Window (0, 0) leaves exactly key i + sk - sq: out is that value row and lse its score."""
    rng = np.random.default_rng(106)
    sq, sk, q, k, v = _multi_seq(rng)
    H, Hkv = q.shape[1], k.shape[1]
    G = H // Hkv
    out, lse = attn("f16", q, k, v, cu(sq), cu(sk), None, 0.25, 0, 0)
    out = out.reshape(len(q), H, -1)
    lse = lse.reshape(len(q), H)
    cq, ck = cu(sq), cu(sk)
    for b in range(len(sq)):
        for i in range(sq[b]):
            j = i + sk[b] - sq[b]
            for h in range(H):
                t = cq[b] + i
                if j < 0:
                    assert lse[t, h] == -np.inf
                    continue
                krow = k[ck[b] + j, h // G].astype(np.float64)
                vrow = v[ck[b] + j, h // G].astype(np.float64)
                assert np.array_equal(out[t, h], vrow)
                assert abs(lse[t, h] - 0.25 * float(np.dot(q[t, h].astype(np.float64), krow))) < 1e-12


def pin_gqa_repeat(attn):
    """Grouped-query heads equal multi-head attention on the kv heads repeated G times
    (query head h reads kv head h // G)."""
    rng = np.random.default_rng(107)
    sq, sk, q6, _, _ = _multi_seq(rng, Hkv=2, H=6)
    k = f16(rng, (sum(sk), 2, 16))
    v = f16(rng, (sum(sk), 2, 16))
    o1, l1 = attn("f16", q6, k, v, cu(sq), cu(sk), None, 0.25, -1, 0)
    o2, l2 = attn("f16", q6, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), cu(sq), cu(sk),
                  None, 0.25, -1, 0)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def pin_chunking(attn):
    """Chunked prefill: queries [a, b) of a sequence run against its first b keys reproduce
    rows a..b-1 of the full causal prefill (bottom-right alignment)."""
    rng = np.random.default_rng(108)
    S, H, D = 50, 2, 16
    q = f16(rng, (S, H, D))
    k = f16(rng, (S, 1, D))
    v = f16(rng, (S, 1, D))
    full_o, full_l = attn("f16", q, k, v, cu([S]), cu([S]), None, 0.25, -1, 0)
    bounds = [(0, 20), (20, 35), (35, 50)]
    # three sequences: each chunk's queries, keys 0..end of the same sequence
    qc = np.concatenate([q[a:b] for a, b in bounds])
    kc = np.concatenate([k[:b] for _, b in bounds])
    vc = np.concatenate([v[:b] for _, b in bounds])
    o, l = attn("f16", qc, kc, vc, cu([b - a for a, b in bounds]), cu([b for _, b in bounds]),
                None, 0.25, -1, 0)
    assert np.array_equal(o, full_o) and np.array_equal(l, full_l)


def pin_closed_form(attn):
    """Worked two-key example from tests/golden/closed_form_two_keys.json."""
    with open(os.path.join(GOLDEN, "closed_form_two_keys.json")) as f:
        g = json.load(f)
    q = np.array(g["q"], dtype=np.float16)[:, None, :]
    k = np.array(g["k"], dtype=np.float16)[:, None, :]
    v = np.array(g["v"], dtype=np.float16)[:, None, :]
    out, lse = attn("f16", q, k, v, cu([1]), cu([2]), None, g["softmax_scale"], -1, -1)
    assert np.allclose(out[0], g["out"], rtol=0, atol=1e-15)
    assert abs(lse[0] - g["lse"]) < 1e-15


def pin_bf16_path(attn):
    """bf16 inputs: the oracle equals the dense reference on the bf16 values (via torch's
    bf16 -> float64 conversion)."""
    import torch
    rng = np.random.default_rng(109)
    sq, sk = [3, 7], [20, 7]
    D = 8
    qt = torch.from_numpy(rng.standard_normal((sum(sq), 1, D)).astype(np.float32)).bfloat16()
    kt = torch.from_numpy(rng.standard_normal((sum(sk), 1, D)).astype(np.float32)).bfloat16()
    vt = torch.from_numpy(rng.standard_normal((sum(sk), 1, D)).astype(np.float32)).bfloat16()
    out, lse = attn("bf16", qt, kt, vt, cu(sq), cu(sk), None, 0.5, -1, 0)
    cq, ck = cu(sq), cu(sk)
    for b in range(2):
        m = mask_by_library(sq[b], sk[b], -1, 0)
        o_ref, l_ref = dense_reference(qt[cq[b]:cq[b + 1], 0].double().numpy(),
                                       kt[ck[b]:ck[b + 1], 0].double().numpy(),
                                       vt[ck[b]:ck[b + 1], 0].double().numpy(), m, 0.5)
        assert np.allclose(out[cq[b]:cq[b + 1]], o_ref, rtol=1e-12, atol=1e-13)
        assert np.allclose(lse[cq[b]:cq[b + 1]], l_ref, rtol=1e-12, atol=1e-13)


def alibi_bias_matrix(sq, sk, slope):
    """-slope * (distance of key j from query i's bottom-right aligned diagonal), built
    with numpy's outer difference of the two position ranges."""
    diag = np.arange(sq, dtype=np.float64) + (sk - sq)
    return -slope * np.abs(np.subtract.outer(diag, np.arange(sk, dtype=np.float64)))


def pin_alibi_sdpa(attn):
    """Linear position bias: the oracle equals torch's scaled_dot_product_attention in
    float64 with the bias (and -inf outside the window) as an additive float mask, per
    sequence (sq < sk, so the bottom-right offset matters) and per query head (distinct
    slopes under grouped-query heads); lse equals torch.logsumexp of the biased scores."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(111)
    H, Hkv, D, scale = 4, 2, 16, 0.35
    slopes = np.array([0.5, 0.125, 0.03125, 0.0078125])
    sq, sk = [1, 6, 9], [13, 30, 9]
    q = f16(rng, (sum(sq), H, D))
    k = f16(rng, (sum(sk), Hkv, D))
    v = f16(rng, (sum(sk), Hkv, D))
    cq, ck = cu(sq), cu(sk)
    for wl, wr in ((-1, 0), (-1, -1), (5, 2)):
        out, lse = attn("f16", q, k, v, cq, ck, None, scale, wl, wr, alibi_slopes=slopes)
        for b in range(len(sq)):
            allowed = mask_by_library(sq[b], sk[b], wl, wr)
            for h in range(H):
                hk = h // (H // Hkv)
                bias = np.where(allowed, alibi_bias_matrix(sq[b], sk[b], slopes[h]), -np.inf)
                tq = torch.from_numpy(q[cq[b]:cq[b + 1], h].astype(np.float64))
                tk = torch.from_numpy(k[ck[b]:ck[b + 1], hk].astype(np.float64))
                tv = torch.from_numpy(v[ck[b]:ck[b + 1], hk].astype(np.float64))
                tb = torch.from_numpy(bias)
                live = allowed.any(axis=1)
                ref = F.scaled_dot_product_attention(tq[None], tk[None], tv[None], attn_mask=tb[None],
                                                     scale=scale)[0].numpy()
                lref = torch.logsumexp(scale * (tq @ tk.T) + tb, dim=-1).numpy()
                rows = (cq[b] + np.arange(sq[b])) * H + h
                assert np.allclose(out[rows][live], ref[live], rtol=1e-10, atol=1e-12), (wl, wr, b, h)
                assert np.allclose(lse[rows][live], lref[live], rtol=1e-12, atol=1e-12), (wl, wr, b, h)
                assert np.all(np.isneginf(lse[rows][~live])) and np.all(out[rows][~live] == 0)


def pin_alibi_two_keys(attn):
    """Closed forms with equal scores, so only the bias separates the keys.  q = (1, 0.5)
    and every key (1, 1): each score is 0.5 * 1.5 = 0.75.  (a) sq = 1, sk = 2, causal:
    the query's diagonal is key 1, distances 1 and 0.  (b) sq = 1, sk = 4, window (3, 0):
    distances 3, 2, 1, 0."""
    slope = 0.25
    q = np.array([[[1.0, 0.5]]], dtype=np.float16)
    k2 = np.ones((2, 1, 2), dtype=np.float16)
    v2 = np.array([[[4.0, -2.0]], [[2.0, 0.0]]], dtype=np.float16)
    out, lse = attn("f16", q, k2, v2, cu([1]), cu([2]), None, 0.5, -1, 0, alibi_slopes=[slope])
    w = np.exp(0.75 - slope * np.array([1.0, 0.0]))
    assert np.allclose(out[0], (w[:, None] * v2[:, 0].astype(np.float64)).sum(0) / w.sum(), rtol=1e-14, atol=1e-15)
    assert abs(lse[0] - math.log(w.sum())) < 1e-14
    k4 = np.ones((4, 1, 2), dtype=np.float16)
    v4 = np.array([[[4.0, -2.0]], [[8.0, 8.0]], [[-1.0, 6.0]], [[2.0, 0.0]]], dtype=np.float16)
    out, lse = attn("f16", q, k4, v4, cu([1]), cu([4]), None, 0.5, 3, 0, alibi_slopes=[slope])
    w = np.exp(0.75 - slope * np.array([3.0, 2.0, 1.0, 0.0]))
    assert np.allclose(out[0], (w[:, None] * v4[:, 0].astype(np.float64)).sum(0) / w.sum(), rtol=1e-14, atol=1e-15)
    assert abs(lse[0] - math.log(w.sum())) < 1e-14


def pin_alibi_zero_slopes(attn):
    """Zero slopes leave every output and lse bit-identical to no bias."""
    rng = np.random.default_rng(112)
    sq, sk, q, k, v = _multi_seq(rng)
    a = attn("f16", q, k, v, cu(sq), cu(sk), None, 0.25, -1, 0)
    b = attn("f16", q, k, v, cu(sq), cu(sk), None, 0.25, -1, 0, alibi_slopes=np.zeros(q.shape[1]))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


ALL_PINS = [
    pin_mask_bruteforce,
    lambda a: pin_mask_bruteforce(a, paged=True),
    pin_sdpa,
    pin_paging_identity,
    pin_block_permutation,
    pin_rows_sum_to_one,
    pin_zero_query,
    pin_single_key,
    pin_gqa_repeat,
    pin_chunking,
    pin_closed_form,
    pin_bf16_path,
    pin_alibi_sdpa,
    pin_alibi_two_keys,
    pin_alibi_zero_slopes,
]
