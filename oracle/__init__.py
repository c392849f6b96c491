"""Oracle for paged-KV varlen attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product library never loads it.  It wraps the
plain fp64 C restatement in ``pa_oracle.c`` (which cites the pages it follows)
and shares no code with the CUDA library.

Parity pins: every function here is pinned by ``tests/test_oracle.py`` against
closed forms, library routines (numpy masks, torch SDPA in float64) and
invariances; none is "parity unpinned".  ``kv_append`` (a plain numpy scatter) is
pinned by a gather through the block table written independently in the tests and by
the attention oracle's non-paged mode.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libpa_oracle.so")
_lib = None

DTYPES = {"f16": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load(path: str):
    """Open an oracle library at ``path`` (the tests also open mutated builds this way)."""
    lib = ctypes.CDLL(path)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i32p = ctypes.POINTER(ctypes.c_int32)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    lib.pa_oracle_fwd.restype = ctypes.c_int
    lib.pa_oracle_fwd.argtypes = [
        ctypes.c_int, u16p, i64p, u16p, u16p, i64p, i32p, i32p, ctypes.c_int64,
        i32p, ctypes.c_int64, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_double, ctypes.c_int, ctypes.c_int, f64p, i64p, ctypes.c_int64, f64p, f64p,
    ]
    lib.pa_oracle_threads.restype = ctypes.c_int
    lib.pa_oracle_decode.restype = ctypes.c_double
    lib.pa_oracle_decode.argtypes = [ctypes.c_int, ctypes.c_uint16]
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = load(build())
    return _lib


def threads() -> int:
    """Threads the oracle's OpenMP loop uses."""
    return _load().pa_oracle_threads()


def decode(dtype: str, bits: int, lib=None) -> float:
    """The oracle's own fp16 / bf16 bit decoder (pinned against numpy and torch)."""
    lib = lib if lib is not None else _load()
    return lib.pa_oracle_decode(DTYPES[dtype], int(bits) & 0xFFFF)


def _bits(a) -> np.ndarray:
    """Raw 16-bit patterns of an fp16/bf16 array (numpy or torch CPU tensor)."""
    if hasattr(a, "detach"):  # torch tensor: reinterpret without importing torch here
        a = a.detach().contiguous().cpu()
        return np.ascontiguousarray(a.view(dtype=__import__("torch").int16).numpy().view(np.uint16))
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype in (np.uint16, np.int16):
        return a.view(np.uint16)
    raise TypeError(f"oracle wants fp16/bf16 data, got {a.dtype}")


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def attention(dtype, q, k, v, cu_seqlens_q, cu_seqlens_k, block_table, softmax_scale,
              window_left=-1, window_right=0, rows=None, lib=None, alibi_slopes=None):
    """Masked softmax attention through the block table, in fp64.

    q: (total_q, H, D); k, v: (num_blocks, P, Hkv, D) when ``block_table`` is given,
    else (total_k, Hkv, D).  Arrays are fp16/bf16 (torch CPU tensors or numpy fp16
    or uint16 bit patterns), contiguous.  ``rows``: optional int64 array of
    token * H + head.  Returns (out float64 [n, D], lse float64 [n]) where n is
    len(rows) or total_q * H (row r = token * H + head).  ``alibi_slopes``: optional
    per-query-head slopes (H values); the score of query i and key j then gets
    -slope_h * |i + sk - sq - j|.
    """
    lib = lib if lib is not None else _load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    if qb.ndim != 3:
        raise ValueError("q must be (total_q, num_heads, head_dim)")
    total_q, H, D = qb.shape
    paged = block_table is not None
    if paged and kb.ndim != 4:
        raise ValueError("paged k/v must be (num_blocks, page_block_size, num_heads_k, head_dim)")
    if not paged and kb.ndim != 3:
        raise ValueError("non-paged k/v must be (total_k, num_heads_k, head_dim)")
    if kb.shape != vb.shape:
        raise ValueError("k and v shapes differ")
    Hkv = kb.shape[-2]
    cu_q = np.ascontiguousarray(np.asarray(cu_seqlens_q, dtype=np.int32))
    cu_k = np.ascontiguousarray(np.asarray(cu_seqlens_k, dtype=np.int32))
    batch = len(cu_q) - 1
    if int(cu_q[-1]) != total_q:
        raise ValueError("cu_seqlens_q[-1] must equal total_q")
    q_stride = np.array([H * D, D], dtype=np.int64)
    if paged:
        P = kb.shape[1]
        kv_stride = np.array([P * Hkv * D, Hkv * D, D], dtype=np.int64)
        bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
        if bt.ndim != 2:
            raise ValueError("block_table must be (batch, max_pages)")
        bt_ptr, bt_stride = _ptr(bt, ctypes.c_int32), bt.shape[1]
    else:
        P = 0
        kv_stride = np.array([Hkv * D, D, 0], dtype=np.int64)
        bt, bt_ptr, bt_stride = None, None, 0
    if rows is None:
        n = total_q * H
        rows_arr, rows_ptr = None, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = len(rows_arr)
        rows_ptr = _ptr(rows_arr, ctypes.c_int64)
    if alibi_slopes is not None:
        slopes = np.ascontiguousarray(np.asarray(alibi_slopes, dtype=np.float64).reshape(-1))
        if slopes.shape != (H,):
            raise ValueError("alibi_slopes must hold one slope per query head")
        slopes_ptr = _ptr(slopes, ctypes.c_double)
    else:
        slopes, slopes_ptr = None, None
    out = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = lib.pa_oracle_fwd(
        DTYPES[dtype], _ptr(qb, ctypes.c_uint16), _ptr(q_stride, ctypes.c_int64),
        _ptr(kb, ctypes.c_uint16), _ptr(vb, ctypes.c_uint16), _ptr(kv_stride, ctypes.c_int64),
        _ptr(cu_q, ctypes.c_int32), _ptr(cu_k, ctypes.c_int32), batch,
        bt_ptr, bt_stride, P, H, Hkv, D, float(softmax_scale), int(window_left), int(window_right),
        slopes_ptr, rows_ptr, n, _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out, lse


def kv_append(k_new, v_new, cu_seqlens_new, cu_seqlens_k, block_table, k_cache, v_cache):
    """Writes new key/value rows into a paged cache, in place (numpy arrays, any dtype).

    Sequence b owns sk_b = cu_seqlens_k[b+1] - cu_seqlens_k[b] keys after the append, the
    last n_b = cu_seqlens_new[b+1] - cu_seqlens_new[b] of which are its new tokens (the same
    bottom-right alignment as the mask: new token t sits at key position sk_b - n_b + t).
    Logical position j lives at slot j mod P of block block_table[b, j // P] ("flash-attn-
    varlen paged expects k/v tensors of rank 4", What it means: the block table maps a
    sequence's logical pages to physical blocks of the (num_blocks, P, Hkv, D) caches).

    k_new, v_new: (total_new, Hkv, D); k_cache, v_cache: (num_blocks, P, Hkv, D), modified.
    Raises ValueError when a sequence has more new tokens than keys, or a position falls
    outside the block table or the pool.
    """
    cu_new = np.asarray(cu_seqlens_new, dtype=np.int64)
    cu_k = np.asarray(cu_seqlens_k, dtype=np.int64)
    bt = np.asarray(block_table, dtype=np.int64)
    P = k_cache.shape[1]
    for b in range(len(cu_new) - 1):
        n_b = int(cu_new[b + 1] - cu_new[b])
        sk_b = int(cu_k[b + 1] - cu_k[b])
        if n_b > sk_b:
            raise ValueError(f"sequence {b}: {n_b} new tokens but only {sk_b} keys")
        for t in range(n_b):
            j = sk_b - n_b + t
            if j // P >= bt.shape[1]:
                raise ValueError(f"sequence {b}: position {j} is past its block table row")
            blk = int(bt[b, j // P])
            if not 0 <= blk < k_cache.shape[0]:
                raise ValueError(f"sequence {b}: block id {blk} outside the pool")
            k_cache[blk, j % P] = k_new[cu_new[b] + t]
            v_cache[blk, j % P] = v_new[cu_new[b] + t]


def attention_padded(dtype, q, k, v, softmax_scale, window_left=-1, window_right=0, alibi_slopes=None, lib=None):
    """Attention over a padded batch: q (B, Sq, H, D), k and v (B, Sk, Hkv, D), every sequence
    of length Sq / Sk.  By definition this is the varlen attention of the packed tokens with
    uniform cumulative lengths (cu_q[b] = b Sq, cu_k[b] = b Sk) in the non-paged mode, so it
    calls ``attention`` on that packing.  Returns (out float64 (B, Sq, H, D), lse float64
    (B, H, Sq))."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    if qb.ndim != 4 or kb.ndim != 4 or kb.shape != vb.shape:
        raise ValueError("q must be (B, Sq, H, D) and k, v (B, Sk, Hkv, D) of one shape")
    B, Sq, H, D = qb.shape
    Sk, Hkv = kb.shape[1], kb.shape[2]
    cu_q = np.arange(B + 1, dtype=np.int32) * Sq
    cu_k = np.arange(B + 1, dtype=np.int32) * Sk
    out, lse = attention(dtype, qb.reshape(B * Sq, H, D), kb.reshape(B * Sk, Hkv, D), vb.reshape(B * Sk, Hkv, D),
                         cu_q, cu_k, None, softmax_scale, window_left, window_right, lib=lib,
                         alibi_slopes=alibi_slopes)
    return out.reshape(B, Sq, H, D), lse.reshape(B, Sq, H).transpose(0, 2, 1).copy()
