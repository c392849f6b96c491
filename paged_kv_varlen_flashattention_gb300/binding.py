"""ctypes binding of libpa_varlen (argument marshalling only).

Every step of the attention runs in the library's CUDA kernels; this module only
turns torch tensors into ``pa_tensor`` descriptors, passes the current CUDA
stream, and raises :class:`PaError` with the library's message on failure.
There is no fallback: if the library is missing, calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libpa_varlen.so")
_lib = None

PA_F16, PA_BF16, PA_F32, PA_I32 = 0, 1, 2, 3

STATUS = {
    0: "PA_OK", 1: "PA_ERR_RANK", 2: "PA_ERR_RANK_PAGED", 3: "PA_ERR_NONCONTIG", 4: "PA_ERR_SHAPE",
    5: "PA_ERR_PAGE_UNSET", 6: "PA_ERR_PAGE_MISMATCH", 7: "PA_ERR_PAGE_MULT32", 8: "PA_ERR_HEADDIM",
    9: "PA_ERR_NOT_DEVICE", 10: "PA_ERR_ARG", 11: "PA_ERR_UNSUPPORTED", 12: "PA_ERR_CUDA",
    13: "PA_ERR_DEVICE_TIMEOUT", 14: "PA_ERR_DEVICE_BOUNDS", 15: "PA_ERR_WORKSPACE",
}


class PaError(RuntimeError):
    """A non-zero status from the library; ``code`` is the status, ``name`` its enum name."""

    def __init__(self, code: int, message: str):
        self.code = code
        self.name = STATUS.get(code, str(code))
        super().__init__(f"{self.name}: {message}")


class PaTensor(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("ndim", ctypes.c_int32),
        ("shape", ctypes.c_int64 * 4),
        ("stride", ctypes.c_int64 * 4),
    ]


_TP = ctypes.POINTER(PaTensor)
_FWD_ARGS = [_TP, _TP, _TP, _TP, _TP, _TP, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
             ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_int32, ctypes.c_int32, _TP, _TP]
# the same with alibi_slopes between window_right and out
_FWD_ALIBI_ARGS = _FWD_ARGS[:15] + [_TP] + _FWD_ARGS[15:]


def library_path() -> str:
    return _LIB_PATH


def load():
    """Open libpa_varlen.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libpa_varlen.so is not built ({_LIB_PATH}); run __graft_entry__.build()")
        lib = ctypes.CDLL(_LIB_PATH)
        lib.pa_varlen_fwd.restype = ctypes.c_int
        lib.pa_varlen_fwd.argtypes = _FWD_ARGS + [ctypes.c_void_p]
        lib.pa_varlen_check.restype = ctypes.c_int
        lib.pa_varlen_check.argtypes = list(_FWD_ARGS)
        lib.pa_varlen_fwd_alibi.restype = ctypes.c_int
        lib.pa_varlen_fwd_alibi.argtypes = _FWD_ALIBI_ARGS + [ctypes.c_void_p]
        lib.pa_varlen_check_alibi.restype = ctypes.c_int
        lib.pa_varlen_check_alibi.argtypes = list(_FWD_ALIBI_ARGS)
        lib.pa_last_error.restype = ctypes.c_char_p
        lib.pa_device_status.restype = ctypes.c_int
        lib.pa_device_status.argtypes = [ctypes.c_void_p]
        lib.pa_version.restype = ctypes.c_int
        lib.pa_kernel_launches.restype = ctypes.c_uint64
        lib.pa_set_wait_limit_ns.restype = None
        lib.pa_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        lib.pa_set_withhold_loads.restype = None
        lib.pa_set_withhold_loads.argtypes = [ctypes.c_int]
        lib.pa_kv_append.restype = ctypes.c_int
        lib.pa_kv_append.argtypes = [_TP] * 7 + [ctypes.c_int32, ctypes.c_void_p]
        lib.pa_kv_append_check.restype = ctypes.c_int
        lib.pa_kv_append_check.argtypes = [_TP] * 7 + [ctypes.c_int32]
        _PAD = [_TP, _TP, _TP, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_int32,
                ctypes.c_int32, _TP, _TP, _TP]
        lib.pa_fwd_padded.restype = ctypes.c_int
        lib.pa_fwd_padded.argtypes = _PAD + [ctypes.c_void_p]
        lib.pa_check_padded.restype = ctypes.c_int
        lib.pa_check_padded.argtypes = list(_PAD)
        lib.pa_kernel_timing.restype = None
        lib.pa_kernel_timing.argtypes = [ctypes.c_int]
        lib.pa_kernel_times.restype = ctypes.c_int
        lib.pa_kernel_times.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_uint64)]
        _lib = lib
    return _lib


_DTYPE_CODES = None


def _dtype_code(t) -> int:
    global _DTYPE_CODES
    if _DTYPE_CODES is None:
        import torch
        _DTYPE_CODES = {torch.float16: PA_F16, torch.bfloat16: PA_BF16, torch.float32: PA_F32, torch.int32: PA_I32}
    return _DTYPE_CODES.get(t.dtype, -1)


_I64x4 = ctypes.c_int64 * 4


def describe(t) -> Optional[PaTensor]:
    """A pa_tensor descriptor borrowing a torch tensor's storage (None stays None)."""
    if t is None:
        return None
    shape, stride = t.shape, t.stride()
    n = len(shape)
    if n >= 4:
        return PaTensor(t.data_ptr(), _dtype_code(t), n, _I64x4(*shape[:4]), _I64x4(*stride[:4]))
    return PaTensor(t.data_ptr(), _dtype_code(t), n, _I64x4(*shape), _I64x4(*stride))


def _ref(d):
    return ctypes.byref(d) if d is not None else None


def kernel_launches() -> int:
    """Kernels the library has launched in this process so far."""
    return int(load().pa_kernel_launches())


KERNEL_CLASSES = ("prefill", "splitkv", "combine", "append")  # PA_KC_PREFILL, _SPLITKV, _COMBINE, _APPEND


def kernel_timing(enable: bool) -> None:
    """Start (or stop) bracketing every launch with CUDA events on its stream."""
    load().pa_kernel_timing(1 if enable else 0)


def kernel_times() -> dict:
    """{class: (summed ms, launches)} of the launches timed since the last read; clears them."""
    n = len(KERNEL_CLASSES)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_uint64 * n)()
    rc = load().pa_kernel_times(ms, cnt)
    if rc != 0:
        raise PaError(rc, last_error())
    return {name: (float(ms[i]), int(cnt[i])) for i, name in enumerate(KERNEL_CLASSES)}


def set_wait_limit_ns(ns: int) -> None:
    """Bound, in ns of wall time, on every in-kernel wait (0 restores the 2 s default)."""
    load().pa_set_wait_limit_ns(int(ns))


def set_withhold_loads(enable: bool) -> None:
    """Test hook: while enabled the kernels issue no loads and their waits run out."""
    load().pa_set_withhold_loads(1 if enable else 0)


def last_error() -> str:
    return load().pa_last_error().decode()


def device_status(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the kernels' device error status."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return load().pa_device_status(ctypes.c_void_p(s.cuda_stream))


def check(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_table, max_seqlen_q, max_seqlen_k,
          softmax_scale, window_left, window_right, out, softmax_lse, page_block_size=None,
          num_heads=None, num_heads_k=None, head_dim=None, descriptors=None, alibi_slopes=None) -> int:
    """Host-only validation (no CUDA call); returns the status code.  ``alibi_slopes`` (a
    tensor, or a ready descriptor) selects pa_varlen_check_alibi."""
    lib = load()
    ds = descriptors or [describe(t) for t in (q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_table,
                                                out, softmax_lse)]
    H = num_heads if num_heads is not None else q.shape[1]
    D = head_dim if head_dim is not None else q.shape[-1]
    Hkv = num_heads_k if num_heads_k is not None else k_cache.shape[-2]
    P = page_block_size if page_block_size is not None else (k_cache.shape[1] if block_table is not None else 0)
    scalars = (int(max_seqlen_q), int(max_seqlen_k), int(H), int(Hkv), int(D), int(P), float(softmax_scale),
               int(window_left), int(window_right))
    if alibi_slopes is not None:
        da = alibi_slopes if isinstance(alibi_slopes, PaTensor) else describe(alibi_slopes)
        return lib.pa_varlen_check_alibi(*[_ref(d) for d in ds[:6]], *scalars, _ref(da), _ref(ds[6]),
                                         _ref(ds[7]))
    return lib.pa_varlen_check(*[_ref(d) for d in ds[:6]], *scalars, _ref(ds[6]), _ref(ds[7]))


def varlen_fwd(q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_table=None, max_seqlen_q=None,
               max_seqlen_k=None, softmax_scale=None, window_left=-1, window_right=0, out=None,
               softmax_lse=None, page_block_size=None, num_heads=None, num_heads_k=None, head_dim=None,
               stream=None, alibi_slopes=None) -> Tuple[object, object]:
    """pa_varlen_fwd (pa_varlen_fwd_alibi when ``alibi_slopes`` is given) on torch CUDA
    tensors; returns (out, softmax_lse).

    ``out`` (total_q, H, D) and ``softmax_lse`` (H, total_q) fp32 are allocated with torch
    when not given.  ``max_seqlen_q/k`` must be given (no device read is made to find them).
    ``page_block_size`` defaults to ``k_cache.shape[1]`` in paged mode.  ``alibi_slopes``:
    (num_heads,) fp32 CUDA tensor of per-head linear position-bias slopes.
    """
    import torch
    lib = load()
    if max_seqlen_q is None or max_seqlen_k is None:
        raise ValueError("max_seqlen_q and max_seqlen_k are required")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(q.shape[-1])
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if softmax_lse is None:
        softmax_lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    H = num_heads if num_heads is not None else q.shape[1]
    D = head_dim if head_dim is not None else q.shape[-1]
    Hkv = num_heads_k if num_heads_k is not None else k_cache.shape[-2]
    if page_block_size is None:
        page_block_size = k_cache.shape[1] if block_table is not None and k_cache.dim() == 4 else 0
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    ds = [describe(t) for t in (q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_table, out, softmax_lse)]
    scalars = (int(max_seqlen_q), int(max_seqlen_k), int(H), int(Hkv), int(D), int(page_block_size),
               float(softmax_scale), int(window_left), int(window_right))
    if alibi_slopes is not None:
        rc = lib.pa_varlen_fwd_alibi(*[_ref(d) for d in ds[:6]], *scalars, _ref(describe(alibi_slopes)),
                                     _ref(ds[6]), _ref(ds[7]), ctypes.c_void_p(s.cuda_stream))
    else:
        rc = lib.pa_varlen_fwd(*[_ref(d) for d in ds[:6]], *scalars, _ref(ds[6]), _ref(ds[7]),
                               ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise PaError(rc, lib.pa_last_error().decode())
    return out, softmax_lse


def kv_append(k_new, v_new, cu_seqlens_new, cu_seqlens_k, block_table, k_cache, v_cache, page_block_size=None,
              stream=None) -> None:
    """pa_kv_append on torch CUDA tensors: writes the new tokens of every sequence (the last
    n_b of its sk_b keys) into their pages of ``k_cache`` / ``v_cache``, in place."""
    import torch
    lib = load()
    P = page_block_size if page_block_size is not None else k_cache.shape[1]
    s = stream if stream is not None else torch.cuda.current_stream(k_new.device)
    ds = [describe(t) for t in (k_new, v_new, cu_seqlens_new, cu_seqlens_k, block_table, k_cache, v_cache)]
    rc = lib.pa_kv_append(*[_ref(d) for d in ds], int(P), ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise PaError(rc, lib.pa_last_error().decode())


def kv_append_check(descriptors, page_block_size) -> int:
    """Host-only checks of pa_kv_append on seven descriptors (PaTensor or None)."""
    return load().pa_kv_append_check(*[_ref(d) for d in descriptors], int(page_block_size))


def fwd_padded(q, k, v, softmax_scale=None, window_left=-1, window_right=0, alibi_slopes=None, out=None,
               softmax_lse=None, stream=None) -> Tuple[object, object]:
    """pa_fwd_padded on torch CUDA tensors: q (B, Sq, H, D), k and v (B, Sk, Hkv, D); returns
    (out (B, Sq, H, D), softmax_lse (B, H, Sq) fp32), allocated with torch when not given."""
    import torch
    lib = load()
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(q.shape[-1])
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if softmax_lse is None:
        softmax_lse = torch.empty((q.shape[0], q.shape[2], q.shape[1]), dtype=torch.float32, device=q.device)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    ds = [describe(t) for t in (q, k, v, alibi_slopes, out, softmax_lse)]
    rc = lib.pa_fwd_padded(_ref(ds[0]), _ref(ds[1]), _ref(ds[2]), int(q.shape[2]), int(k.shape[2]), int(q.shape[3]),
                           float(softmax_scale), int(window_left), int(window_right), _ref(ds[3]), _ref(ds[4]),
                           _ref(ds[5]), ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise PaError(rc, lib.pa_last_error().decode())
    return out, softmax_lse


def check_padded(descriptors, num_heads, num_heads_k, head_dim, softmax_scale=0.125, window_left=-1,
                 window_right=0) -> int:
    """Host-only checks of pa_fwd_padded on (q, k, v, alibi_slopes, out, softmax_lse) descriptors."""
    d = [_ref(x) for x in descriptors]
    return load().pa_check_padded(d[0], d[1], d[2], int(num_heads), int(num_heads_k), int(head_dim),
                                  float(softmax_scale), int(window_left), int(window_right), d[3], d[4], d[5])
