"""pa_varlen_fwd_noalloc, the entry point for callers that cannot allocate device memory
(runtimes that own all device memory through their own arena, latency-critical loops where
an allocation could stall, plug-in hosts that only lend their buffers).  It is called
through the C ABI and must give the same results as pa_varlen_fwd, call after call, while
using the library's fixed scratch array for the split-KV partial results.

This file is collected last so that a failure here never hides the other tests."""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_varlen_flashattention_gb300 import binding, workloads
from tests import _gpu

pytestmark = pytest.mark.gpu


def _noalloc(inp, out, lse):
    lib = binding.load()
    fn = lib.pa_varlen_fwd_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = binding._FWD_ARGS + [ctypes.c_void_p]
    lay = inp.layout
    ds = [binding.describe(t) for t in (inp.q, inp.k_cache, inp.v_cache, inp.cu_seqlens_q, inp.cu_seqlens_k,
                                         inp.block_table, out, lse)]
    ref = lambda d: None if d is None else ctypes.byref(d)  # noqa: E731
    rc = fn(ref(ds[0]), ref(ds[1]), ref(ds[2]), ref(ds[3]), ref(ds[4]), ref(ds[5]), lay.max_seqlen_q,
            lay.max_seqlen_k, lay.num_heads, lay.num_heads_k, lay.head_dim, lay.page_block_size,
            lay.softmax_scale, lay.window_left, lay.window_right, ref(ds[6]), ref(ds[7]),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, binding.last_error()
    torch.cuda.synchronize()
    assert binding.device_status() == 0, binding.last_error()


@pytest.mark.parametrize("name", ["decode", "long"])
def test_noalloc_matches_pa_varlen_fwd_twice(name, monkeypatch):
    # one 64-key tile per split forces several splits, so the scratch array is used
    monkeypatch.setenv("PA_SPLIT_TILES", "1")
    lay = workloads.small(name)
    inp = workloads.materialize(lay, device="cuda")
    want_o, want_l = _gpu.run_cuda(inp)
    atol, rtol = _gpu.TOL[lay.dtype]
    for _ in range(2):  # the second call reuses scratch that still holds the first call's data
        out = torch.full_like(inp.q, float("nan"))
        lse = torch.full((lay.num_heads, lay.total_q), float("nan"), dtype=torch.float32, device="cuda")
        _noalloc(inp, out, lse)
        o, w = out.float().cpu().numpy(), want_o.float().cpu().numpy()
        assert np.all(np.abs(o - w) <= atol + rtol * np.abs(w))
        l, wl = lse.cpu().numpy(), want_l.cpu().numpy()
        assert np.array_equal(np.isneginf(l), np.isneginf(wl))
        fin = np.isfinite(wl)
        assert np.all(np.abs(l[fin] - wl[fin]) <= _gpu.LSE_TOL)
