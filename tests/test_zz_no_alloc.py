"""pa_varlen_fwd_noalloc, the entry point for callers that cannot allocate device memory
(runtimes that own all device memory through their own arena, latency-critical loops where
an allocation could stall, plug-in hosts that only lend their buffers).  It is called
through the C ABI and must give exactly the results of pa_varlen_fwd under the same split
plan, call after call, while keeping its split-KV partial results (and the decode launch
order of large batches) in the library's fixed scratch array instead of allocating.

This file is collected last so that a failure here never hides the other tests."""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_varlen_flashattention_gb300 import binding, workloads
from tests import _gpu
from tests.test_large_batch_gpu import skewed_layout

pytestmark = pytest.mark.gpu


def _noalloc(inp, out, lse, stream=None):
    lib = binding.load()
    fn = lib.pa_varlen_fwd_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = binding._FWD_ARGS + [ctypes.c_void_p]
    lay = inp.layout
    ds = [binding.describe(t) for t in (inp.q, inp.k_cache, inp.v_cache, inp.cu_seqlens_q, inp.cu_seqlens_k,
                                         inp.block_table, out, lse)]
    ref = lambda d: None if d is None else ctypes.byref(d)  # noqa: E731
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = fn(ref(ds[0]), ref(ds[1]), ref(ds[2]), ref(ds[3]), ref(ds[4]), ref(ds[5]), lay.max_seqlen_q,
            lay.max_seqlen_k, lay.num_heads, lay.num_heads_k, lay.head_dim, lay.page_block_size,
            lay.softmax_scale, lay.window_left, lay.window_right, ref(ds[6]), ref(ds[7]),
            ctypes.c_void_p(s.cuda_stream))
    assert rc == 0, binding.last_error()


def _fresh_outputs(lay):
    out = torch.full((lay.total_q, lay.num_heads, lay.head_dim), float("nan"),
                     dtype=workloads._torch_dtype(lay.dtype), device="cuda")
    lse = torch.full((lay.num_heads, lay.total_q), float("nan"), dtype=torch.float32, device="cuda")
    return out, lse


def _layout(name):
    if name == "large":  # 300 sequences: the work list, then the partials
        # (max_seqlen_k 500: nine one-tile splits of ~2.3 MB each fit the 32 MiB array)
        return skewed_layout(300, seed=41, long_k=500, short_hi=400)
    if name == "wide":  # head_dim 256 prefill rows (their kernel) beside decode rows (split)
        return workloads.make_layout("noalloc_wide", "bf16", [150, 1, 4, 1], [300, 700, 200, 90], num_heads=8,
                                     num_heads_k=2, head_dim=256, page_block_size=64, seed=43, spare=0.1)
    return workloads.small(name)


@pytest.mark.parametrize("name", ["decode", "long", "large", "wide"])
def test_noalloc_equals_pa_varlen_fwd_and_oracle(name, monkeypatch):
    # one 64-key tile per split forces several splits, so the scratch array is used
    monkeypatch.setenv("PA_SPLIT_TILES", "1")
    lay = _layout(name)
    inp = workloads.materialize(lay, device="cuda")
    other = workloads.materialize(lay, device="cuda", seed=lay.seed + 101)  # same shapes, other values
    want_o, want_l = _gpu.run_cuda(inp)  # pa_varlen_fwd under the same split plan
    rows = _gpu.sample_rows(lay, 2048)
    ref_o, ref_l = _gpu.oracle_for(inp.to("cpu"), rows)
    # the scratch first holds another call's partial results; a stale read would show
    o_other, l_other = _fresh_outputs(lay)
    _noalloc(other, o_other, l_other)
    for _ in range(2):
        out, lse = _fresh_outputs(lay)
        _noalloc(inp, out, lse)
        torch.cuda.synchronize()
        assert binding.device_status() == 0, binding.last_error()
        assert torch.equal(out, want_o), "output differs from pa_varlen_fwd's"
        assert torch.equal(lse, want_l), "lse differs from pa_varlen_fwd's"
        _gpu.compare(lay, out, lse, ref_o, ref_l, rows)


def test_noalloc_allocates_nothing(monkeypatch):
    """On a stream the library has never seen, pa_varlen_fwd grows a workspace for it
    (device memory goes down); pa_varlen_fwd_noalloc leaves the free device memory as it was."""
    monkeypatch.setenv("PA_SPLIT_TILES", "1")
    lay = workloads.small("long")  # ~6 MB of split partials
    inp = workloads.materialize(lay, device="cuda")
    out, lse = _fresh_outputs(lay)
    _noalloc(inp, out, lse)  # the first call on the device looks the array's address up
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        _noalloc(inp, out, lse, stream=s1)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
    with torch.cuda.stream(s2):  # the test can see an allocation: pa_varlen_fwd's workspace
        binding.varlen_fwd(inp.q, inp.k_cache, inp.v_cache, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.block_table,
                           max_seqlen_q=lay.max_seqlen_q, max_seqlen_k=lay.max_seqlen_k,
                           softmax_scale=lay.softmax_scale, window_left=lay.window_left,
                           window_right=lay.window_right, out=out, softmax_lse=lse)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] < free1
