"""CUDA path vs the oracle on the same seeded inputs (GPU)."""
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_varlen_flashattention_gb300 import binding, workloads
from tests import _gpu

pytestmark = pytest.mark.gpu


def test_tiny_fp16_all_rows():
    _gpu.check_layout(workloads.tiny_fp16(), gen_device="cpu")


@pytest.mark.parametrize("name", ["decode", "prefill", "mixed", "long", "d512"])
def test_reduced_workloads_all_rows(name):
    _gpu.check_layout(workloads.small(name))


@pytest.mark.parametrize("name,limit", [("decode_bf16", 1024), ("prefill_bf16", 768), ("mixed_bf16", 768),
                                        ("long_bf16", 96), ("long_d512_bf16", 256)])
def test_full_size_sampled_rows(name, limit):
    _gpu.check_layout(workloads.CONFIGS[name](), limit=limit)


def _custom(sq, sk, H=4, Hkv=2, D=64, P=32, dtype="bf16", wl=-1, wr=0, seed=21, **kw):
    return workloads.make_layout("custom", dtype, sq, sk, num_heads=H, num_heads_k=Hkv, head_dim=D,
                                 page_block_size=P, seed=seed, spare=0.2, window_left=wl, window_right=wr, **kw)


def test_empty_sequences():
    _gpu.check_layout(_custom([0, 3, 2, 1], [5, 0, 40, 70]))


def test_more_queries_than_keys_fully_masked_rows():
    _gpu.check_layout(_custom([10, 7], [4, 7]))


@pytest.mark.parametrize("wl,wr", [(-1, -1), (3, 2), (0, 0), (17, -1), (-1, 5)])
def test_windows(wl, wr):
    _gpu.check_layout(_custom([1, 9, 40, 3], [100, 64, 200, 33], wl=wl, wr=wr))


@pytest.mark.parametrize("D", [8, 80, 96, 192, 256, 320, 512])
def test_head_dims(D):
    _gpu.check_layout(_custom([1, 5, 12], [77, 150, 12], H=4, Hkv=1, D=D))


@pytest.mark.parametrize("P", [32, 96, 160, 256])
def test_page_sizes(P):
    _gpu.check_layout(_custom([2, 33, 1], [300, 99, 520], P=P, H=8, Hkv=2, D=128))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_decode_dtypes(dtype):
    lay = workloads.small("decode")
    lay.dtype = dtype
    _gpu.check_layout(lay)


@pytest.mark.parametrize("tiles", ["1", "2", "5"])
def test_forced_split_counts(tiles, monkeypatch):
    monkeypatch.setenv("PA_SPLIT_TILES", tiles)
    _gpu.check_layout(workloads.small("decode"))
    _gpu.check_layout(workloads.small("long"))


def test_non_paged_mode():
    lay = _custom([3, 1, 20], [50, 129, 20], H=8, Hkv=2, D=128)
    lay.paged = False
    _gpu.check_layout(lay)


def test_strided_q_and_out():
    lay = _custom([3, 4], [40, 70], H=4, Hkv=2, D=64)
    inp = workloads.materialize(lay, device="cuda")
    big = torch.zeros((lay.total_q, 8, 72), dtype=inp.q.dtype, device="cuda")
    big[:, 2:6, :64] = inp.q
    q_view = big[:, 2:6, :64]
    out_big = torch.zeros((lay.total_q, 6, 72), dtype=inp.q.dtype, device="cuda")
    out_view = out_big[:, 1:5, :64]
    inp2 = workloads.Inputs(lay, q_view, inp.k_cache, inp.v_cache, inp.cu_seqlens_q, inp.cu_seqlens_k,
                            inp.block_table)
    out, lse = _gpu.run_cuda(inp2, out=out_view)
    assert out.data_ptr() == out_view.data_ptr()
    ref_o, ref_l = _gpu.oracle_for(inp.to("cpu"))
    _gpu.compare(lay, out.contiguous(), lse, ref_o, ref_l)
    assert torch.all(out_big[:, 0] == 0) and torch.all(out_big[:, 5] == 0)


def test_block_permutation_bit_identical():
    lay = workloads.small("mixed")
    inp = workloads.materialize(lay, device="cuda")
    out1, lse1 = _gpu.run_cuda(inp)
    inp2 = workloads.with_block_permutation(inp, seed=5)
    out2, lse2 = _gpu.run_cuda(inp2)
    assert torch.equal(out1, out2)
    assert torch.equal(lse1, lse2)


def test_bad_block_id_is_reported_not_faulted():
    lay = _custom([1, 1], [100, 64], H=4, Hkv=2, D=64)
    inp = workloads.materialize(lay, device="cuda")
    inp.block_table[0, 1] = lay.num_blocks + 1000
    inp.block_table[1, 0] = -7
    binding.varlen_fwd(inp.q, inp.k_cache, inp.v_cache, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.block_table,
                       max_seqlen_q=1, max_seqlen_k=100)
    st = binding.device_status()
    assert binding.STATUS[st] == "PA_ERR_DEVICE_BOUNDS", binding.last_error()
    assert binding.device_status() == 0  # cleared


def test_sequence_longer_than_max_seqlen_k_is_reported():
    lay = _custom([1, 1], [300, 64], H=4, Hkv=2, D=64)
    inp = workloads.materialize(lay, device="cuda")
    binding.varlen_fwd(inp.q, inp.k_cache, inp.v_cache, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.block_table,
                       max_seqlen_q=1, max_seqlen_k=64)
    assert binding.STATUS[binding.device_status()] == "PA_ERR_DEVICE_BOUNDS"


def test_host_memory_is_rejected():
    lay = workloads.tiny_fp16()
    inp = workloads.materialize(lay, device="cuda")
    with pytest.raises(binding.PaError) as ei:
        binding.varlen_fwd(inp.q, inp.k_cache, inp.v_cache, inp.cu_seqlens_q, inp.cu_seqlens_k,
                           inp.block_table.cpu(), max_seqlen_q=5, max_seqlen_k=70)
    assert ei.value.name == "PA_ERR_NOT_DEVICE" and "block_table must be a cuda tensor" in str(ei.value)


def test_zero_queries_is_a_no_op():
    lay = _custom([0, 0], [5, 7])
    inp = workloads.materialize(lay, device="cuda")
    out, lse = _gpu.run_cuda(inp)
    assert out.numel() == 0 and lse.numel() == 0


def test_prefill_fp16():
    lay = workloads.small("prefill")
    lay.dtype = "f16"
    _gpu.check_layout(lay)


@pytest.mark.parametrize("H,Hkv", [(6, 2), (12, 1), (8, 8)])
def test_group_sizes(H, Hkv):
    """G = 3 and 12 do not divide the 128-row tensor-core tile (42 and 10 whole queries a
    tile, 2 and 8 padding rows); G = 1 does."""
    _gpu.check_layout(_custom([70, 1, 150], [70, 300, 200], H=H, Hkv=Hkv, D=64))


@pytest.mark.parametrize("G", [3, 5, 6, 7, 12, 24])
@pytest.mark.parametrize("D", [64, 128])
def test_prefill_group_sizes_not_dividing_the_tile(G, D):
    """Long query rows on the tensor-core prefill kernel with G not dividing 128: several
    tile pairs per sequence, a ragged last pair, chunked prefill (sk > sq) and a window."""
    lay = _custom([300, 77, 1, 129], [300, 500, 40, 200], H=2 * G, Hkv=2, D=D, seed=70 + G)
    _gpu.check_layout(lay, limit=4096)
    lay = _custom([260, 33], [900, 33], H=G, Hkv=1, D=D, wl=100, wr=0, seed=80 + G, dtype="f16")
    _gpu.check_layout(lay, limit=4096)


def test_prefill_group_not_dividing_with_bias():
    lay = _custom([200, 90], [500, 90], H=6, Hkv=2, D=128, seed=91)
    _gpu.check_layout(lay, alibi=_gpu.alibi_slopes(6), limit=4096)


def test_long_prefill_spans_many_tiles_and_pages():
    _gpu.check_layout(_custom([1000, 517], [1000, 900], H=4, Hkv=1, D=128, P=32), limit=4096)


def test_non_causal_prefill_with_sq_below_sk():
    _gpu.check_layout(_custom([200, 64], [1000, 64], H=8, Hkv=2, D=128, wl=-1, wr=-1))


def test_kernel_timing_counts_each_class():
    """Per-kernel timing sees one prefill launch per call for a prefill-only batch and the
    split-KV pass (plus its combine when split) for a decode batch; times are positive."""
    for name, cls in (("prefill", "prefill"), ("decode", "splitkv")):
        lay = workloads.small(name)
        lay.nan_fill = False
        g = workloads.materialize(lay, device="cuda")
        out = torch.empty_like(g.q)
        lse = torch.empty((lay.num_heads, lay.total_q), dtype=torch.float32, device="cuda")
        binding.kernel_times()
        binding.kernel_timing(True)
        try:
            for _ in range(3):
                binding.varlen_fwd(g.q, g.k_cache, g.v_cache, g.cu_seqlens_q, g.cu_seqlens_k, g.block_table,
                                   max_seqlen_q=lay.max_seqlen_q, max_seqlen_k=lay.max_seqlen_k,
                                   softmax_scale=lay.softmax_scale, window_left=lay.window_left,
                                   window_right=lay.window_right, out=out, softmax_lse=lse)
            torch.cuda.synchronize()
        finally:
            binding.kernel_timing(False)
        t = binding.kernel_times()
        assert t[cls][1] >= 3 and t[cls][0] > 0.0, (name, t)
        assert binding.kernel_times() == {k: (0.0, 0) for k in binding.KERNEL_CLASSES}


# ---- linear position bias (alibi_slopes) ----------------------------------------------------

@pytest.mark.parametrize("name", ["decode", "prefill", "mixed", "long", "d512"])
def test_alibi_reduced_workloads_all_rows(name):
    lay = workloads.small(name)
    _gpu.check_layout(lay, alibi=_gpu.alibi_slopes(lay.num_heads))


@pytest.mark.parametrize("D", [64, 128, 256])
def test_alibi_head_dims_random_slopes(D):
    """Random slopes under GQA; prefill rows (tensor-core kernel up to D = 128), long-query
    rows past it and decode rows in one batch."""
    _gpu.check_layout(_custom([150, 1, 40, 1], [150, 300, 700, 64], H=8, Hkv=2, D=D),
                      alibi=_gpu.alibi_slopes(8, "random", seed=D))


def test_alibi_windows_and_fp16():
    lay = _custom([200, 33, 1], [260, 33, 500], H=4, Hkv=1, D=128, dtype="f16", wl=50, wr=7)
    _gpu.check_layout(lay, alibi=_gpu.alibi_slopes(4))


@pytest.mark.parametrize("tiles", [1, 3])
def test_alibi_forced_splits(tiles, monkeypatch):
    """Split-KV partials and the combine carry the bias (a split count forced small)."""
    monkeypatch.setenv("PA_SPLIT_TILES", str(tiles))
    lay = workloads.small("decode")
    _gpu.check_layout(lay, alibi=_gpu.alibi_slopes(lay.num_heads, "random", seed=7))


def test_alibi_zero_slopes_match_no_bias():
    lay = workloads.small("mixed")
    _gpu.check_layout(lay, alibi=np.zeros(lay.num_heads, dtype=np.float32))


@pytest.mark.parametrize("name,limit", [("decode_bf16", 1024), ("prefill_bf16", 768)])
def test_alibi_full_size_sampled_rows(name, limit):
    lay = workloads.CONFIGS[name]()
    _gpu.check_layout(lay, limit=limit, alibi=_gpu.alibi_slopes(lay.num_heads))


def test_alibi_slopes_on_host_are_rejected():
    lay = workloads.small("decode")
    lay.nan_fill = False
    g = workloads.materialize(lay, device="cuda")
    with pytest.raises(binding.PaError) as ei:
        binding.varlen_fwd(g.q, g.k_cache, g.v_cache, g.cu_seqlens_q, g.cu_seqlens_k, g.block_table,
                           max_seqlen_q=lay.max_seqlen_q, max_seqlen_k=lay.max_seqlen_k,
                           alibi_slopes=torch.zeros(lay.num_heads, dtype=torch.float32))
    assert ei.value.name == "PA_ERR_NOT_DEVICE"


# ---- padded (non-varlen) batches ------------------------------------------------------------

def _padded_check(B, Sq, Sk, H=8, Hkv=2, D=128, dtype=torch.bfloat16, wl=-1, wr=0, alibi=None, seed=31):
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn((B, Sq, H, D), generator=g, device="cuda").to(dtype)
    k = torch.randn((B, Sk, Hkv, D), generator=g, device="cuda").to(dtype)
    v = torch.randn((B, Sk, Hkv, D), generator=g, device="cuda").to(dtype)
    sl = None if alibi is None else torch.from_numpy(alibi).cuda()
    out, lse = binding.fwd_padded(q, k, v, 1.0 / D ** 0.5, wl, wr, alibi_slopes=sl)
    torch.cuda.synchronize()
    assert binding.device_status() == 0, binding.last_error()
    name = "bf16" if dtype == torch.bfloat16 else "f16"
    ref_o, ref_l = oracle.attention_padded(name, q.cpu(), k.cpu(), v.cpu(), 1.0 / D ** 0.5, wl, wr,
                                           alibi_slopes=None if alibi is None else alibi.astype(np.float64))
    lay = workloads.Layout.__new__(workloads.Layout)
    lay.name, lay.num_heads, lay.head_dim, lay.dtype = "padded", H, D, name
    _gpu.compare(lay, out.reshape(B * Sq, H, D), lse.permute(1, 0, 2).reshape(H, B * Sq),
                 ref_o.reshape(B * Sq * H, D), ref_l.transpose(0, 2, 1).reshape(-1))


@pytest.mark.parametrize("B,Sq,Sk", [(3, 100, 100), (4, 1, 300), (2, 5, 40), (2, 300, 700), (1, 1, 1)])
def test_padded_causal(B, Sq, Sk):
    _padded_check(B, Sq, Sk)


def test_padded_full_window_fp16_alibi():
    _padded_check(2, 150, 150, H=4, Hkv=4, D=64, dtype=torch.float16, wl=-1, wr=-1,
                  alibi=_gpu.alibi_slopes(4))


@pytest.mark.parametrize("D", [256, 512])
def test_padded_large_head_dims(D):
    _padded_check(2, 40, 90, H=4, Hkv=1, D=D)


def test_padded_noncontiguous_lse_and_out():
    """out and lse as views with strides of larger tensors (batch strides honoured)."""
    B, S, H, Hkv, D = 2, 64, 4, 2, 64
    q = torch.randn((B, S, H, D), device="cuda").bfloat16()
    k = torch.randn((B, S, Hkv, D), device="cuda").bfloat16()
    v = torch.randn((B, S, Hkv, D), device="cuda").bfloat16()
    lse_big = torch.full((B, H + 2, S + 16), 7.0, device="cuda")
    lse = lse_big[:, 1:H + 1, 8:S + 8]
    out, _ = binding.fwd_padded(q, k, v, 0.125, -1, 0, softmax_lse=lse)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attention_padded("bf16", q.cpu(), k.cpu(), v.cpu(), 0.125, -1, 0)
    assert np.allclose(lse.cpu().numpy(), ref_l, atol=1e-3)
    assert torch.all(lse_big[:, 0] == 7.0) and torch.all(lse_big[:, :, :8] == 7.0)
    assert np.allclose(out.float().cpu().numpy(), ref_o, atol=1.6e-2, rtol=2e-2)


def test_padded_full_size_sampled():
    """8 x 2048 causal, H=32, Hkv=8, D=128 (the tensor-core path), sampled rows."""
    B, S, H, Hkv, D = 8, 2048, 32, 8, 128
    g = torch.Generator(device="cuda").manual_seed(41)
    q = torch.randn((B, S, H, D), generator=g, device="cuda").bfloat16()
    k = torch.randn((B, S, Hkv, D), generator=g, device="cuda").bfloat16()
    v = torch.randn((B, S, Hkv, D), generator=g, device="cuda").bfloat16()
    out, lse = binding.fwd_padded(q, k, v, 1.0 / D ** 0.5, -1, 0)
    torch.cuda.synchronize()
    rows = np.random.default_rng(0).choice(B * S * H, size=512, replace=False)
    rows = np.unique(np.concatenate([rows, [0, B * S * H - 1]]))
    cu = np.arange(B + 1, dtype=np.int32) * S
    ref_o, ref_l = oracle.attention("bf16", q.cpu().reshape(B * S, H, D), k.cpu().reshape(B * S, Hkv, D),
                                    v.cpu().reshape(B * S, Hkv, D), cu, cu, None, 1.0 / D ** 0.5, -1, 0, rows=rows)
    lay = workloads.Layout.__new__(workloads.Layout)
    lay.name, lay.num_heads, lay.head_dim, lay.dtype = "padded_full", H, D, "bf16"
    _gpu.compare(lay, out.reshape(B * S, H, D), lse.permute(1, 0, 2).reshape(H, B * S), ref_o, ref_l, rows)


def test_cuda_graph_capture_and_replay():
    """A serving step (KV append, then the forward call with a mixed batch) captured in a
    CUDA graph after one warm-up call on the capture stream (which sizes the library's
    per-stream workspace) replays to the
    same result as the direct calls, and a new q written into the captured input buffer is
    picked up by the replay."""
    lay = workloads.small("mixed")
    lay.nan_fill = False
    g = workloads.materialize(lay, device="cuda")
    out = torch.empty_like(g.q)
    lse = torch.empty((lay.num_heads, lay.total_q), dtype=torch.float32, device="cuda")
    kw = dict(max_seqlen_q=lay.max_seqlen_q, max_seqlen_k=lay.max_seqlen_k, softmax_scale=lay.softmax_scale,
              window_left=lay.window_left, window_right=lay.window_right, out=out, softmax_lse=lse)
    kn = torch.randn((lay.total_q, lay.num_heads_k, lay.head_dim), device="cuda").to(g.k_cache.dtype)
    vn = torch.randn_like(kn)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        binding.kv_append(kn, vn, g.cu_seqlens_q, g.cu_seqlens_k, g.block_table, g.k_cache, g.v_cache, stream=s)
        binding.varlen_fwd(g.q, g.k_cache, g.v_cache, g.cu_seqlens_q, g.cu_seqlens_k, g.block_table, stream=s, **kw)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref_out, ref_lse = out.clone(), lse.clone()
    graph = torch.cuda.CUDAGraph()
    # the split-KV workspace is per (device, stream): capture on the stream that was warmed up
    with torch.cuda.graph(graph, stream=s):
        stream = torch.cuda.current_stream()
        binding.kv_append(kn, vn, g.cu_seqlens_q, g.cu_seqlens_k, g.block_table, g.k_cache, g.v_cache,
                          stream=stream)
        binding.varlen_fwd(g.q, g.k_cache, g.v_cache, g.cu_seqlens_q, g.cu_seqlens_k, g.block_table,
                           stream=stream, **kw)
    out.zero_()
    lse.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert binding.device_status() == 0, binding.last_error()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    # new queries through the same captured buffers
    g.q.copy_(torch.randn_like(g.q.float()).to(g.q.dtype))
    graph.replay()
    torch.cuda.synchronize()
    inp_cpu = workloads.Inputs(lay, g.q.cpu(), g.k_cache.cpu(), g.v_cache.cpu(), g.cu_seqlens_q.cpu(),
                               g.cu_seqlens_k.cpu(), g.block_table.cpu())
    ref_o, ref_l = _gpu.oracle_for(inp_cpu)
    _gpu.compare(lay, out, lse, ref_o, ref_l)
