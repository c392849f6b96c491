"""pa_kv_append on the GPU against the oracle's scatter: the whole caches must match byte
for byte (GPU)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_varlen_flashattention_gb300 import binding, workloads
from tests import _gpu

pytestmark = pytest.mark.gpu


def _cu(lengths):
    c = np.zeros(len(lengths) + 1, dtype=np.int32)
    c[1:] = np.cumsum(lengths)
    return c


def _pool(sk, P, Hkv, D, dtype, seed, spare=3):
    """Random caches (NaN-free) and a shuffled block table for sequences of sk keys."""
    g = torch.Generator().manual_seed(seed)
    pages = [(s + P - 1) // P for s in sk]
    nb = sum(pages) + spare
    perm = torch.randperm(nb, generator=g).numpy()
    bt = np.full((len(sk), max(max(pages), 1) + 1), -1, dtype=np.int32)
    cur = 0
    for b, p in enumerate(pages):
        bt[b, :p] = perm[cur:cur + p]
        cur += p
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    kc = torch.randn((nb, P, Hkv, D), generator=g).to(tdt)
    vc = torch.randn((nb, P, Hkv, D), generator=g).to(tdt)
    return kc, vc, bt


def run_and_compare(sk, n, P=32, Hkv=2, D=64, dtype="bf16", seed=0, new_token_stride=None):
    kc, vc, bt = _pool(sk, P, Hkv, D, dtype, seed)
    g = torch.Generator().manual_seed(seed + 1)
    tdt = kc.dtype
    total = int(sum(n))
    if new_token_stride:  # K and V rows inside a wider per-token buffer (e.g. a fused projection)
        buf = torch.randn((total, new_token_stride // (Hkv * D), Hkv, D), generator=g).to(tdt)
        kn, vn = buf[:, 0], buf[:, 1]
    else:
        kn = torch.randn((total, Hkv, D), generator=g).to(tdt)
        vn = torch.randn((total, Hkv, D), generator=g).to(tdt)
    kc_ref, vc_ref = kc.clone(), vc.clone()
    oracle.kv_append(kn.view(torch.int16).numpy(), vn.view(torch.int16).numpy(), _cu(n), _cu(sk), bt,
                     kc_ref.view(torch.int16).numpy(), vc_ref.view(torch.int16).numpy())
    dev = "cuda"
    kc_d, vc_d = kc.to(dev), vc.to(dev)
    binding.kv_append(kn.to(dev) if not new_token_stride else buf.to(dev)[:, 0],
                      vn.to(dev) if not new_token_stride else buf.to(dev)[:, 1],
                      torch.from_numpy(_cu(n)).to(dev), torch.from_numpy(_cu(sk)).to(dev),
                      torch.from_numpy(bt).to(dev), kc_d, vc_d)
    torch.cuda.synchronize()
    assert binding.device_status() == 0, binding.last_error()
    assert torch.equal(kc_d.cpu().view(torch.int16), kc_ref.view(torch.int16))
    assert torch.equal(vc_d.cpu().view(torch.int16), vc_ref.view(torch.int16))
    return kc_d, vc_d, bt


def test_append_mixed_batch():
    """Fresh prompts, decode steps, chunks, and sequences without new tokens in one call."""
    run_and_compare([70, 33, 1, 96, 40, 5, 300], [7, 0, 1, 96, 40, 2, 129])


@pytest.mark.parametrize("P,D,Hkv", [(32, 128, 8), (64, 64, 1), (256, 256, 2), (32, 512, 1)])
def test_append_page_and_head_sizes(P, D, Hkv):
    run_and_compare([513, 1, 257, 1000], [513, 1, 100, 31], P=P, D=D, Hkv=Hkv, seed=P + D)


def test_append_fp16_and_strided_new_tokens():
    run_and_compare([90, 17], [30, 17], dtype="f16", D=128, Hkv=2, new_token_stride=2 * 2 * 128, seed=5)


def test_append_empty_and_all_zero_counts():
    run_and_compare([5, 9], [0, 0])


def test_append_bad_block_is_reported_others_written():
    sk, n = [40, 40], [40, 40]
    kc, vc, bt = _pool(sk, 32, 2, 64, "bf16", 9)
    bt[0, 1] = kc.shape[0] + 5  # second page of sequence 0 points past the pool
    kn = torch.randn((80, 2, 64)).bfloat16()
    vn = torch.randn((80, 2, 64)).bfloat16()
    kc_d, vc_d = kc.cuda(), vc.cuda()
    binding.kv_append(kn.cuda(), vn.cuda(), torch.from_numpy(_cu(n)).cuda(), torch.from_numpy(_cu(sk)).cuda(),
                      torch.from_numpy(bt).cuda(), kc_d, vc_d)
    torch.cuda.synchronize()
    assert binding.STATUS[binding.device_status()] == "PA_ERR_DEVICE_BOUNDS"
    assert binding.device_status() == 0  # the word was cleared
    # sequence 1 went through
    pos = np.arange(40)
    got = kc_d.cpu()[torch.from_numpy(bt[1, pos // 32]).long(), torch.from_numpy(pos % 32).long()]
    assert torch.equal(got.view(torch.int16), kn[40:].view(torch.int16))


def test_append_more_new_tokens_than_keys_is_reported():
    sk, n = [3], [5]
    kc, vc, bt = _pool(sk, 32, 1, 64, "bf16", 11)
    kc_d = kc.cuda()
    binding.kv_append(torch.zeros((5, 1, 64), dtype=torch.bfloat16, device="cuda"),
                      torch.zeros((5, 1, 64), dtype=torch.bfloat16, device="cuda"),
                      torch.from_numpy(_cu(n)).cuda(), torch.from_numpy(_cu(sk)).cuda(),
                      torch.from_numpy(bt).cuda(), kc_d, vc.cuda())
    torch.cuda.synchronize()
    assert binding.STATUS[binding.device_status()] == "PA_ERR_DEVICE_BOUNDS"
    assert torch.equal(kc_d.cpu().view(torch.int16), kc.view(torch.int16))


def test_append_full_prefill_prompt_then_attention():
    """The causal-prefill workload's prompts appended into an empty pool, then attention over
    the result equals the oracle on the same cache (the serving step: append, then attend)."""
    lay = workloads.small("prefill")
    lay.nan_fill = False
    g = workloads.materialize(lay, device="cuda")
    k_pool = torch.zeros_like(g.k_cache)
    v_pool = torch.zeros_like(g.v_cache)
    # the prompt's K/V rows, gathered from the materialised cache through its block table
    cq, ck = lay.cu_seqlens()
    bt = g.block_table.cpu().numpy()
    P = lay.page_block_size
    kn = torch.cat([g.k_cache[torch.from_numpy(bt[b, np.arange(ck[b + 1] - ck[b]) // P]).long().cuda(),
                              torch.from_numpy(np.arange(ck[b + 1] - ck[b]) % P).long().cuda()]
                    for b in range(lay.batch)])
    vn = torch.cat([g.v_cache[torch.from_numpy(bt[b, np.arange(ck[b + 1] - ck[b]) // P]).long().cuda(),
                              torch.from_numpy(np.arange(ck[b + 1] - ck[b]) % P).long().cuda()]
                    for b in range(lay.batch)])
    binding.kv_append(kn, vn, g.cu_seqlens_k, g.cu_seqlens_k, g.block_table, k_pool, v_pool)
    inp = workloads.Inputs(lay, g.q, k_pool, v_pool, g.cu_seqlens_q, g.cu_seqlens_k, g.block_table)
    out, lse = _gpu.run_cuda(inp)
    ref_o, ref_l = _gpu.oracle_for(inp.to("cpu"))
    _gpu.compare(lay, out, lse, ref_o, ref_l)


@pytest.mark.parametrize("name", ["decode_bf16", "prefill_bf16"])
def test_append_full_size_bit_exact(name):
    """Every token of the workload appended (a whole prompt per sequence) into a shuffled
    pool: byte-identical to the oracle's scatter."""
    lay = workloads.CONFIGS[name]()
    sk = list(lay.seqlens_k)
    n = list(lay.seqlens_k) if name == "prefill_bf16" else [1] * lay.batch
    run_and_compare(sk, n, P=lay.page_block_size, Hkv=lay.num_heads_k, D=lay.head_dim, seed=3)
