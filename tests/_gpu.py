"""Helpers shared by the GPU tests: run the CUDA path through the C-ABI binding and
compare it with the oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_varlen_flashattention_gb300 import binding, workloads

TOL = {"f16": (2e-3, 1e-2), "bf16": (1.6e-2, 2e-2)}  # |out - ref| <= atol + rtol * |ref|
LSE_TOL = 1e-3


def run_cuda(inp: workloads.Inputs, **overrides):
    lay = inp.layout
    kw = dict(max_seqlen_q=lay.max_seqlen_q, max_seqlen_k=lay.max_seqlen_k, softmax_scale=lay.softmax_scale,
              window_left=lay.window_left, window_right=lay.window_right)
    kw.update(overrides)
    out, lse = binding.varlen_fwd(inp.q, inp.k_cache, inp.v_cache, inp.cu_seqlens_q, inp.cu_seqlens_k,
                                  inp.block_table, **kw)
    torch.cuda.synchronize()
    st = binding.device_status()
    assert st == 0, f"device status {st}: {binding.last_error()}"
    return out, lse


def sample_rows(lay, limit, seed=0):
    """All (token, head) rows when there are at most ``limit``; else a seeded sample that
    always includes the first and last query of every sequence (first and last head)."""
    n = lay.total_q * lay.num_heads
    if n <= limit:
        return None
    cq, _ = lay.cu_seqlens()
    must = []
    for b in range(lay.batch):
        if cq[b + 1] > cq[b]:
            for t in (cq[b], cq[b + 1] - 1):
                must += [t * lay.num_heads, t * lay.num_heads + lay.num_heads - 1]
    rng = np.random.default_rng(seed)
    extra = rng.choice(n, size=max(0, limit - len(must)), replace=False)
    return np.unique(np.concatenate([np.array(must, dtype=np.int64), extra.astype(np.int64)]))


def oracle_for(inp_cpu: workloads.Inputs, rows=None, alibi_slopes=None):
    lay = inp_cpu.layout
    bt = inp_cpu.block_table.numpy() if inp_cpu.block_table is not None else None
    return oracle.attention(lay.dtype, inp_cpu.q, inp_cpu.k_cache, inp_cpu.v_cache,
                            inp_cpu.cu_seqlens_q.numpy(), inp_cpu.cu_seqlens_k.numpy(), bt, lay.softmax_scale,
                            lay.window_left, lay.window_right, rows=rows, alibi_slopes=alibi_slopes)


def alibi_slopes(num_heads, kind="geometric", seed=0):
    """Slopes for the linear position bias: the usual geometric sequence 2^(-8 (h + 1) / H),
    or seeded uniform values in [0, 0.5) ("random"), as float32."""
    if kind == "geometric":
        return np.array([2.0 ** (-8.0 * (h + 1) / num_heads) for h in range(num_heads)], dtype=np.float32)
    return (np.random.default_rng(seed).random(num_heads) * 0.5).astype(np.float32)


def compare(lay, out, lse, ref_o, ref_l, rows=None):
    """Element-wise comparison at the stated tolerances; returns (max out err, max lse err)."""
    H, D = lay.num_heads, lay.head_dim
    got_o = out.float().cpu().numpy().reshape(-1, D).astype(np.float64)   # row = t * H + h
    got_l = lse.t().contiguous().cpu().numpy().reshape(-1).astype(np.float64)
    if rows is not None:
        got_o, got_l = got_o[rows], got_l[rows]
    atol, rtol = TOL[lay.dtype]
    assert np.all(np.isfinite(got_o)), "non-finite output"
    err = np.abs(got_o - ref_o)
    bad = err > atol + rtol * np.abs(ref_o)
    assert not bad.any(), (
        f"{lay.name}: {bad.sum()} of {bad.size} outputs out of tolerance; max err {err.max():.3e}; "
        f"first bad row {np.argwhere(bad)[0]}")
    ninf_ref, ninf_got = np.isneginf(ref_l), np.isneginf(got_l)
    assert np.array_equal(ninf_ref, ninf_got), f"{lay.name}: -inf lse rows differ"
    fin = ~ninf_ref
    lerr = np.abs(got_l[fin] - ref_l[fin]) if fin.any() else np.zeros(1)
    assert np.all(lerr <= LSE_TOL), f"{lay.name}: lse max err {lerr.max():.3e}"
    return float(err.max()), float(lerr.max())


def check_layout(lay, limit=1 << 30, gen_device="cuda", seed_rows=0, alibi=None, **overrides):
    """Materialise ``lay``, run the CUDA path, and check (sampled) rows against the oracle.
    ``alibi``: optional float32 numpy slopes (one per query head) given to both sides."""
    inp_gpu = workloads.materialize(lay, device=gen_device).to("cuda")
    if alibi is not None:
        overrides["alibi_slopes"] = torch.from_numpy(np.asarray(alibi, dtype=np.float32)).to("cuda")
    out, lse = run_cuda(inp_gpu, **overrides)
    inp_cpu = inp_gpu.to("cpu")
    rows = sample_rows(lay, limit, seed_rows)
    ref_o, ref_l = oracle_for(inp_cpu, rows, alibi_slopes=None if alibi is None else np.asarray(alibi, np.float64))
    return compare(lay, out, lse, ref_o, ref_l, rows)
