"""Host-side pieces of bench.py that decide how a workload is timed and what its work is:
the L2-flush decision follows the size of the K/V pools that a call re-reads, and the
algorithmic byte and FLOP counts follow the mask (checked by brute force on a small
layout)."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_kv_varlen_flashattention_gb300 import workloads  # noqa: E402


def test_pool_bytes_is_the_materialised_kv_pools():
    lay = workloads.make_layout("t", "bf16", [3, 5], [40, 70], num_heads=4, num_heads_k=2, head_dim=64,
                                page_block_size=32, seed=1, extra_blocks=3)
    inp = workloads.materialize(lay, device="cpu")
    assert bench.pool_bytes(lay) == inp.k_cache.numel() * 2 + inp.v_cache.numel() * 2


def test_flush_decision_and_labels():
    small, large = 2 * bench.L2_BYTES, 2 * bench.L2_BYTES + 1
    assert "flushed" in bench.l2_label(small) and "no flush" in bench.l2_label(large)
    assert not bench.L2Flush(large)  # large pools: no buffer, calls timed back to back
    for name, flushed in [("decode_bf16", False), ("long_bf16", False), ("mixed_bf16", False),
                          ("prefill_bf16", True), ("long_d512_bf16", True), ("skewed_decode_bf16", False),
                          ("prefill_d256_bf16", True)]:
        lay = workloads.CONFIGS[name]()
        assert (bench.pool_bytes(lay) <= 2 * bench.L2_BYTES) == flushed, name


def test_algorithmic_counts_match_brute_force():
    lay = workloads.make_layout("t", "f16", [1, 7, 4], [9, 20, 4], num_heads=6, num_heads_k=2, head_dim=16,
                                page_block_size=32, seed=3, window_left=5, window_right=0)
    flops, nbytes = bench.algorithmic(lay)
    H, Hkv, D = 6, 2, 16
    pairs, keys = 0, 0
    for sq, sk in zip(lay.seqlens_q, lay.seqlens_k):
        att = set()
        for i in range(sq):
            for j in range(sk):
                if j <= i + sk - sq and j >= i + sk - sq - 5:
                    pairs += 1
                    att.add(j)
        keys += (max(att) - min(att) + 1) if att else 0
    rows = sum(lay.seqlens_q)
    assert flops == 4 * D * H * pairs
    assert nbytes == 2 * Hkv * D * 2 * keys + 2 * rows * H * D * 2 + 4 * H * rows
    assert np.isclose(bench.headline_unit(flops, nbytes)[1], nbytes / 1e9)  # a tiny decode is bandwidth-bound
