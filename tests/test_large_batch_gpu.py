"""Decode batches of serving size against the oracle (GPU).

The decode kernel launches sequences longest first.  When the plan splits some sequence
of a batch of 16 to 1,024 sequences, a one-CTA pass lists the (sequence, split) items on
the device, longest sequences first, and persistent CTAs take them in turn (the list sits
at the start of the call's scratch, the split partial results after it).  Otherwise it
ranks batches of up to 160 sequences inside every CTA, batches of 161 to 1,024 through a
separate one-CTA ranking pass whose order sits at the start of the scratch, and keeps the
index order above 1,024 and for grids that fit one wave of resident CTAs.  These cases reach each branch on
both sides of its bounds, with skewed lengths (a few sequences far longer than the rest),
q_len 1 and 4 mixed in one batch, sequences with fewer keys than queries (rows that attend
nothing), a few prefill-class sequences in the same batch, and NaN in every cache slot
no sequence owns.  Sampled rows always include the first and last query of every
sequence (first and last head); all compared element by element at the stated tolerances.

The block table is the per-sequence map of "flash-attn-varlen paged expects k/v tensors
of rank 4" (What it means): one shared pool, one row of physical blocks per sequence.
"""
import numpy as np
import pytest

from paged_kv_varlen_flashattention_gb300 import workloads
from tests import _gpu

pytestmark = pytest.mark.gpu


def skewed_layout(batch, seed, *, H=8, Hkv=2, D=128, P=32, long_n=3, long_k=20000, q4_frac=0.3,
                  prefill_n=0, short_hi=600, dtype="bf16"):
    """`batch` sequences: sk ~ U[1, short_hi] except `long_n` of about `long_k` keys; q_len 4
    for a fraction of them (else 1); `prefill_n` of them get 64 queries (prefill class)."""
    rng = np.random.default_rng(seed)
    sk = rng.integers(1, short_hi, size=batch, endpoint=True)
    longs = rng.choice(batch, size=long_n, replace=False)
    sk[longs] = long_k - rng.integers(0, 100, size=long_n)
    sq = np.where(rng.random(batch) < q4_frac, 4, 1)
    if prefill_n:
        pre = rng.choice(np.setdiff1d(np.arange(batch), longs), size=prefill_n, replace=False)
        sq[pre] = 64
        sk[pre] = np.maximum(sk[pre], 64 + rng.integers(0, 300, size=prefill_n))
    return workloads.make_layout(f"skewed_{batch}", dtype, sq.tolist(), sk.tolist(), num_heads=H, num_heads_k=Hkv,
                                 head_dim=D, page_block_size=P, seed=seed, spare=0.05)


@pytest.mark.parametrize("batch", [160, 161])
def test_in_cta_ranking_bound(batch):
    """160 and 161 sequences with a few long ones (split): the persistent work-list mode."""
    _gpu.check_layout(skewed_layout(batch, seed=31), limit=2048)


@pytest.mark.parametrize("batch", [160, 161])
def test_ranking_without_splits(batch):
    """No sequence split (all under the split cap, more units than CTA slots): 160 ranked
    inside every CTA, 161 by the separate ranking pass."""
    _gpu.check_layout(skewed_layout(batch, seed=37, long_n=2, long_k=6000, short_hi=2000), limit=2048)


@pytest.mark.parametrize("tiles", [None, "8"])
def test_in_cta_ranking_with_splits_small_batch(tiles, monkeypatch):
    """Below 16 sequences the split plan keeps the grid of (split, kv head, sequence) CTAs:
    the plan's own splits fill one wave of resident CTAs (index order); 8-tile splits make
    several waves, ranked inside every CTA."""
    if tiles:
        monkeypatch.setenv("PA_SPLIT_TILES", tiles)
    _gpu.check_layout(skewed_layout(12, seed=38, long_n=2, long_k=30000, short_hi=700), limit=2048)


def test_work_list_rows_without_keys_and_empty_sequences():
    """Work-list mode with sequences whose rows attend nothing (fewer keys than queries, and
    no keys at all) and sequences with no queries: every real row is written."""
    rng = np.random.default_rng(39)
    batch = 40
    sk = rng.integers(1, 900, size=batch, endpoint=True)
    sq = np.where(rng.random(batch) < 0.3, 4, 1)
    sk[[3, 17]] = 25000  # split
    sk[[5, 9]] = [2, 0]  # rows past the keys
    sq[[5, 9]] = 4
    sq[[11, 23]] = 0     # no queries
    lay = workloads.make_layout("worklist_edges", "bf16", sq.tolist(), sk.tolist(), num_heads=8, num_heads_k=2,
                                head_dim=128, page_block_size=32, seed=39, spare=0.05)
    _gpu.check_layout(lay, limit=4096)


def test_ranking_pass_group_of_eight_with_prefill_rows():
    """300 sequences, G = 8 (q_len 4 -> 32 rows), a few prefill-class sequences beside them."""
    _gpu.check_layout(skewed_layout(300, seed=32, H=16, Hkv=2, prefill_n=3), limit=2048)


def test_ranking_pass_upper_bound_head_dim_64():
    """1,024 sequences, the largest batch the ranking pass orders."""
    _gpu.check_layout(skewed_layout(1024, seed=33, D=64, long_n=5), limit=4096)


def test_index_order_above_1024_head_dim_256():
    """1,500 sequences: launched in index order (no ranking)."""
    _gpu.check_layout(skewed_layout(1500, seed=34, D=256, P=64, long_n=4, long_k=12000, short_hi=300),
                      limit=6000)


@pytest.mark.parametrize("tiles", ["1", "3"])
def test_ranking_pass_with_forced_splits(tiles, monkeypatch):
    """The order and the split partials share the scratch: order first, partials after it."""
    monkeypatch.setenv("PA_SPLIT_TILES", tiles)
    _gpu.check_layout(skewed_layout(400, seed=35, long_k=3000), limit=2048)


def test_fp16_large_batch():
    _gpu.check_layout(skewed_layout(200, seed=36, dtype="f16"), limit=2048)


def test_skewed_batch_one_very_long_sequence():
    """The skewed decode workload at full size (63 sequences of 512..4,096 keys and one of
    131,072): the long sequence's keys are split over many CTAs (at most 8,192 keys each) and
    merged by the combine, the short ones stay whole.  All heads of the long sequence's query
    and sampled rows of the others."""
    import torch

    lay = workloads.CONFIGS["skewed_decode_bf16"]()
    long_b = int(np.argmax(lay.seqlens_k))
    inp = workloads.materialize(lay, device="cuda")
    out, lse = _gpu.run_cuda(inp)
    cq, _ = lay.cu_seqlens()
    t = int(cq[long_b])  # the long sequence's one query token
    long_rows = np.arange(t * lay.num_heads, (t + 1) * lay.num_heads, dtype=np.int64)
    rows = np.unique(np.concatenate([_gpu.sample_rows(lay, 512), long_rows]))
    ref_o, ref_l = _gpu.oracle_for(inp.to("cpu"), rows)
    _gpu.compare(lay, out, lse, ref_o, ref_l, rows)
    torch.cuda.synchronize()


@pytest.mark.parametrize("wl", [-1, 1000])
def test_work_list_with_bias_and_window(wl):
    """Work-list mode (40 sequences, two split) with the position bias, causal and windowed."""
    rng = np.random.default_rng(40 + max(wl, 0))
    sk = rng.integers(1, 900, size=40, endpoint=True)
    sk[[4, 29]] = 22000
    sq = np.where(rng.random(40) < 0.3, 4, 1)
    lay = workloads.make_layout("worklist_bias", "bf16", sq.tolist(), sk.tolist(), num_heads=8, num_heads_k=2,
                                head_dim=128, page_block_size=64, seed=41, spare=0.05, window_left=wl,
                                window_right=0)
    _gpu.check_layout(lay, limit=4096, alibi=_gpu.alibi_slopes(8, "random", seed=5))



@pytest.mark.parametrize("D,batch,long_n,wl,bias", [(128, 12, 2, -1, False), (128, 60, 3, -1, False),
                                                     (64, 200, 2, 300, False), (256, 40, 2, -1, True),
                                                     (128, 300, 0, -1, False)])
def test_two_group_kernel_with_narrow_units(D, batch, long_n, wl, bias):
    """G = 8: q_len 1 gives 8 rows, q_len 4 gives 32, so the plan runs the two-row-group
    decode kernel, and every unit of 16 rows or fewer takes the one-group body on the same
    shared-memory layout.  The batches cover the grid of CTAs (12, 300 sequences), the
    persistent work list with split sequences (60, 200, 40), a window and the bias."""
    lay = skewed_layout(batch, seed=40 + batch + D, H=16, Hkv=2, D=D, long_n=long_n, long_k=9000, q4_frac=0.25,
                        short_hi=1500)
    lay.window_left = wl
    alibi = _gpu.alibi_slopes(16, "random", seed=batch) if bias else None
    _gpu.check_layout(lay, alibi=alibi, limit=2048)
