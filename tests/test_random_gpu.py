"""Seeded random configurations against the oracle (GPU): head counts and group sizes,
head dims, page sizes, windows, lengths (empty sequences, sq > sk, long-query and decode
rows in one batch), dtypes and the linear position bias, all rows compared at the stated
tolerances; each case is small enough for the oracle to finish in well under a second.
A second family draws batches of 16..48 sequences with a few long (split) ones and some
prefill-class ones, sometimes with forced split sizes (sampled rows)."""
import numpy as np
import pytest

from paged_kv_varlen_flashattention_gb300 import workloads
from tests import _gpu

pytestmark = pytest.mark.gpu

N_CASES = 64


def random_layout(seed):
    rng = np.random.default_rng(1000 + seed)
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 3, 4, 8]))
    D = int(rng.choice([64, 96, 128, 256, 512]))
    P = int(rng.choice([32, 64, 128]))
    batch = int(rng.integers(1, 6))
    sq, sk = [], []
    for _ in range(batch):
        kind = rng.choice(["decode", "chunk", "prompt", "empty", "short"])
        if kind == "decode":
            k = int(rng.integers(1, 400)); q = int(rng.integers(1, 5))
        elif kind == "chunk":
            k = int(rng.integers(64, 500)); q = int(rng.integers(16, 128))
        elif kind == "prompt":
            k = int(rng.integers(33, 300)); q = k
        elif kind == "empty":
            k = int(rng.integers(0, 50)); q = 0
        else:  # more queries than keys: the first rows attend nothing under a causal mask
            k = int(rng.integers(0, 20)); q = int(rng.integers(1, 40))
        sq.append(q); sk.append(k)
    wl, wr = [(-1, 0), (-1, -1), (int(rng.integers(0, 100)), 0), (int(rng.integers(0, 60)), int(rng.integers(0, 30)))][
        int(rng.integers(0, 4))]
    dtype = "bf16" if rng.random() < 0.6 else "f16"
    lay = workloads.make_layout(f"random_{seed}", dtype, sq, sk, num_heads=Hkv * G, num_heads_k=Hkv, head_dim=D,
                                page_block_size=P, seed=seed, spare=0.2, window_left=wl, window_right=wr)
    alibi = _gpu.alibi_slopes(Hkv * G, "random", seed=seed) if rng.random() < 0.3 else None
    return lay, alibi


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_configuration(seed):
    lay, alibi = random_layout(seed)
    if lay.total_q == 0:
        pytest.skip("no queries drawn")
    _gpu.check_layout(lay, alibi=alibi)


N_BATCH_CASES = 24


def random_batch_layout(seed):
    """16..48 sequences: mostly decode rows, one to three longer ones, a few prefill-class
    ones.  With fewer (sequence, kv head) units than CTA slots every sequence is split, so
    the persistent work-list mode runs for head dims up to 256."""
    rng = np.random.default_rng(5000 + seed)
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4, 8]))
    D = int(rng.choice([64, 96, 128, 192, 256, 320, 512]))
    P = int(rng.choice([32, 64, 128]))
    batch = int(rng.integers(16, 49))
    sq = [int(x) for x in np.where(rng.random(batch) < 0.3, rng.integers(2, 5, size=batch), 1)]
    sk = [int(x) for x in rng.integers(1, 600, size=batch, endpoint=True)]
    for b in rng.choice(batch, size=int(rng.integers(1, 4)), replace=False):
        sk[b] = int(rng.integers(3000, 6000))
    for b in rng.choice(batch, size=int(rng.integers(0, 3)), replace=False):
        sq[b] = int(rng.integers(40, 120))
        sk[b] = max(sk[b], sq[b] + int(rng.integers(0, 200)))
    wl, wr = [(-1, 0), (-1, 0), (int(rng.integers(0, 3000)), 0), (-1, -1)][int(rng.integers(0, 4))]
    dtype = "bf16" if rng.random() < 0.6 else "f16"
    lay = workloads.make_layout(f"random_batch_{seed}", dtype, sq, sk, num_heads=Hkv * G, num_heads_k=Hkv,
                                head_dim=D, page_block_size=P, seed=seed, spare=0.1, window_left=wl, window_right=wr)
    alibi = _gpu.alibi_slopes(Hkv * G, "random", seed=seed) if rng.random() < 0.25 else None
    split_tiles = str(int(rng.integers(1, 40))) if rng.random() < 0.3 else None
    return lay, alibi, split_tiles


@pytest.mark.parametrize("seed", range(N_BATCH_CASES))
def test_random_batch(seed, monkeypatch):
    lay, alibi, split_tiles = random_batch_layout(seed)
    if split_tiles is not None:
        monkeypatch.setenv("PA_SPLIT_TILES", split_tiles)
    _gpu.check_layout(lay, alibi=alibi, limit=800)
