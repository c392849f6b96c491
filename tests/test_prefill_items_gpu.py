"""The persistent prefill kernels over many work items per CTA (GPU).

Both prefill kernels run one CTA per SM and take (query-tile pair or query tile, kv head)
items from a device counter; rings, S/P handshakes and barrier phases run on from item to
item.  These batches hold a few hundred prefill-class sequences, so every CTA takes several
items of different lengths: causal and chunked sequences, sequences whose first rows attend
no key (more queries than keys), sequences with no keys at all, decode-class rows beside
them (the split-KV pass, with or without key splits depending on how many SMs the prefill
grid may take), a window, and group sizes that do and do not divide 128.  Rows are
sampled (always including each sequence's first and last query) and compared with the
oracle at the stated tolerances."""
import numpy as np
import pytest

from paged_kv_varlen_flashattention_gb300 import workloads
from tests import _gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _default_kernels(monkeypatch):
    monkeypatch.delenv("PA_DISABLE_TC_PREFILL", raising=False)
    monkeypatch.delenv("PA_FORCE_GENERIC", raising=False)


def _batch(n, seed, *, lo=20, hi=420, short_frac=0.15, nokv_frac=0.03):
    """n sequences: q lengths U[lo, hi]; keys = queries plus U[0, 300] cached (chunked
    prefill), fewer keys than queries for ~10 %, no keys for nokv_frac, and q_len 1..4
    (decode class) for short_frac."""
    rng = np.random.default_rng(seed)
    sq, sk = [], []
    for _ in range(n):
        u = rng.random()
        if u < short_frac:
            q = int(rng.integers(1, 5))
            sq.append(q)
            sk.append(q + int(rng.integers(0, 500)))
        elif u < short_frac + nokv_frac:
            sq.append(int(rng.integers(lo, hi + 1)))
            sk.append(0)
        elif u < short_frac + nokv_frac + 0.1:
            q = int(rng.integers(lo, hi + 1))
            sq.append(q)
            sk.append(int(rng.integers(1, q)))
        else:
            q = int(rng.integers(lo, hi + 1))
            sq.append(q)
            sk.append(q + int(rng.integers(0, 301)))
    return sq, sk


@pytest.mark.parametrize("D,H,Hkv", [(128, 32, 8), (64, 16, 4), (256, 16, 4), (128, 12, 4), (256, 24, 2)])
def test_many_items_per_cta(D, H, Hkv):
    """300 sequences: G = 4 (pairs of 32-query tiles), G = 3 and 12 (padding rows)."""
    sq, sk = _batch(300, seed=200 + D + H)
    lay = workloads.make_layout("items", "bf16", sq, sk, num_heads=H, num_heads_k=Hkv, head_dim=D,
                                page_block_size=64, seed=201 + D, spare=0.1)
    _gpu.check_layout(lay, limit=1500)


def test_many_items_window_fp16():
    sq, sk = _batch(200, seed=210, lo=40, hi=700)
    lay = workloads.make_layout("items_w", "f16", sq, sk, num_heads=16, num_heads_k=2, head_dim=128,
                                page_block_size=32, seed=211, spare=0.1, window_left=150, window_right=0)
    _gpu.check_layout(lay, limit=1500)


def test_many_items_bias():
    sq, sk = _batch(160, seed=220, lo=33, hi=300)
    lay = workloads.make_layout("items_b", "bf16", sq, sk, num_heads=16, num_heads_k=4, head_dim=256,
                                page_block_size=64, seed=221, spare=0.1)
    _gpu.check_layout(lay, alibi=_gpu.alibi_slopes(16, "random", seed=7), limit=1200)


N_RANDOM = 16


def random_items_layout(seed):
    """60..200 sequences drawn around the prefill kernels' item boundaries: query lengths
    that end a tile pair inside its first tile (items without tile B), exactly on a tile,
    just past one; chunked prefill, more queries than keys, no keys, and decode rows; a
    random head dim, group size, page size, window, dtype and (sometimes) position bias."""
    rng = np.random.default_rng(5000 + seed)
    D = int(rng.choice([64, 96, 128, 192, 256]))
    G = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
    Hkv = int(rng.choice([1, 2, 4]))
    P = int(rng.choice([32, 64, 128, 256]))
    qpt = 128 // G
    n = int(rng.integers(60, 201))
    sq, sk = [], []
    for _ in range(n):
        kind = rng.choice(["pair_edge", "tile_edge", "chunk", "fewer_keys", "no_keys", "decode"],
                          p=[0.25, 0.2, 0.25, 0.1, 0.05, 0.15])
        if kind == "pair_edge":    # ends within the first tile of its last pair
            q = int(rng.integers(0, 4)) * 2 * qpt + int(rng.integers(1, qpt + 1))
            k = q + int(rng.integers(0, 200))
        elif kind == "tile_edge":  # a multiple of the tile, or one past it
            q = int(rng.integers(1, 6)) * qpt + int(rng.integers(0, 2))
            k = q
        elif kind == "chunk":
            q = int(rng.integers(33, 300)); k = q + int(rng.integers(1, 600))
        elif kind == "fewer_keys":
            q = int(rng.integers(40, 300)); k = int(rng.integers(1, q))
        elif kind == "no_keys":
            q = int(rng.integers(40, 200)); k = 0
        else:
            q = int(rng.integers(1, 4)); k = int(rng.integers(1, 800))
        sq.append(max(q, 1)); sk.append(k)
    wl, wr = [(-1, 0), (-1, 0), (-1, -1), (int(rng.integers(0, 300)), 0), (int(rng.integers(0, 120)), int(rng.integers(0, 40)))][
        int(rng.integers(0, 5))]
    dtype = "bf16" if rng.random() < 0.6 else "f16"
    lay = workloads.make_layout(f"items_random_{seed}", dtype, sq, sk, num_heads=Hkv * G, num_heads_k=Hkv,
                                head_dim=D, page_block_size=P, seed=6000 + seed, spare=0.1, window_left=wl,
                                window_right=wr)
    alibi = _gpu.alibi_slopes(Hkv * G, "random", seed=seed) if rng.random() < 0.3 else None
    return lay, alibi


@pytest.mark.parametrize("seed", range(N_RANDOM))
def test_random_many_items(seed):
    lay, alibi = random_items_layout(seed)
    _gpu.check_layout(lay, alibi=alibi, limit=1200)


@pytest.mark.parametrize("case", ["prefill_takes_every_sm", "small_prefill"])
def test_decode_pass_beside_prefill(case):
    """The decode-class pass planned beside the prefill kernel.  Eight 1,024-query prompts
    bound the prefill grid at every SM, so the decode sequences beside them (5,000 keys,
    under the per-split key cap) run one CTA per (sequence, kv head) with no combine; one
    64-query prompt leaves the plan's splits (and the combine) to four 8,000-key decode
    sequences.  Sampled rows, always including every sequence's first and last query."""
    if case == "prefill_takes_every_sm":
        sq = [1024] * 8 + [1, 4, 1, 2, 1, 3]
        sk = [1024 + 200 * i for i in range(8)] + [5000, 4990, 4321, 5000, 17, 3000]
    else:
        sq = [64, 1, 1, 4, 1]
        sk = [64, 8000, 7999, 8000, 6500]
    lay = workloads.make_layout(f"beside_{case}", "bf16", sq, sk, num_heads=32, num_heads_k=8, head_dim=128,
                                page_block_size=32, seed=97, spare=0.1)
    _gpu.check_layout(lay, limit=1536)
