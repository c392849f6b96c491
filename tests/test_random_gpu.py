"""Seeded random configurations against the oracle (GPU): head counts and group sizes,
head dims, page sizes, windows, lengths (empty sequences, sq > sk, long-query and decode
rows in one batch), dtypes and the linear position bias, all rows compared at the stated
tolerances.  Each case is small enough for the oracle to finish in well under a second."""
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
