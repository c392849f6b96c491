"""The quarter-column decode kernel (head_dim 257..512, at most 32 rows a kv head) against
the oracle (GPU).

Eight consumer warps split the head dim in quarters of 128 columns and exchange partial
scores every 32-key tile; with 16 rows the two warp groups take the two 16-key halves of
every tile and are merged at the end.  These cases cover both row counts with padding rows,
head dims that leave quarters partly or wholly empty (264, 320, 448), every page size, the
windows (tiles inside every row's interval skip the mask), forced split counts with the
combine, more queries than keys (rows that attend nothing), fp16, the position bias, the
non-paged mode, a batch ranked by the separate pass, scores rising in steps along the keys
(every row's running reference raised many times inside a split) and the long-context
workload at full size.  The caches hold NaN in every slot no sequence owns.  All rows are compared at the
stated tolerances."""
import pytest

from paged_kv_varlen_flashattention_gb300 import workloads
from tests import _gpu

pytestmark = pytest.mark.gpu


def _lay(sq, sk, H, Hkv, D, P=32, wl=-1, wr=0, dtype="bf16", seed=71, paged=True, std=1.0):
    lay = workloads.make_layout("d512", dtype, sq, sk, num_heads=H, num_heads_k=Hkv, head_dim=D, page_block_size=P,
                                seed=seed, spare=0.2, window_left=wl, window_right=wr, std=std)
    lay.paged = paged
    return lay


@pytest.fixture(autouse=True)
def _default_kernels(monkeypatch):
    monkeypatch.delenv("PA_DECODE_TC", raising=False)
    monkeypatch.delenv("PA_FORCE_GENERIC", raising=False)


@pytest.mark.parametrize("D", [264, 320, 448, 512])
@pytest.mark.parametrize("G,q", [(4, 1), (8, 4), (4, 3), (16, 1)])
def test_head_dims_and_rows(D, G, q):
    """rows = q x G: 4, 12 and 16 (16-row CTA, two key halves; 4 and 12 leave padding rows)
    and 32 (32-row CTA).  A 32-row batch with an 8-row sequence (the page-size cases) gives
    a row group of padding only."""
    _gpu.check_layout(_lay([q, q, q], [1, 300, 1000], H=2 * G, Hkv=2, D=D, seed=72 + D + G))


@pytest.mark.parametrize("P", [32, 64, 128, 256])
def test_page_sizes(P):
    _gpu.check_layout(_lay([1, 4, 2], [777, 129, 2000], H=16, Hkv=2, D=512, P=P, seed=73))


@pytest.mark.parametrize("wl,wr", [(-1, -1), (100, 0), (0, 0), (257, 3), (-1, 7), (31, 0)])
def test_windows(wl, wr):
    _gpu.check_layout(_lay([1, 4, 3, 2], [600, 1030, 5, 129], H=8, Hkv=2, D=512, wl=wl, wr=wr, seed=74))


@pytest.mark.parametrize("tiles", ["1", "2", "3", "5"])
def test_forced_splits(tiles, monkeypatch):
    monkeypatch.setenv("PA_SPLIT_TILES", tiles)
    _gpu.check_layout(_lay([4, 1, 4], [1100, 2000, 129], H=16, Hkv=2, D=512, seed=75))
    _gpu.check_layout(_lay([1, 2], [700, 1500], H=4, Hkv=2, D=384, seed=76))


def test_more_queries_than_keys():
    _gpu.check_layout(_lay([4, 4, 1, 2], [2, 3, 0, 1], H=16, Hkv=2, D=512, seed=77))


def test_fp16_and_scale():
    _gpu.check_layout(_lay([4, 1], [900, 333], H=16, Hkv=2, D=512, dtype="f16", seed=78))
    _gpu.check_layout(_lay([2, 3], [500, 64], H=8, Hkv=4, D=320, dtype="f16", seed=79, std=2.0))


def test_non_paged():
    _gpu.check_layout(_lay([4, 1, 3], [300, 129, 1000], H=16, Hkv=2, D=512, paged=False, seed=80))
    _gpu.check_layout(_lay([1, 2], [33, 1000], H=4, Hkv=1, D=448, paged=False, seed=81))


def test_alibi():
    lay = _lay([4, 1, 2], [800, 200, 1300], H=16, Hkv=2, D=512, seed=82)
    _gpu.check_layout(lay, alibi=_gpu.alibi_slopes(16, "random", seed=3))
    lay = _lay([1, 1], [4000, 77], H=8, Hkv=2, D=512, wl=1000, seed=83)
    _gpu.check_layout(lay, alibi=_gpu.alibi_slopes(8))


@pytest.mark.parametrize("tiles", [None, "8"])
def test_ranked_in_cta_and_by_pass(tiles, monkeypatch):
    """40 sequences (one wave of 120 CTAs in index order with the plan's splits; ranked
    inside every CTA over the 480 CTAs of 8-tile splits) and 300 (the ranking pass's order
    in the scratch)."""
    from tests.test_large_batch_gpu import skewed_layout
    if tiles:
        monkeypatch.setenv("PA_SPLIT_TILES", tiles)
    _gpu.check_layout(skewed_layout(40, seed=84, H=8, Hkv=1, D=512, long_n=2, long_k=3000, short_hi=300),
                      limit=2048)
    _gpu.check_layout(skewed_layout(300, seed=85, H=16, Hkv=2, D=512, long_k=5000, short_hi=300), limit=2048)


def test_long_context_full_size():
    _gpu.check_layout(workloads.CONFIGS["long_d512_bf16"](), limit=256)


@pytest.mark.parametrize("G,q", [(8, 4), (4, 1)])
def test_scores_rising_in_steps(G, q, monkeypatch):
    """Scores that jump by about 10 (in log2 units) every 64 keys: every row's running
    reference is raised many times inside one split, and with 32 rows the four quarter
    warps of a group, each holding the softmax of its own 8 keys of a tile, must raise it
    together; with 16 rows (two key halves) the halves are merged at the end.  q is all
    ones, key j of a sequence is N(0, 0.1^2) + 0.3 floor(j / 64) in every column; the plan's
    own splits, then forced 3-tile splits; every row compared with the oracle."""
    import torch
    sks = [700, 1000]
    lay = _lay([q, q], sks, H=2 * G, Hkv=2, D=512, seed=91)
    inp = workloads.materialize(lay, device="cuda").to("cuda")
    gen = torch.Generator(device="cuda").manual_seed(91)
    inp.q.fill_(1.0)
    P = lay.page_block_size
    for b, sk in enumerate(sks):
        for page in range((sk + P - 1) // P):
            blk = int(lay.block_table[b, page])
            n = min(P, sk - page * P)
            keys = torch.arange(page * P, page * P + n, device="cuda")
            ramp = (0.3 * torch.div(keys, 64, rounding_mode="floor")).view(n, 1, 1)
            noise = torch.randn((n, lay.num_heads_k, lay.head_dim), generator=gen, device="cuda") * 0.1
            inp.k_cache[blk, :n] = (ramp + noise).to(inp.k_cache.dtype)
    ref_o, ref_l = _gpu.oracle_for(inp.to("cpu"))
    for tiles in (None, "3"):
        if tiles:
            monkeypatch.setenv("PA_SPLIT_TILES", tiles)
        out, lse = _gpu.run_cuda(inp)
        _gpu.compare(lay, out, lse, ref_o, ref_l)
