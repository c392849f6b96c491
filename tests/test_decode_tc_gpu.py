"""The tensor-core decode kernel (tcgen05, keys in the MMA rows) against the oracle (GPU).

Decode-class rows (q_len x GQA group <= 32) of head_dim 128..512 run on it when
PA_DECODE_TC=1 (otherwise on the warp-sliced mma.sync kernel, or the general kernel above
256), which these cases set, so that one kernel is checked over every row count (16- and
32-row MMAs, padding rows), head dim (192, 320 and 448 leave part of the last 128-column
chunk empty), page size, window, split count, dtype, bias and the non-paged mode.  The
caches hold NaN in every slot no sequence owns, and sequences with fewer keys than queries
give rows that attend nothing.  All rows are compared at the stated tolerances."""
import pytest

from paged_kv_varlen_flashattention_gb300 import workloads
from tests import _gpu

pytestmark = pytest.mark.gpu


def _lay(sq, sk, H, Hkv, D, P=32, wl=-1, wr=0, dtype="bf16", seed=51, paged=True, std=1.0):
    lay = workloads.make_layout("tc", dtype, sq, sk, num_heads=H, num_heads_k=Hkv, head_dim=D, page_block_size=P,
                                seed=seed, spare=0.2, window_left=wl, window_right=wr, std=std)
    lay.paged = paged
    return lay


@pytest.fixture(autouse=True)
def _tc(monkeypatch):
    monkeypatch.setenv("PA_DECODE_TC", "1")


@pytest.mark.parametrize("D", [128, 192, 256, 320, 448, 512])
@pytest.mark.parametrize("G,q", [(4, 1), (8, 4), (4, 3)])
def test_head_dims_and_rows(D, G, q):
    """rows = q x G: 4 (16-row MMA), 32 and 12 (32- and 16-row MMAs with padding rows)."""
    _gpu.check_layout(_lay([q, q, q], [1, 300, 1000], H=2 * G, Hkv=2, D=D, seed=52 + D + G))


@pytest.mark.parametrize("P", [32, 64, 128, 256])
def test_page_sizes(P):
    _gpu.check_layout(_lay([1, 4, 2], [777, 129, 2000], H=16, Hkv=2, D=512, P=P, seed=53))


@pytest.mark.parametrize("wl,wr", [(-1, -1), (100, 0), (0, 0), (257, 3), (-1, 7)])
def test_windows(wl, wr):
    _gpu.check_layout(_lay([1, 4, 3, 2], [600, 1030, 5, 129], H=8, Hkv=2, D=512, wl=wl, wr=wr, seed=54))


@pytest.mark.parametrize("tiles", ["1", "2", "3"])
def test_forced_splits(tiles, monkeypatch):
    monkeypatch.setenv("PA_SPLIT_TILES", tiles)
    _gpu.check_layout(_lay([4, 1, 4], [1100, 2000, 129], H=16, Hkv=2, D=512, seed=55))
    _gpu.check_layout(_lay([1, 2], [700, 1500], H=8, Hkv=2, D=128, seed=56))


def test_more_queries_than_keys():
    _gpu.check_layout(_lay([4, 4, 1], [2, 3, 0], H=16, Hkv=2, D=512, seed=57))


def test_fp16_and_scale():
    _gpu.check_layout(_lay([4, 1], [900, 333], H=16, Hkv=2, D=512, dtype="f16", seed=58))
    _gpu.check_layout(_lay([2, 3], [500, 64], H=8, Hkv=4, D=256, dtype="f16", seed=59, std=2.0))


def test_non_paged():
    _gpu.check_layout(_lay([4, 1, 3], [300, 129, 1000], H=16, Hkv=2, D=512, paged=False, seed=60))


def test_alibi():
    lay = _lay([4, 1, 2], [800, 200, 1300], H=16, Hkv=2, D=512, seed=61)
    _gpu.check_layout(lay, alibi=_gpu.alibi_slopes(16, "random", seed=3))
    lay = _lay([1, 1], [4000, 77], H=8, Hkv=2, D=128, wl=1000, seed=62)
    _gpu.check_layout(lay, alibi=_gpu.alibi_slopes(8))


def test_large_batch_ranked():
    """300 sequences: the ranking pass's order in the scratch, read by this kernel."""
    from tests.test_large_batch_gpu import skewed_layout
    _gpu.check_layout(skewed_layout(300, seed=63, H=16, Hkv=2, D=512, long_k=5000, short_hi=300), limit=2048)


def test_long_context_full_size():
    _gpu.check_layout(workloads.CONFIGS["long_d512_bf16"](), limit=256)
    _gpu.check_layout(workloads.CONFIGS["long_bf16"](), limit=96)
