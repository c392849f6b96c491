"""The tensor-core prefill kernel for head_dim 129..256 against the oracle (GPU).

One 128-row query tile per CTA, q held in tensor memory, 64-key K/V tiles, S double-buffered
over consecutive key tiles.  These cases cover head dims that leave the last 64-column chunk
partly or wholly empty (136, 192), group sizes that divide 128 and one that does not (3:
padding rows), several query tiles per sequence and single-tile sequences, chunked prefill
(fewer queries than keys), sequences whose rows attend nothing (more queries than keys),
windows, every page size (32-key boxes below 64), fp16, the position bias, the non-paged
mode, and a batch mixing prefill-class sequences with decode-class ones (which the split-KV
pass takes).  The caches hold NaN in every slot no sequence owns.  Rows are sampled (always
including each sequence's first and last query) and compared at the stated tolerances."""
import pytest

from paged_kv_varlen_flashattention_gb300 import workloads
from tests import _gpu

pytestmark = pytest.mark.gpu


def _lay(sq, sk, H, Hkv, D=256, P=64, wl=-1, wr=0, dtype="bf16", seed=91, paged=True):
    lay = workloads.make_layout("pf256", dtype, sq, sk, num_heads=H, num_heads_k=Hkv, head_dim=D,
                                page_block_size=P, seed=seed, spare=0.1, window_left=wl, window_right=wr)
    lay.paged = paged
    return lay


@pytest.fixture(autouse=True)
def _tensor_core_prefill(monkeypatch):
    monkeypatch.delenv("PA_DISABLE_TC_PREFILL", raising=False)
    monkeypatch.delenv("PA_FORCE_GENERIC", raising=False)


@pytest.mark.parametrize("D", [136, 192, 256])
@pytest.mark.parametrize("G", [1, 2, 3, 8])
def test_head_dims_and_groups(D, G):
    """Causal prefill: 300 and 77 queries (several tiles, a ragged last one) and one sequence
    of 40 queries over 300 keys (chunked)."""
    _gpu.check_layout(_lay([300, 77, 40], [300, 77, 300], H=2 * G, Hkv=2, D=D, seed=92 + D + G), limit=3000)


@pytest.mark.parametrize("P", [32, 64, 128, 256])
def test_page_sizes(P):
    _gpu.check_layout(_lay([200, 129], [700, 129], H=8, Hkv=2, P=P, seed=93), limit=3000)


@pytest.mark.parametrize("wl,wr", [(-1, -1), (100, 0), (0, 0), (63, 5), (-1, 64)])
def test_windows(wl, wr):
    _gpu.check_layout(_lay([160, 90], [400, 90], H=8, Hkv=4, wl=wl, wr=wr, seed=94), limit=3000)


def test_more_queries_than_keys():
    """Rows before the first key attend nothing (out 0, lse -inf); one sequence has no keys."""
    _gpu.check_layout(_lay([120, 64, 33], [40, 0, 33], H=8, Hkv=2, seed=95), limit=3000)


def test_fp16():
    _gpu.check_layout(_lay([150, 70], [150, 300], H=8, Hkv=2, dtype="f16", seed=96), limit=3000)


def test_non_paged():
    _gpu.check_layout(_lay([130, 300], [130, 500], H=4, Hkv=1, paged=False, seed=97), limit=3000)


def test_alibi():
    lay = _lay([140, 60], [300, 60], H=8, Hkv=2, seed=98)
    _gpu.check_layout(lay, alibi=_gpu.alibi_slopes(8, "random", seed=4), limit=3000)
    lay = _lay([100], [900], H=4, Hkv=2, wl=300, seed=99)
    _gpu.check_layout(lay, alibi=_gpu.alibi_slopes(4), limit=3000)


def test_mixed_with_decode_rows():
    """Prefill-class sequences beside decode-class ones (q_len 1 and 4, G = 4)."""
    _gpu.check_layout(_lay([1, 200, 4, 1, 90, 4], [900, 250, 300, 17, 600, 5], H=8, Hkv=2, seed=100), limit=3000)


@pytest.mark.parametrize("G", [16, 64, 128])
def test_large_groups(G):
    """128 / G queries per tile: 8, 2 and 1 (a group of 128 heads fills a tile with one query)."""
    _gpu.check_layout(_lay([70, 9], [200, 9], H=G, Hkv=1, D=192, seed=102 + G), limit=3000)


def test_long_causal():
    """Two sequences of 2,048 and 1,500 queries (16 and 12 query tiles over up to 32 key tiles)."""
    _gpu.check_layout(_lay([2048, 1500], [2048, 1500], H=16, Hkv=4, seed=101), limit=2048)
