"""The KV-append oracle against its pins (CPU only), and planted mistakes in copies of it."""
import inspect
import textwrap

import numpy as np
import pytest

import oracle
from tests import _pins


def _case(rng, P=32, Hkv=2, D=16, dtype=np.float16):
    """Sequences after the append: sk keys, the last n of them new (n = 0, a decode step, a
    chunk, a whole fresh prompt); pages from a shuffled pool with spare blocks."""
    sk = [70, 33, 1, 96, 40, 5]
    n = [7, 0, 1, 96, 40, 2]
    pages = [(s + P - 1) // P for s in sk]
    nb = sum(pages) + 4
    perm = rng.permutation(nb)
    bt = np.full((len(sk), max(pages) + 1), -1, dtype=np.int32)
    cur = 0
    for b, p in enumerate(pages):
        bt[b, :p] = perm[cur:cur + p]
        cur += p
    k_cache = (rng.standard_normal((nb, P, Hkv, D))).astype(dtype)
    v_cache = (rng.standard_normal((nb, P, Hkv, D))).astype(dtype)
    k_new = rng.standard_normal((sum(n), Hkv, D)).astype(dtype)
    v_new = rng.standard_normal((sum(n), Hkv, D)).astype(dtype)
    return sk, n, bt, k_cache, v_cache, k_new, v_new


def gather(cache, bt, b, sk):
    """Key rows 0..sk-1 of sequence b, read through the block table with numpy indexing."""
    P = cache.shape[1]
    pos = np.arange(sk)
    return cache[bt[b, pos // P], pos % P]


def pin_append_gather(kv_append):
    """After the append, sequence b read through its block table holds its old keys followed
    by its new ones, bit for bit; every other cache slot keeps its bytes."""
    rng = np.random.default_rng(201)
    sk, n, bt, kc, vc, kn, vn = _case(rng)
    kc0, vc0 = kc.copy(), vc.copy()
    kv_append(kn, vn, _pins.cu(n), _pins.cu(sk), bt, kc, vc)
    off = 0
    written = np.zeros(kc.shape[:2], dtype=bool)
    for b in range(len(sk)):
        for cache, old, new in ((kc, kc0, kn), (vc, vc0, vn)):
            got = gather(cache, bt, b, sk[b])
            assert np.array_equal(got[sk[b] - n[b]:].view(np.uint16), new[off:off + n[b]].view(np.uint16)), b
            assert np.array_equal(got[:sk[b] - n[b]].view(np.uint16),
                                  gather(old, bt, b, sk[b])[:sk[b] - n[b]].view(np.uint16)), b
        pos = np.arange(sk[b] - n[b], sk[b])
        written[bt[b, pos // kc.shape[1]], pos % kc.shape[1]] = True
        off += n[b]
    assert np.array_equal(kc[~written].view(np.uint16), kc0[~written].view(np.uint16))
    assert np.array_equal(vc[~written].view(np.uint16), vc0[~written].view(np.uint16))


def pin_append_then_attention(kv_append):
    """Attention over the paged cache after the append equals attention over the packed
    keys in the non-paged mode (the oracle's paging identity), bit for bit."""
    rng = np.random.default_rng(202)
    sk, n, bt, kc, vc, kn, vn = _case(rng)
    kv_append(kn, vn, _pins.cu(n), _pins.cu(sk), bt, kc, vc)
    k_packed = np.concatenate([gather(kc, bt, b, sk[b]) for b in range(len(sk))])
    v_packed = np.concatenate([gather(vc, bt, b, sk[b]) for b in range(len(sk))])
    H = 4
    q = _pins.f16(rng, (sum(n), H, kc.shape[-1]))
    a = oracle.attention("f16", q, kc, vc, _pins.cu(n), _pins.cu(sk), bt, 0.25, -1, 0)
    b = oracle.attention("f16", q, k_packed, v_packed, _pins.cu(n), _pins.cu(sk), None, 0.25, -1, 0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def pin_append_rejects(kv_append):
    rng = np.random.default_rng(203)
    sk, n, bt, kc, vc, kn, vn = _case(rng)
    n_bad = list(n)
    n_bad[2] = 2  # two new tokens in a sequence of one key
    kn2 = np.zeros((sum(n_bad),) + kn.shape[1:], dtype=kn.dtype)
    with pytest.raises(ValueError):
        kv_append(kn2, kn2, _pins.cu(n_bad), _pins.cu(sk), bt, kc, vc)
    bt_bad = bt.copy()
    bt_bad[0, 2] = kc.shape[0]  # a block id past the pool
    with pytest.raises(ValueError):
        kv_append(kn, vn, _pins.cu(n), _pins.cu(sk), bt_bad, kc, vc)


APPEND_PINS = [pin_append_gather, pin_append_then_attention, pin_append_rejects]


@pytest.mark.parametrize("pin", APPEND_PINS, ids=[p.__name__ for p in APPEND_PINS])
def test_append_pins(pin):
    pin(oracle.kv_append)


APPEND_MUTANTS = {
    "start_at_zero": ("j = sk_b - n_b + t", "j = t"),
    "off_by_one": ("j = sk_b - n_b + t", "j = sk_b - n_b + t + 1"),
    "slot_as_page": ("k_cache[blk, j % P] = ", "k_cache[blk, j // P] = "),
    "values_from_keys": ("v_cache[blk, j % P] = v_new[", "v_cache[blk, j % P] = k_new["),
    "page_from_slot": ("blk = int(bt[b, j // P])", "blk = int(bt[b, j % P])"),
}


@pytest.mark.parametrize("name", sorted(APPEND_MUTANTS))
def test_append_mutant_is_caught(name):
    old, new = APPEND_MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(oracle.kv_append))
    assert src.count(old) == 1, name
    ns = {"np": np}
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    caught = False
    for pin in APPEND_PINS:
        try:
            pin(ns["kv_append"])
        except (AssertionError, IndexError, ValueError):
            caught = True
            break
    assert caught, f"append mutant {name} passed every pin"
