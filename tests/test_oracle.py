"""The oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
from tests import _pins


def test_decoders_match_numpy_and_torch():
    _pins.pin_decoders(oracle.decode)


@pytest.mark.parametrize("paged", [False, True])
def test_mask_bruteforce(paged):
    _pins.pin_mask_bruteforce(oracle.attention, paged=paged)


def test_sdpa_float64():
    _pins.pin_sdpa(oracle.attention)


def test_paging_identity():
    _pins.pin_paging_identity(oracle.attention)


def test_block_permutation_bit_identical():
    _pins.pin_block_permutation(oracle.attention)


def test_rows_sum_to_one():
    _pins.pin_rows_sum_to_one(oracle.attention)


def test_zero_query_mean_and_log_count():
    _pins.pin_zero_query(oracle.attention)


def test_single_key_window():
    _pins.pin_single_key(oracle.attention)


def test_gqa_equals_repeated_mha():
    _pins.pin_gqa_repeat(oracle.attention)


def test_chunked_prefill_rows():
    _pins.pin_chunking(oracle.attention)


def test_closed_form_two_keys():
    _pins.pin_closed_form(oracle.attention)


def test_bf16_inputs():
    _pins.pin_bf16_path(oracle.attention)


def test_row_subset_matches_full():
    """Computing a subset of rows gives the same values as the full run."""
    rng = np.random.default_rng(1)
    sq, sk, q, k, v = _pins._multi_seq(rng)
    full_o, full_l = oracle.attention("f16", q, k, v, _pins.cu(sq), _pins.cu(sk), None, 0.3, -1, 0)
    rows = np.array([0, 5, 17, len(full_l) - 1])
    o, l = oracle.attention("f16", q, k, v, _pins.cu(sq), _pins.cu(sk), None, 0.3, -1, 0, rows=rows)
    assert np.array_equal(o, full_o[rows]) and np.array_equal(l, full_l[rows])


def test_rejects_bad_arguments():
    rng = np.random.default_rng(2)
    sq, sk, q, k, v = _pins._multi_seq(rng)
    with pytest.raises(ValueError):
        oracle.attention("f16", q, k, v, _pins.cu(sq), _pins.cu(sk), None, 0.3, -1, 0,
                         rows=np.array([10 ** 6]))


def test_alibi_equals_sdpa_with_bias_mask():
    _pins.pin_alibi_sdpa(oracle.attention)


def test_alibi_two_key_closed_forms():
    _pins.pin_alibi_two_keys(oracle.attention)


def test_alibi_zero_slopes_is_no_bias():
    _pins.pin_alibi_zero_slopes(oracle.attention)


def test_padded_equals_batched_sdpa():
    """The padded-batch oracle equals torch's scaled_dot_product_attention on the batched
    (B, H, S, D) float64 tensors (full and causal, grouped-query heads), and its lse (B, H,
    Sq) equals torch.logsumexp of the scaled scores."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(121)
    B, S, H, Hkv, D, scale = 3, 23, 4, 2, 16, 0.3
    q = _pins.f16(rng, (B, S, H, D))
    k = _pins.f16(rng, (B, S, Hkv, D))
    v = _pins.f16(rng, (B, S, Hkv, D))
    tq = torch.from_numpy(q.astype(np.float64)).permute(0, 2, 1, 3)
    tk = torch.from_numpy(k.astype(np.float64)).permute(0, 2, 1, 3)
    tv = torch.from_numpy(v.astype(np.float64)).permute(0, 2, 1, 3)
    for causal in (False, True):
        out, lse = oracle.attention_padded("f16", q, k, v, scale, -1, 0 if causal else -1)
        ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale, enable_gqa=True)
        assert np.allclose(out, ref.permute(0, 2, 1, 3).numpy(), rtol=1e-10, atol=1e-12), causal
        sc = scale * (tq @ tk.repeat_interleave(H // Hkv, dim=1).transpose(-1, -2))
        if causal:
            sc = sc.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
        assert np.allclose(lse, torch.logsumexp(sc, dim=-1).numpy(), rtol=1e-12, atol=1e-12), causal
