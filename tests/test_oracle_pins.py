"""The fp64 oracle against what the MARS pages and the mathematics fix (CPU only)."""
import numpy as np
import pytest

import oracle
from tests import pins


def test_mask_matches_fig2_golden():
    pins.check_mask_golden(oracle.mars_mask)


def test_mask_matches_block_construction():
    pins.check_mask_vs_blocks(oracle.mars_mask)


def test_mask_visible_pair_count():
    pins.check_mask_pair_count(oracle.mars_mask)


def test_mask_is_causal_within_blocks():
    pins.check_mask_not_bidirectional(oracle.mars_mask)


def test_mask_eq4_printed_ratios():
    pins.check_mask_eq4_ratio(oracle.mars_mask)


def test_mask_sec33_placeholder_counts():
    pins.check_mask_sec33_counts(oracle.mars_mask)


def test_mask_rows_agree_with_full_mask():
    full = oracle.mars_mask(21, 4)
    rows = np.array([0, 3, 20, 21, 22, 30, 41])
    assert np.array_equal(oracle.mask_rows(21, 4, rows), full[rows])


def test_block_index_is_ceil():
    assert list(oracle.block_index(np.arange(1, 10), 4)) == [1, 1, 1, 1, 2, 2, 2, 2, 3]


def test_train_clean_half_is_causal_attention():
    pins.check_train_clean_half_is_causal(oracle.train_attn)


@pytest.mark.parametrize("L,B", [(22, 4), (24, 8), (10, 3), (5, 1)])
def test_train_noisy_blocks_are_prefix_causal(L, B):
    pins.check_train_noisy_blocks_are_prefix_causal(oracle.train_attn, L=L, B=B)


def test_train_single_key_rows_return_v():
    pins.check_train_single_key_rows(oracle.train_attn)


def test_train_equal_keys_give_mean_of_visible_values():
    pins.check_train_equal_keys_give_mean(oracle.train_attn)


def test_train_bruteforce_triple_loop():
    pins.check_train_bruteforce(oracle.train_attn)


def test_train_lse_matches_logsumexp():
    pins.check_train_lse(oracle.train_attn)


def test_train_block_larger_than_L():
    pins.check_train_block_ge_L(oracle.train_attn)


def test_train_gqa_mapping():
    pins.check_train_gqa_is_repeat_kv(oracle.train_attn)


def test_train_rows_subset():
    pins.check_train_rows_subset(oracle.train_attn)


def test_decode_reproduces_training_noisy_block():
    pins.check_decode_matches_train_block(oracle.decode_attn, oracle.train_attn)


def test_decode_empty_cache_is_causal():
    pins.check_decode_empty_cache_is_causal(oracle.decode_attn)


def test_decode_bruteforce():
    pins.check_decode_bruteforce(oracle.decode_attn)


def test_accept_one_hot_closed_form():
    pins.check_accept_one_hot_closed_form(oracle.accept_rows)


def test_accept_ties_go_to_lowest_index():
    pins.check_accept_ties_lowest_index(oracle.accept_rows)


def test_accept_matches_scipy_and_numpy():
    pins.check_accept_vs_library(oracle.accept_rows)


def test_margin_closed_forms():
    pins.check_margin_closed_forms(oracle.accept_rows)


def test_margin_matches_scipy_and_bounds():
    pins.check_margin_vs_library(oracle.accept_rows)


def test_commit_rule():
    pins.check_commit_rule(oracle.commit_count)


def test_accept_tau_extremes():
    pins.check_accept_tau_extremes(oracle.accept)


def test_batch_min_mode():
    pins.check_batch_min(oracle.accept)


def test_deferred_matches_append_then_decode():
    pins.check_deferred_matches_append_then_decode(oracle.decode_attn_deferred, oracle.decode_attn, oracle.append_kv)


def test_deferred_pending_rows_are_causal():
    pins.check_deferred_pending_rows_are_causal(oracle.decode_attn_deferred, oracle.train_attn)


def test_deferred_invalid_slots():
    pins.check_deferred_invalid_slots(oracle.decode_attn_deferred)


def test_accept_deferred():
    pins.check_accept_deferred(oracle.accept_deferred, oracle.accept)


def test_append():
    pins.check_append(oracle.append_kv)


def test_accept_rejects_non_finite():
    x = np.zeros((1, 1, 8))
    x[0, 0, 3] = np.inf
    with pytest.raises(AssertionError):
        oracle.accept_rows(x)


def test_near_threshold_band():
    flags = oracle.near_threshold(np.array([0.95, 0.95005, 0.9502, 0.94991]), 0.95)
    assert list(flags) == [True, True, False, True]


def test_bwd_vs_autograd():
    pins.check_bwd_vs_autograd(oracle.train_attn_bwd)


def test_bwd_finite_differences():
    pins.check_bwd_finite_differences(oracle.train_attn_bwd, oracle.train_attn)


def test_bwd_gqa_is_repeat_kv():
    pins.check_bwd_gqa_is_repeat_kv(oracle.train_attn_bwd)


def test_bwd_closed_forms():
    pins.check_bwd_closed_forms(oracle.train_attn_bwd)


def test_lm_head_logits_bruteforce():
    pins.check_lm_head_logits_bruteforce(oracle.lm_head_logits)


def test_lm_head_logits_one_hot():
    pins.check_lm_head_logits_one_hot(oracle.lm_head_logits)


def test_lm_head_accept_closed_form():
    pins.check_lm_head_accept_closed_form(oracle.lm_head_accept)
