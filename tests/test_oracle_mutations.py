"""Plant plausible mistakes in copies of the oracle and check that a pin fails.

Each mutant is the oracle's source with one textual change, executed in a
fresh namespace on the CPU; the real oracle is untouched.
"""
import inspect
import types

import pytest

import oracle.mars_oracle as real
from tests import pins

SOURCE = inspect.getsource(real)


def mutant(old, new):
    assert SOURCE.count(old) == 1, f"mutation anchor not unique: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(SOURCE.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


def all_pins(m):
    """Run every pin against module m; return the names of the pins that fail."""
    checks = {
        "mask_golden": lambda: pins.check_mask_golden(m.mars_mask),
        "mask_blocks": lambda: pins.check_mask_vs_blocks(m.mars_mask, Ls=(5, 10, 13), Bs=(1, 3, 4)),
        "mask_pairs": lambda: pins.check_mask_pair_count(m.mars_mask),
        "mask_causal_in_block": lambda: pins.check_mask_not_bidirectional(m.mars_mask),
        "mask_eq4": lambda: pins.check_mask_eq4_ratio(m.mars_mask),
        "mask_sec33": lambda: pins.check_mask_sec33_counts(m.mars_mask),
        "train_clean": lambda: pins.check_train_clean_half_is_causal(m.train_attn),
        "train_noisy": lambda: pins.check_train_noisy_blocks_are_prefix_causal(m.train_attn),
        "train_single": lambda: pins.check_train_single_key_rows(m.train_attn),
        "train_equal_keys": lambda: pins.check_train_equal_keys_give_mean(m.train_attn),
        "train_lse": lambda: pins.check_train_lse(m.train_attn),
        "train_gqa": lambda: pins.check_train_gqa_is_repeat_kv(m.train_attn),
        "decode_train": lambda: pins.check_decode_matches_train_block(m.decode_attn, m.train_attn),
        "decode_empty": lambda: pins.check_decode_empty_cache_is_causal(m.decode_attn),
        "decode_brute": lambda: pins.check_decode_bruteforce(m.decode_attn),
        "accept_closed": lambda: pins.check_accept_one_hot_closed_form(m.accept_rows),
        "accept_ties": lambda: pins.check_accept_ties_lowest_index(m.accept_rows),
        "accept_lib": lambda: pins.check_accept_vs_library(m.accept_rows),
        "margin_closed": lambda: pins.check_margin_closed_forms(m.accept_rows),
        "margin_lib": lambda: pins.check_margin_vs_library(m.accept_rows),
        "commit": lambda: pins.check_commit_rule(m.commit_count),
        "tau": lambda: pins.check_accept_tau_extremes(m.accept),
        "append": lambda: pins.check_append(m.append_kv),
        "batch_min": lambda: pins.check_batch_min(m.accept),
        "deferred_eq": lambda: pins.check_deferred_matches_append_then_decode(m.decode_attn_deferred, m.decode_attn,
                                                                              m.append_kv),
        "deferred_causal": lambda: pins.check_deferred_pending_rows_are_causal(m.decode_attn_deferred, m.train_attn),
        "deferred_invalid": lambda: pins.check_deferred_invalid_slots(m.decode_attn_deferred),
        "accept_deferred": lambda: pins.check_accept_deferred(m.accept_deferred, m.accept),
        "bwd_autograd": lambda: pins.check_bwd_vs_autograd(m.train_attn_bwd),
        "bwd_fd": lambda: pins.check_bwd_finite_differences(m.train_attn_bwd, m.train_attn),
        "bwd_gqa": lambda: pins.check_bwd_gqa_is_repeat_kv(m.train_attn_bwd),
        "bwd_closed": lambda: pins.check_bwd_closed_forms(m.train_attn_bwd),
        "lm_brute": lambda: pins.check_lm_head_logits_bruteforce(m.lm_head_logits),
        "lm_one_hot": lambda: pins.check_lm_head_logits_one_hot(m.lm_head_logits),
        "lm_accept": lambda: pins.check_lm_head_accept_closed_form(m.lm_head_accept),
    }
    failed = []
    for name, fn in checks.items():
        try:
            fn()
        except (AssertionError, IndexError, ValueError, FloatingPointError):
            failed.append(name)
    return failed


MUTATIONS = [
    # Eq. 2 read with floor() instead of ceil() for beta
    ("return -((-t) // B)", "return t // B"),
    # clean causal without the diagonal
    ("(i <= L) & (j <= L) & (j <= i)", "(i <= L) & (j <= L) & (j < i)"),
    # bidirectional placeholders inside a block (Block Diffusion)
    ("(block_index(i - L, B) == block_index(j - L, B)) & (j <= i)",
     "(block_index(i - L, B) == block_index(j - L, B))"),
    # noisy block also sees the clean tokens of its own block
    ("block_index(j, B) < block_index(i - L, B)", "block_index(j, B) <= block_index(i - L, B)"),
    # wrong GQA mapping (interleaved instead of contiguous groups)
    ("            g = h // group\n            scores = scale * (q[b, rows, h, :]",
     "            g = h % hkv\n            scores = scale * (q[b, rows, h, :]"),
    # scale dropped in the training forward
    ("scores = scale * (q[b, rows, h, :] @ k[b, :, g, :].T)", "scores = (q[b, rows, h, :] @ k[b, :, g, :].T)"),
    # K used as V in the training forward (transposed operands)
    ("_softmax_attend(scores, visible, v[b, :, g, :])", "_softmax_attend(scores, visible, k[b, :, g, :])"),
    # placeholder does not see itself in decode
    ("visible[i, n + i + 1:] = False", "visible[i, n + i:] = False"),
    # placeholders see each other bidirectionally in decode
    ("visible[i, n + i + 1:] = False", "pass"),
    # decode reads the wrong KV head
    ("            g = h // group\n            keys = np.concatenate([k_cache[b, g, :n, :], k_new[b, :, g, :]]",
     "            g = 0\n            keys = np.concatenate([k_cache[b, g, :n, :], k_new[b, :, g, :]]"),
    # deferred decode reads the wrong KV head
    ("            g = h // group\n            keys = np.concatenate([k_cache[b, g, :n, :], k_new[b, slots, g, :]]",
     "            g = 0\n            keys = np.concatenate([k_cache[b, g, :n, :], k_new[b, slots, g, :]]"),
    # argmax ties go to the last index
    ("tok = int(np.flatnonzero(row == m)[0])", "tok = int(np.flatnonzero(row == m)[-1])"),
    # confidence taken as the sum instead of its inverse
    ("conf[r] = 1.0 / np.exp(row - m).sum()", "conf[r] = np.exp(row - m).sum() / row.size"),
    # margin: the top token is not removed before taking the runner-up (always 0)
    ("others = np.delete(p, tok)", "others = p"),
    # margin: the smallest other probability instead of the largest
    ("conf[r] = p[tok] - (others.max() if others.size else 0.0)",
     "conf[r] = p[tok] - (others.min() if others.size else 0.0)"),
    # margin: runner-up of a one-token vocabulary taken as p1 (margin 0 instead of 1)
    ("(others.max() if others.size else 0.0)", "(others.max() if others.size else p[tok])"),
    # margin: unnormalised (logit-domain) difference
    ("            p /= p.sum()\n", ""),
    # deferred: the masks do not see the pending rows
    ("        slots = list(range(p)) + list(range(B, 2 * B))  # valid slots in position order",
     "        slots = list(range(B, 2 * B)) + list(range(p))"),
    # deferred: invalid pending slots treated as valid
    ("list(range(p)) + list(range(B, 2 * B))", "list(range(2 * B))"),
    # deferred: pending rows written one slot too far
    ("            kc[b, g, n:n + p, :] = k_new[b, :p, g, :]", "            kc[b, g, n + 1:n + p + 1, :] = k_new[b, :p, g, :]"),
    # deferred acceptance advancing by the new count instead of the pending one
    ("np.asarray(cache_len, dtype=np.int64) + np.asarray(pending, dtype=np.int64)",
     "np.asarray(cache_len, dtype=np.int64) + n"),
    # backward: the softmax Jacobian without its row-sum term
    ("            ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))", "            ds = p * dp"),
    # backward: dQ without the scale
    ("            dq[b, :, h, :] = scale * (ds @ k[b, :, g, :])", "            dq[b, :, h, :] = ds @ k[b, :, g, :]"),
    # backward: dV from P instead of its transpose
    ("            dv[b, :, g, :] += p.T @ do[b, :, h, :]", "            dv[b, :, g, :] += p @ do[b, :, h, :]"),
    # backward: GQA heads overwrite instead of adding into dK
    ("            dk[b, :, g, :] += scale * (ds.T @ q[b, :, h, :])", "            dk[b, :, g, :] = scale * (ds.T @ q[b, :, h, :])"),
    # backward: dP against K instead of V
    ("            dp = do[b, :, h, :] @ v[b, :, g, :].T", "            dp = do[b, :, h, :] @ k[b, :, g, :].T"),
    # batch-minimum mode taking the maximum
    ("n = np.full_like(n, n.min())", "n = np.full_like(n, n.max())"),
    # strict > instead of >= tau
    ("if c >= tau:", "if c > tau:"),
    # the at-least-one rule dropped
    ("return max(n, 1)", "return n"),
    # confident later positions counted (no early stop)
    ("        else:\n            break\n", "        else:\n            pass\n"),
    # append one slot too far
    ("kc[b, :, ln[b] + i, :] = k_new[b, i, :, :]", "kc[b, :, ln[b] + i + 1, :] = k_new[b, i, :, :]"),
    # length not advanced
    ("ln[b] += n", "ln[b] += 0"),
    # LM head: the weight used untransposed (columns as vocabulary rows)
    ("np.asarray(weight, dtype=np.float64).T", "np.asarray(weight, dtype=np.float64)"),
    # LM head: the acceptance reads the hidden states instead of the logits
    ("return accept(lm_head_logits(hidden, weight), tau)", "return accept(np.asarray(hidden, dtype=np.float64), tau)"),
]


@pytest.mark.parametrize("old,new", MUTATIONS, ids=[f"m{i}" for i in range(len(MUTATIONS))])
def test_mutant_is_caught(old, new):
    failed = all_pins(mutant(old, new))
    assert failed, f"no pin caught the mutation {old!r} -> {new!r}"


def test_unmutated_copy_passes_every_pin():
    assert all_pins(mutant("import numpy as np\n", "import numpy as np\n")) == []
