"""Checks that pin the fp64 oracle to facts fixed outside itself.

Each ``check_*`` takes the oracle function(s) under test as arguments, so the
same check runs against the real oracle (tests/test_oracle_pins.py) and
against deliberately broken copies of it (tests/test_oracle_mutations.py),
which shows that a plausible mistake in the oracle fails at least one pin.

What the pins rest on (never on the oracle itself):

* the worked 16 x 16 mask of Fig. 2 (L=8, B=4), written out by hand in
  tests/golden/ from the caption of "MARS: Enabling Autoregressive Models
  Multi-Token Generation" and the three cases listed after its Eq. 2;
* an independent 0-indexed construction of the mask from the blocks, as the
  authors' blog post ("The construction, and the part that turned out to
  matter") describes it in words;
* the ratios the paper prints under Eq. 4 (25%, 12.5%, 6.25% for B = 4, 8, 16)
  and the Sec. 3.3 statement that in-block position t sees t-1 placeholders;
* textbook / library routines on special cases: torch's
  scaled_dot_product_attention (causal) for the clean half and for each
  noisy block, scipy's softmax / logsumexp, numpy's argmax;
* closed forms: one visible key gives that key's value; equal keys give the
  mean of the visible values; a one-hot logit row of height a has top-1
  probability 1 / (1 + (V-1) e^-a);
* the acceptance rules of the blog post ("Inference: a knob, not a mode
  switch"): stop at the first position below tau, tau = 1.0 is plain AR, and
  (aitrends.kr summary) at least one token is always committed.
"""

from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------
# helpers independent of the oracle
# --------------------------------------------------------------------------

def load_golden_mask(name="fig2_mask_L8_B4.txt"):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([c == "1" for c in line])
    return np.array(rows, dtype=bool)


def blocks_of(L, B):
    """0-indexed blocks of one stream: [start, stop) pairs; the last may be short."""
    return [(s, min(s + B, L)) for s in range(0, L, B)]


def mask_from_blocks(L, B):
    """Visibility built from the blocks in words, 0-indexed, without Eq. 2's ceil().

    The clean half is causal; a placeholder of noisy block k sees every clean
    token before the start of block k and the placeholders of its own block
    up to itself.
    """
    m = np.zeros((2 * L, 2 * L), dtype=bool)
    for i in range(L):
        m[i, : i + 1] = True
    for start, stop in blocks_of(L, B):
        for t in range(start, stop):
            m[L + t, :start] = True
            m[L + t, L + start: L + t + 1] = True
    return m


def sdpa_causal(q, k, v, scale):
    """torch's causal scaled-dot-product attention in float64 (one head).

    q: [n, D]; k, v: [n, D].  Query r sees keys 0..r.
    """
    import torch

    tq = torch.from_numpy(np.ascontiguousarray(q))[None, None]
    tk = torch.from_numpy(np.ascontiguousarray(k))[None, None]
    tv = torch.from_numpy(np.ascontiguousarray(v))[None, None]
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=scale)
    return out[0, 0].numpy()


def rand(shape, seed, sigma=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * sigma


# --------------------------------------------------------------------------
# mask pins
# --------------------------------------------------------------------------

def check_mask_golden(mars_mask):
    got = mars_mask(8, 4)
    want = load_golden_mask()
    assert got.shape == (16, 16)
    assert np.array_equal(got, want), "Eq. 2 mask differs from the hand-written Fig. 2 mask"


def check_mask_vs_blocks(mars_mask, Ls=(1, 2, 3, 5, 8, 10, 13, 16, 33), Bs=(1, 2, 3, 4, 5, 8, 16)):
    for L in Ls:
        for B in Bs:
            assert np.array_equal(mars_mask(L, B), mask_from_blocks(L, B)), (L, B)


def check_mask_pair_count(mars_mask):
    for L, B in [(64, 4), (37, 5), (16, 16), (20, 32)]:
        assert int(mars_mask(L, B).sum()) == L * (L + 1), (L, B)


def check_mask_not_bidirectional(mars_mask):
    """Block Diffusion's intra-block bidirectional mask is the contrast case (Fig. 2 caption)."""
    L, B = 8, 4
    m = mars_mask(L, B)
    for start, stop in blocks_of(L, B):
        for t in range(start, stop):
            for u in range(t + 1, stop):
                assert not m[L + t, L + u], "a placeholder sees a later placeholder"


def check_mask_eq4_ratio(mars_mask):
    """Eq. 4: the fraction of noisy positions with fully clean context is 1/B,
    printed as 25%, 12.5%, 6.25% for B = 4, 8, 16."""
    L = 64
    for B, printed in [(4, 0.25), (8, 0.125), (16, 0.0625)]:
        m = mars_mask(L, B)
        noisy_keys_seen = m[L:, L:].sum(axis=1)
        frac = np.mean(noisy_keys_seen == 1)
        assert frac == printed, (B, frac)


def check_mask_sec33_counts(mars_mask):
    """Sec. 3.3: in-block position t (1-indexed) sees t-1 placeholders besides
    itself plus the clean prefix of the earlier blocks."""
    L, B = 24, 8
    m = mars_mask(L, B)
    for k, (start, stop) in enumerate(blocks_of(L, B)):
        for t in range(start, stop):
            t1 = t - start + 1
            row = m[L + t]
            assert row[L:].sum() == t1
            assert row[:L].sum() == k * B
            assert row[: k * B].all()


# --------------------------------------------------------------------------
# training attention pins
# --------------------------------------------------------------------------

def check_train_clean_half_is_causal(train_attn):
    L, B, D = 24, 4, 16
    q, k, v = rand((1, 2 * L, 1, D), 1), rand((1, 2 * L, 1, D), 2), rand((1, 2 * L, 1, D), 3)
    scale = D ** -0.5
    o, _ = train_attn(q, k, v, L, B, scale)
    want = sdpa_causal(q[0, :L, 0], k[0, :L, 0], v[0, :L, 0], scale)
    assert np.max(np.abs(o[0, :L, 0] - want)) < 1e-12


def check_train_noisy_blocks_are_prefix_causal(train_attn, L=22, B=4, D=16):
    """Each noisy block equals causal attention over [clean tokens of earlier
    blocks ; that block's placeholders] (taking the block's rows)."""
    q, k, v = rand((1, 2 * L, 1, D), 4), rand((1, 2 * L, 1, D), 5), rand((1, 2 * L, 1, D), 6)
    scale = D ** -0.5
    o, _ = train_attn(q, k, v, L, B, scale)
    for start, stop in blocks_of(L, B):
        idx = list(range(start)) + [L + t for t in range(start, stop)]
        ref = sdpa_causal(q[0, idx, 0], k[0, idx, 0], v[0, idx, 0], scale)
        got = o[0, L + start: L + stop, 0]
        assert np.max(np.abs(got - ref[start:])) < 1e-12, (start, stop)


def check_train_single_key_rows(train_attn):
    """Clean position 0 and the first placeholder of block 1 see one key: out = v."""
    L, B, D = 12, 4, 8
    q, k, v = rand((2, 2 * L, 2, D), 7), rand((2, 2 * L, 1, D), 8), rand((2, 2 * L, 1, D), 9)
    o, _ = train_attn(q, k, v, L, B, 0.3)
    for b in range(2):
        for h in range(2):
            assert np.array_equal(o[b, 0, h], v[b, 0, 0])
            assert np.array_equal(o[b, L, h], v[b, L, 0])


def check_train_equal_keys_give_mean(train_attn):
    L, B, D = 14, 3, 8
    q = rand((1, 2 * L, 1, D), 10)
    k = np.tile(rand((1, 1, 1, D), 11), (1, 2 * L, 1, 1))
    v = rand((1, 2 * L, 1, D), 12)
    o, _ = train_attn(q, k, v, L, B, 0.5)
    vis = mask_from_blocks(L, B)
    for i in range(2 * L):
        want = v[0, vis[i], 0].mean(axis=0)
        assert np.max(np.abs(o[0, i, 0] - want)) < 1e-12


def check_train_bruteforce(train_attn):
    """Naive triple loop, no max subtraction, on tiny shapes (small scale keeps exp finite)."""
    L, B, D = 7, 3, 4
    q, k, v = rand((1, 2 * L, 2, D), 13), rand((1, 2 * L, 1, D), 14), rand((1, 2 * L, 1, D), 15)
    scale = 0.37
    vis = mask_from_blocks(L, B)
    o, lse = train_attn(q, k, v, L, B, scale)
    for h in range(2):
        for i in range(2 * L):
            num = np.zeros(D)
            den = 0.0
            for j in range(2 * L):
                if vis[i, j]:
                    w = np.exp(scale * sum(q[0, i, h, d] * k[0, j, 0, d] for d in range(D)))
                    num += w * v[0, j, 0]
                    den += w
            assert np.max(np.abs(o[0, i, h] - num / den)) < 1e-12
            assert abs(lse[0, h, i] - np.log(den)) < 1e-12


def check_train_lse(train_attn):
    from scipy.special import logsumexp

    L, B, D = 10, 4, 8
    q, k, v = rand((1, 2 * L, 1, D), 16), rand((1, 2 * L, 1, D), 17), rand((1, 2 * L, 1, D), 18)
    scale = D ** -0.5
    _, lse = train_attn(q, k, v, L, B, scale)
    vis = mask_from_blocks(L, B)
    s = scale * q[0, :, 0] @ k[0, :, 0].T
    for i in range(2 * L):
        assert abs(lse[0, 0, i] - logsumexp(s[i, vis[i]])) < 1e-12


def check_train_block_ge_L(train_attn):
    """B >= L: one noisy block, so placeholders see no clean token at all."""
    L, B, D = 9, 16, 8
    q, k, v = rand((1, 2 * L, 1, D), 19), rand((1, 2 * L, 1, D), 20), rand((1, 2 * L, 1, D), 21)
    scale = D ** -0.5
    o, _ = train_attn(q, k, v, L, B, scale)
    ref = sdpa_causal(q[0, L:, 0], k[0, L:, 0], v[0, L:, 0], scale)
    assert np.max(np.abs(o[0, L:, 0] - ref)) < 1e-12


# --------------------------------------------------------------------------
# training attention backward pins
# --------------------------------------------------------------------------

def _autograd_bwd(q, k, v, do, L, B, scale):
    """dq, dk, dv of sum(O * dO) by torch autograd (float64) through a dense
    attention whose mask is the block construction above (not Eq. 2's cases)."""
    import torch

    nb, n2, hq, d = q.shape
    hkv = k.shape[2]
    group = hq // hkv
    allowed = torch.from_numpy(mask_from_blocks(L, B))
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    loss = 0.0
    for b in range(nb):
        for h in range(hq):
            g = h // group
            s = (tq[b, :, h, :] @ tk[b, :, g, :].T) * scale
            p = torch.softmax(s.masked_fill(~allowed, float("-inf")), dim=1)
            loss = loss + ((p @ tv[b, :, g, :]) * torch.from_numpy(do[b, :, h, :])).sum()
    loss.backward()
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


def check_bwd_vs_autograd(train_attn_bwd):
    for (nb, L, B, hq, hkv, d) in [(2, 12, 3, 4, 2, 8), (1, 13, 4, 3, 1, 6), (1, 7, 8, 2, 2, 4)]:
        q, k, v = rand((nb, 2 * L, hq, d), 60), rand((nb, 2 * L, hkv, d), 61), rand((nb, 2 * L, hkv, d), 62)
        do = rand((nb, 2 * L, hq, d), 63)
        scale = d ** -0.5
        got = train_attn_bwd(q, k, v, do, L, B, scale)
        want = _autograd_bwd(q, k, v, do, L, B, scale)
        for g_, w_ in zip(got, want):
            assert np.max(np.abs(g_ - w_)) < 1e-11, np.max(np.abs(g_ - w_))


def check_bwd_finite_differences(train_attn_bwd, train_attn):
    """Central differences of sum(O * dO) through the (independently pinned) forward."""
    L, B, d = 5, 2, 4
    q, k, v = rand((1, 2 * L, 2, d), 64), rand((1, 2 * L, 1, d), 65), rand((1, 2 * L, 1, d), 66)
    do = rand((1, 2 * L, 2, d), 67)
    scale = 0.7
    dq, dk, dv = train_attn_bwd(q, k, v, do, L, B, scale)
    f = lambda q_, k_, v_: float(np.sum(train_attn(q_, k_, v_, L, B, scale)[0] * do))  # noqa: E731
    eps = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        base = [q, k, v]
        x = base[which]
        for idx in [(0, 0, 0, 0), (0, 3, 0, 1), (0, 2 * L - 1, 0, 3), (0, L + 1, 0, 2), (0, L - 1, 0, 0)]:
            if idx[2] >= x.shape[2]:
                continue
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p, args_m = list(base), list(base)
            args_p[which], args_m[which] = xp, xm
            fd = (f(*args_p) - f(*args_m)) / (2 * eps)
            assert abs(fd - grad[idx]) < 1e-7, (which, idx, fd, grad[idx])


def check_bwd_gqa_is_repeat_kv(train_attn_bwd):
    """dK, dV of a KV head are the sums over its query heads of the per-head gradients."""
    L, B, d, hq, hkv = 9, 3, 8, 6, 2
    q, k, v = rand((1, 2 * L, hq, d), 68), rand((1, 2 * L, hkv, d), 69), rand((1, 2 * L, hkv, d), 70)
    do = rand((1, 2 * L, hq, d), 71)
    dq, dk, dv = train_attn_bwd(q, k, v, do, L, B, 0.4)
    kr, vr = np.repeat(k, hq // hkv, axis=2), np.repeat(v, hq // hkv, axis=2)
    dq2, dk2, dv2 = train_attn_bwd(q, kr, vr, do, L, B, 0.4)
    assert np.max(np.abs(dq - dq2)) < 1e-12
    assert np.max(np.abs(dk - dk2.reshape(1, 2 * L, hkv, hq // hkv, d).sum(axis=3))) < 1e-12
    assert np.max(np.abs(dv - dv2.reshape(1, 2 * L, hkv, hq // hkv, d).sum(axis=3))) < 1e-12


def check_bwd_closed_forms(train_attn_bwd):
    """Each row of P sums to 1, so the keys' dV rows sum to the rows of dO; a query
    that sees a single key (z position 0, and the first placeholder of block 1) has
    an all-zero softmax Jacobian, so its dQ row is exactly zero."""
    L, B, d = 10, 4, 8
    q, k, v = rand((2, 2 * L, 2, d), 72), rand((2, 2 * L, 1, d), 73), rand((2, 2 * L, 1, d), 74)
    do = rand((2, 2 * L, 2, d), 75)
    dq, dk, dv = train_attn_bwd(q, k, v, do, L, B, 0.35)
    assert np.max(np.abs(dv.sum(axis=1)[:, 0, :] - do.sum(axis=(1, 2)))) < 1e-12
    assert np.all(dq[:, 0] == 0) and np.all(dq[:, L] == 0)
    assert np.all(dq[:, 1] != 0)


def check_train_gqa_is_repeat_kv(train_attn):
    """Query head h uses KV head h // (Hq/Hkv): same as repeating each KV head
    Hq/Hkv times in a row (the Hugging Face repeat_kv layout)."""
    L, B, D, hq, hkv = 10, 4, 8, 6, 2
    q, k, v = rand((2, 2 * L, hq, D), 22), rand((2, 2 * L, hkv, D), 23), rand((2, 2 * L, hkv, D), 24)
    o1, l1 = train_attn(q, k, v, L, B, 0.3)
    o2, l2 = train_attn(q, np.repeat(k, hq // hkv, axis=2), np.repeat(v, hq // hkv, axis=2), L, B, 0.3)
    assert np.max(np.abs(o1 - o2)) < 1e-13 and np.max(np.abs(l1 - l2)) < 1e-13
    # and a hand-picked head: head 4 of 6 with 2 KV heads must read KV head 1
    o3, _ = train_attn(q[:, :, 4:5], k[:, :, 1:2], v[:, :, 1:2], L, B, 0.3)
    assert np.max(np.abs(o1[:, :, 4] - o3[:, :, 0])) < 1e-13


def check_train_rows_subset(train_attn):
    L, B, D = 12, 4, 8
    q, k, v = rand((1, 2 * L, 2, D), 25), rand((1, 2 * L, 1, D), 26), rand((1, 2 * L, 1, D), 27)
    o, lse = train_attn(q, k, v, L, B, 0.4)
    rows = np.array([0, 5, 11, 12, 19, 23])
    o2, lse2 = train_attn(q, k, v, L, B, 0.4, rows=rows)
    assert np.max(np.abs(o[:, rows] - o2)) < 1e-13
    assert np.max(np.abs(lse[:, :, rows] - lse2)) < 1e-13


# --------------------------------------------------------------------------
# decode attention pins
# --------------------------------------------------------------------------

def check_decode_matches_train_block(decode_attn, train_attn):
    """A decode step over cache = clean K/V of blocks < k and new = placeholders
    of block k reproduces noisy block k of the training forward."""
    L, B, D, hq, hkv = 20, 4, 8, 4, 2
    q, k, v = rand((1, 2 * L, hq, D), 28), rand((1, 2 * L, hkv, D), 29), rand((1, 2 * L, hkv, D), 30)
    scale = D ** -0.5
    o_train, _ = train_attn(q, k, v, L, B, scale)
    cap = L
    for kb in range(L // B):
        n = kb * B
        kc = np.zeros((1, hkv, cap, D))
        vc = np.zeros((1, hkv, cap, D))
        kc[0, :, :n] = k[0, :n].transpose(1, 0, 2)
        vc[0, :, :n] = v[0, :n].transpose(1, 0, 2)
        rows = slice(L + n, L + n + B)
        o = decode_attn(q[:, rows], k[:, rows], v[:, rows], kc, vc, np.array([n]), scale)
        assert np.max(np.abs(o - o_train[:, rows])) < 1e-12, kb


def check_decode_empty_cache_is_causal(decode_attn):
    B, D = 6, 8
    q, kn, vn = rand((1, B, 1, D), 31), rand((1, B, 1, D), 32), rand((1, B, 1, D), 33)
    kc = np.zeros((1, 1, 4, D))
    o = decode_attn(q, kn, vn, kc, kc, np.array([0]), 0.5)
    ref = sdpa_causal(q[0, :, 0], kn[0, :, 0], vn[0, :, 0], 0.5)
    assert np.max(np.abs(o[0, :, 0] - ref)) < 1e-12


def check_decode_bruteforce(decode_attn):
    """Per-sequence varlen cache, GQA, loop form."""
    nb, B, D, hq, hkv, cap = 3, 3, 4, 4, 2, 9
    q = rand((nb, B, hq, D), 34)
    kn, vn = rand((nb, B, hkv, D), 35), rand((nb, B, hkv, D), 36)
    kc, vc = rand((nb, hkv, cap, D), 37), rand((nb, hkv, cap, D), 38)
    lens = np.array([0, 5, 9])
    scale = 0.6
    o = decode_attn(q, kn, vn, kc, vc, lens, scale)
    for b in range(nb):
        for h in range(hq):
            g = h // (hq // hkv)
            for i in range(B):
                keys = [kc[b, g, j] for j in range(lens[b])] + [kn[b, c, g] for c in range(i + 1)]
                vals = [vc[b, g, j] for j in range(lens[b])] + [vn[b, c, g] for c in range(i + 1)]
                w = np.array([np.exp(scale * np.dot(q[b, i, h], kk)) for kk in keys])
                want = (w[:, None] * np.array(vals)).sum(axis=0) / w.sum()
                assert np.max(np.abs(o[b, i, h] - want)) < 1e-12


# --------------------------------------------------------------------------
# acceptance pins
# --------------------------------------------------------------------------

def check_accept_one_hot_closed_form(accept_rows):
    V = 1000
    for a, j in [(8.0, 17), (3.0, 999), (0.5, 0), (30.0, 512)]:
        row = np.zeros(V)
        row[j] = a
        tok, conf = accept_rows(row[None, None, :])
        assert tok[0, 0] == j
        assert abs(conf[0, 0] - 1.0 / (1.0 + (V - 1) * np.exp(-a))) < 1e-13  # V-term fp64 sum


def check_accept_ties_lowest_index(accept_rows):
    row = np.zeros((1, 1, 50))
    tok, conf = accept_rows(row)
    assert tok[0, 0] == 0 and abs(conf[0, 0] - 1 / 50) < 1e-16
    row[0, 0, [7, 31, 44]] = 2.5
    tok, _ = accept_rows(row)
    assert tok[0, 0] == 7
    row[0, 0, 3] = -1.0
    row[0, 0, 44] = 2.5
    tok, _ = accept_rows(row)
    assert tok[0, 0] == 7


def check_accept_vs_library(accept_rows):
    from scipy.special import softmax

    x = rand((3, 5, 777), 39, sigma=3.0)
    x = np.round(x * 4) / 4  # coarse grid: ties at the max happen
    tok, conf = accept_rows(x)
    for b in range(3):
        for i in range(5):
            assert tok[b, i] == int(np.argmax(x[b, i]))
            assert abs(conf[b, i] - softmax(x[b, i]).max()) < 1e-12


def check_margin_closed_forms(accept_rows):
    """Margin gate p1 - p2: closed forms on rows whose softmax is known by hand."""
    # V = 2: p1 - p2 = tanh(|l1 - l2| / 2)
    for a, b in [(1.0, 0.0), (0.0, 3.5), (-2.0, -2.25), (7.0, 7.0)]:
        tok, conf = accept_rows(np.array([[[a, b]]]), "margin")
        assert tok[0, 0] == (0 if a >= b else 1)
        assert abs(conf[0, 0] - np.tanh(abs(a - b) / 2)) < 1e-15
    # one spike of height x over V - 1 zeros: (e^x - 1) / (e^x + V - 1)
    V = 1000
    for x, j in [(8.0, 17), (3.0, 999), (0.5, 0)]:
        row = np.zeros(V)
        row[j] = x
        tok, conf = accept_rows(row[None, None, :], "margin")
        assert tok[0, 0] == j
        assert abs(conf[0, 0] - np.expm1(x) / (np.exp(x) + V - 1)) < 1e-13
    # two tokens tie at the max: zero margin; a single token: margin 1
    row = np.zeros((1, 1, 64))
    row[0, 0, [5, 40]] = 3.0
    _, conf = accept_rows(row, "margin")
    assert conf[0, 0] == 0.0
    _, conf = accept_rows(np.array([[[1.5]]]), "margin")
    assert conf[0, 0] == 1.0


def check_margin_vs_library(accept_rows):
    """Margin gate against scipy's softmax sorted by numpy, and its bounds."""
    from scipy.special import softmax

    x = rand((3, 5, 501), 45, sigma=2.0)
    x = np.round(x * 4) / 4  # coarse grid: ties at the max happen
    tok_p, p1 = accept_rows(x, "prob")
    tok, conf = accept_rows(x, "margin")
    assert np.array_equal(tok, tok_p)
    for b in range(3):
        for i in range(5):
            top = np.sort(softmax(x[b, i]))[::-1]
            assert abs(conf[b, i] - (top[0] - top[1])) < 1e-12
    assert np.all(conf <= p1 + 1e-15) and np.all(conf >= 2 * p1 - 1 - 1e-15) and np.all(conf >= 0)


def check_commit_rule(commit_count):
    assert commit_count([0.5, 0.99, 0.99, 0.99], 0.9) == 1      # first below tau: still one token
    assert commit_count([0.99, 0.99, 0.5, 0.99], 0.9) == 2      # stop at the first below tau
    assert commit_count([0.99, 0.95, 0.96, 0.999], 0.95) == 4   # conf == tau passes
    assert commit_count([0.2, 0.3, 0.1], 0.0) == 3              # tau = 0 commits all B
    assert commit_count([0.999999, 0.9999999], 1.0) == 1        # tau = 1.0 is plain AR
    assert commit_count([0.3, 0.95, 0.97, 0.2], 0.9) == 1       # confident later positions never count
    assert commit_count([0.91], 0.9) == 1


def check_accept_tau_extremes(accept):
    x = rand((4, 6, 300), 40, sigma=2.0)
    x[1, :, 5] += 20.0
    tok, conf, n = accept(x, 1.0)
    assert np.all(n == 1)
    tok, conf, n = accept(x, float(conf.max()) + 1e-9)
    assert np.all(n == 1)
    tok, conf, n = accept(x, 0.0)
    assert np.all(n == 6)


def check_batch_min(accept):
    """Batch-minimum mode: every sequence commits the smallest per-sequence count."""
    x = np.full((3, 4, 10), -5.0)
    x[:, :, 0] = 5.0               # confident everywhere: conf = 1 / (1 + 9 e^-10) ~ 0.9996
    x[1, 2, 0] = -5.0              # sequence 1: position 2 is uniform (conf 0.1)
    x[2, 0, 0] = -5.0              # sequence 2: position 0 uniform -> at least one still commits
    _, _, n = accept(x, 0.9)
    assert list(n) == [4, 2, 1]
    _, _, n = accept(x, 0.9, batch_min=True)
    assert list(n) == [1, 1, 1]
    _, _, n = accept(x[:2], 0.9, batch_min=True)
    assert list(n) == [2, 2]
    _, _, n = accept(x[:1], 0.9, batch_min=True)
    assert list(n) == [4]


def _deferred_case(seed, nb=3, B=4, hq=4, hkv=2, D=8, cap=40):
    q = rand((nb, 2 * B, hq, D), seed)
    kn, vn = rand((nb, 2 * B, hkv, D), seed + 1), rand((nb, 2 * B, hkv, D), seed + 2)
    kc, vc = rand((nb, hkv, cap, D), seed + 3), rand((nb, hkv, cap, D), seed + 4)
    return q, kn, vn, kc, vc


def check_deferred_matches_append_then_decode(decode_attn_deferred, decode_attn, append_kv):
    """Deferred step = (append the pending rows, then an ordinary decode step of the masks)
    for the mask slots; the cache ends with the pending rows written."""
    B = 4
    q, kn, vn, kc, vc = _deferred_case(46, B=B)
    lens, pend = np.array([5, 0, 11]), np.array([2, 4, 0])
    o, kc2, vc2 = decode_attn_deferred(q, kn, vn, kc, vc, lens, pend, 0.35)
    kc_a, vc_a, len_a = append_kv(kc, vc, lens, kn[:, :B], vn[:, :B], pend)
    o_ref = decode_attn(q[:, B:], kn[:, B:], vn[:, B:], kc_a, vc_a, len_a, 0.35)
    assert np.allclose(o[:, B:], o_ref, rtol=0, atol=1e-13)
    assert np.array_equal(kc2, kc_a) and np.array_equal(vc2, vc_a)


def check_deferred_pending_rows_are_causal(decode_attn_deferred, train_attn):
    """With an empty cache the valid pending slots are plain causal attention over
    themselves: the clean half of training attention for L = pending."""
    B, p = 4, 3
    q, kn, vn, kc, vc = _deferred_case(47, nb=1, B=B, hq=2, hkv=1)
    o, _, _ = decode_attn_deferred(q, kn, vn, kc, vc, np.array([0]), np.array([p]), 0.5)
    zq = np.concatenate([q[:, :p], q[:, :p]], axis=1)     # [x ; x~] with x~ unused here
    zk = np.concatenate([kn[:, :p], kn[:, :p]], axis=1)
    zv = np.concatenate([vn[:, :p], vn[:, :p]], axis=1)
    ot, _ = train_attn(zq, zk, zv, p, 1, 0.5, rows=range(p))
    assert np.allclose(o[:, :p], ot[:, :p], rtol=0, atol=1e-13)


def check_deferred_invalid_slots(decode_attn_deferred):
    """Invalid pending slots give zero rows and never reach a valid row, even as NaN."""
    B = 4
    q, kn, vn, kc, vc = _deferred_case(48, B=B)
    lens, pend = np.array([3, 7, 1]), np.array([1, 0, 3])
    o1, _, _ = decode_attn_deferred(q, kn, vn, kc, vc, lens, pend, 0.35)
    for b, p in enumerate(pend):
        q[b, p:B] = np.nan
        kn[b, p:B] = np.nan
        vn[b, p:B] = np.nan
    o2, kc2, _ = decode_attn_deferred(q, kn, vn, kc, vc, lens, pend, 0.35)
    assert np.array_equal(o1, o2) and np.all(np.isfinite(kc2))
    for b, p in enumerate(pend):
        assert np.all(o2[b, p:B] == 0)


def check_accept_deferred(accept_deferred, accept):
    x = rand((3, 4, 50), 49, sigma=3.0)
    tok, conf, n, ln = accept_deferred(x, 0.5, np.array([4, 0, 9]), np.array([2, 0, 3]))
    t2, c2, n2 = accept(x, 0.5)
    assert np.array_equal(tok, t2) and np.array_equal(conf, c2) and np.array_equal(n, n2)
    assert list(ln) == [6, 0, 12]


def check_append(append_kv):
    nb, B, hkv, D, cap = 3, 4, 2, 5, 12
    kc, vc = rand((nb, hkv, cap, D), 41), rand((nb, hkv, cap, D), 42)
    kn, vn = rand((nb, B, hkv, D), 43), rand((nb, B, hkv, D), 44)
    lens = np.array([0, 3, 8])
    n = np.array([1, 4, 2])
    kc2, vc2, lens2 = append_kv(kc, vc, lens, kn, vn, n)
    assert np.array_equal(lens2, lens + n)
    for b in range(nb):
        for g in range(hkv):
            for p in range(cap):
                if lens[b] <= p < lens[b] + n[b]:
                    assert np.array_equal(kc2[b, g, p], kn[b, p - lens[b], g])
                    assert np.array_equal(vc2[b, g, p], vn[b, p - lens[b], g])
                else:
                    assert np.array_equal(kc2[b, g, p], kc[b, g, p])
                    assert np.array_equal(vc2[b, g, p], vc[b, g, p])


# --------------------------------------------------------------------------
# LM head fused with acceptance
# --------------------------------------------------------------------------

def check_lm_head_logits_bruteforce(lm_head_logits):
    """Every logit is the dot product of a hidden row with a weight row, written as loops."""
    h = rand((2, 3, 5), 71)
    w = rand((7, 5), 72)
    got = lm_head_logits(h, w)
    assert got.shape == (2, 3, 7)
    for b in range(2):
        for i in range(3):
            for v in range(7):
                want = 0.0
                for k in range(5):
                    want += h[b, i, k] * w[v, k]
                assert abs(got[b, i, v] - want) < 1e-12


def check_lm_head_logits_one_hot(lm_head_logits):
    """A one-hot hidden row e_j reads column j of the weight: logits[v] = weight[v, j]."""
    w = rand((9, 9), 73)  # square, so a transposed weight would still have the right shape
    for j in (0, 4, 8):
        h = np.zeros((1, 1, 9))
        h[0, 0, j] = 1.0
        assert np.array_equal(lm_head_logits(h, w)[0, 0], w[:, j])


def check_lm_head_accept_closed_form(lm_head_accept):
    """Weight row t = a h / |h|^2 and every other row orthogonal to h: the logits are a
    at t and 0 elsewhere, so the token is t and conf = 1 / (1 + (V - 1) e^-a)."""
    K, V = 16, 40
    g = np.random.default_rng(74)
    for a, t in [(6.0, 3), (0.7, 0), (12.0, 39)]:
        h = g.standard_normal(K)
        w = g.standard_normal((V, K))
        w -= np.outer(w @ h, h) / (h @ h)  # every row orthogonal to h
        w[t] = a * h / (h @ h)
        tok, conf, n = lm_head_accept(h[None, None, :], w, 0.0)
        assert tok[0, 0] == t
        assert abs(conf[0, 0] - 1.0 / (1.0 + (V - 1) * np.exp(-a))) < 1e-12
        assert n[0] == 1
