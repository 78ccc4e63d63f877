"""fp64 CPU oracle for the MARS hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The CUDA library never calls it, and it shares no code, header,
table or helper with the CUDA path: it is written directly from the method's
definition so that it can check the kernels.

Sources (cited by page title and section / equation):

* [paper]  "MARS: Enabling Autoregressive Models Multi-Token Generation"
  (arXiv 2604.07023), Sec. 3.2 Eq. 1 (concatenated input), Eq. 2 (attention
  mask), Fig. 2 (mask for L=8, B=4 and sliding-window inference), Sec. 3.1
  gap (4) (strictly left-to-right acceptance), Sec. 3.3 Eq. 4 (the 1/B ratio).
* [blog]   the authors' MARS blog post (xalp.net/posts/2026-06-mars), section
  "Inference: a knob, not a mode switch" (threshold tau, top-1 probability
  gate, block-level KV cache).
* [news]   "MARS: 자기회귀 모델의 멀티 토큰 생성을 가능하게 하는 기법"
  (aitrends.kr), inference paragraph (at least one token is always accepted).

Everything is float64.  bf16 inputs arrive as float64 arrays holding the
exactly widened bf16 values.

Readings taken where the pages are silent:

* softmax scale is a parameter (the kernels are called with 1/sqrt(D));
* GQA: query head h uses KV head h // (Hq // Hkv) (contiguous groups);
* L need not be a multiple of B: ceil() makes the last block short;
* confidence = top-1 softmax probability at temperature 1; a position passes
  when conf >= tau; ties in the argmax go to the lowest vocabulary index;
* the margin gate ([blog] "Inference": the top token's lead over the rest) is read
  as p1 - p2, the top-1 probability minus the largest probability of any
  other token;
* the block-level KV cache advances per sequence by that sequence's own
  commit count, or, in the batch-minimum mode of the paper's original
  sampler, every sequence by the smallest count of the batch.

Parity pins for every function live in ``tests/test_oracle_*.py``; no
function here is unpinned.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "block_index",
    "mask_rows",
    "mars_mask",
    "train_attn",
    "train_attn_bwd",
    "decode_attn",
    "decode_attn_deferred",
    "accept_rows",
    "commit_count",
    "accept",
    "append_kv",
    "accept_deferred",
    "lm_head_logits",
    "lm_head_accept",
    "near_threshold",
]


# --------------------------------------------------------------------------
# Eq. 2 of [paper]: the structured mask over z = [x ; x~]
# --------------------------------------------------------------------------

def block_index(t, B: int):
    """beta(t) = ceil(t / B) for 1-indexed position t within a stream ([paper] Sec. 3.2)."""
    t = np.asarray(t, dtype=np.int64)
    return -((-t) // B)


def mask_rows(L: int, B: int, rows) -> np.ndarray:
    """Rows of M (Eq. 2 of [paper]) as booleans, True where M_ij = 0.

    ``rows`` are 0-indexed query positions in z (0 .. 2L-1); the result has
    shape [len(rows), 2L].  The three cases are written in the paper's own
    1-indexed form: with i = row + 1 and j = col + 1,

      * clean causal:             i <= L, j <= L, j <= i
      * noisy intra-block causal: i > L, j > L, beta(i-L) == beta(j-L), j <= i
      * noisy -> clean:           i > L, j <= L, beta(j) < beta(i-L)

    and every other entry is -inf (False here).
    """
    i = np.asarray(rows, dtype=np.int64).reshape(-1, 1) + 1
    j = np.arange(1, 2 * L + 1, dtype=np.int64).reshape(1, -1)
    clean_causal = (i <= L) & (j <= L) & (j <= i)
    noisy_intra = (i > L) & (j > L) & (block_index(i - L, B) == block_index(j - L, B)) & (j <= i)
    noisy_to_clean = (i > L) & (j <= L) & (block_index(j, B) < block_index(i - L, B))
    return clean_causal | noisy_intra | noisy_to_clean


def mars_mask(L: int, B: int) -> np.ndarray:
    """The full 2L x 2L mask of Eq. 2 ([paper] Sec. 3.2), True = visible."""
    return mask_rows(L, B, np.arange(2 * L))


# --------------------------------------------------------------------------
# Masked attention over z ([paper] Sec. 3.2: both streams share one forward)
# --------------------------------------------------------------------------

def _softmax_attend(scores: np.ndarray, visible: np.ndarray, v: np.ndarray):
    """softmax(scores + M) @ v for one head; returns (out, natural-log lse).

    Masked entries are -inf; the row max is subtracted before exp.  Every row
    handed in here has at least one visible key.
    """
    s = np.where(visible, scores, -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    denom = e.sum(axis=1, keepdims=True)
    p = e / denom
    return p @ v, (m + np.log(denom))[:, 0]


def train_attn(q, k, v, L: int, B: int, scale: float, rows=None):
    """Attention over z = [x ; x~] under the MARS mask (Eqs. 1-2 of [paper]).

    q: [b, 2L, Hq, D]; k, v: [b, 2L, Hkv, D] (float64).  ``rows`` (optional)
    restricts the computation to those 0-indexed query positions.
    Returns (o [b, n_rows, Hq, D], lse [b, Hq, n_rows]) where lse is the
    natural-log log-sum-exp of the scaled, masked scores.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    nb, n2, hq, d = q.shape
    hkv = k.shape[2]
    assert n2 == 2 * L and k.shape == (nb, n2, hkv, d) and v.shape == k.shape
    assert hq % hkv == 0
    group = hq // hkv
    if rows is None:
        rows = np.arange(n2)
    rows = np.asarray(rows, dtype=np.int64)
    visible = mask_rows(L, B, rows)
    out = np.empty((nb, rows.size, hq, d), dtype=np.float64)
    lse = np.empty((nb, hq, rows.size), dtype=np.float64)
    for b in range(nb):
        for h in range(hq):
            g = h // group
            scores = scale * (q[b, rows, h, :] @ k[b, :, g, :].T)
            out[b, :, h, :], lse[b, h, :] = _softmax_attend(scores, visible, v[b, :, g, :])
    return out, lse


def train_attn_bwd(q, k, v, do, L: int, B: int, scale: float):
    """Gradients of the MARS masked attention (the forward of train_attn) with
    respect to q, k and v, given the output gradient do ([paper] Sec. 3.2: both
    streams share one forward, so one backward carries the gradients of
    Eqs. 3 and 5 to q, k and v).

    For one head, with S = scale * q k^T, P = softmax(S + M) over visible keys
    and O = P v, the gradients are the textbook ones:
        dV = P^T dO,   dP = dO v^T,
        dS = P * (dP - rowsum(P * dP))       (the softmax Jacobian, row by row),
        dQ = scale * dS k,   dK = scale * dS^T q.
    With GQA every query head of a group adds its dK and dV to the group's KV
    head.  q, do: [b, 2L, Hq, D]; k, v: [b, 2L, Hkv, D].
    Returns (dq [b, 2L, Hq, D], dk [b, 2L, Hkv, D], dv [b, 2L, Hkv, D]).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    nb, n2, hq, d = q.shape
    hkv = k.shape[2]
    assert n2 == 2 * L and k.shape == (nb, n2, hkv, d) and v.shape == k.shape and do.shape == q.shape
    group = hq // hkv
    visible = mars_mask(L, B)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(nb):
        for h in range(hq):
            g = h // group
            s = np.where(visible, scale * (q[b, :, h, :] @ k[b, :, g, :].T), -np.inf)
            e = np.exp(s - s.max(axis=1, keepdims=True))
            p = e / e.sum(axis=1, keepdims=True)
            dp = do[b, :, h, :] @ v[b, :, g, :].T
            ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dv[b, :, g, :] += p.T @ do[b, :, h, :]
            dq[b, :, h, :] = scale * (ds @ k[b, :, g, :])
            dk[b, :, g, :] += scale * (ds.T @ q[b, :, h, :])
    return dq, dk, dv


# --------------------------------------------------------------------------
# Sliding-window block decode ([paper] Fig. 2 right; [blog] "Inference")
# --------------------------------------------------------------------------

def decode_attn(q, k_new, v_new, k_cache, v_cache, cache_len, scale: float):
    """Attention of the B appended [MASK] queries of one decode step.

    q: [b, B, Hq, D]; k_new, v_new: [b, B, Hkv, D]; k_cache, v_cache:
    [b, Hkv, cap, D]; cache_len: [b].  Query i of sequence b sees all
    cache_len[b] committed keys and the new keys c <= i (causal among the
    placeholders, as in the noisy intra-block case of Eq. 2).
    Returns o [b, B, Hq, D].
    """
    q = np.asarray(q, dtype=np.float64)
    nb, bq, hq, d = q.shape
    hkv = k_new.shape[2]
    group = hq // hkv
    out = np.empty_like(q)
    for b in range(nb):
        n = int(cache_len[b])
        for h in range(hq):
            g = h // group
            keys = np.concatenate([k_cache[b, g, :n, :], k_new[b, :, g, :]], axis=0)
            vals = np.concatenate([v_cache[b, g, :n, :], v_new[b, :, g, :]], axis=0)
            visible = np.ones((bq, n + bq), dtype=bool)
            for i in range(bq):
                visible[i, n + i + 1:] = False
            scores = scale * (q[b, :, h, :] @ keys.T)
            out[b, :, h, :], _ = _softmax_attend(scores, visible, vals)
    return out


def decode_attn_deferred(q, k_new, v_new, k_cache, v_cache, cache_len, pending, scale: float):
    """One decode step of the deferred-KV sampler ([blog] "Inference": KV
    commitment deferred into the next proposal forward, per-sample cursors and
    a cache-validity bitmask).

    The forward of step t carries, per sequence b, 2B slots: slots 0..B-1 hold
    the tokens committed at step t-1 (valid while slot < pending[b]; their K/V
    are computed by this forward, so no extra forward recomputes them) and
    slots B..2B-1 the B new [MASK] placeholders.  q: [b, 2B, Hq, D]; k_new,
    v_new: [b, 2B, Hkv, D].  The valid slots follow the cache_len[b] committed
    cache rows in slot order; a valid query slot sees every cache row and the
    valid slots up to itself.  The valid pending rows are written into the cache
    at cache_len[b] .. cache_len[b] + pending[b] - 1 (cache_len itself is
    advanced by the acceptance step).

    Returns (o [b, 2B, Hq, D] with zero rows at invalid slots, k_cache', v_cache')
    where the caches are updated copies.
    """
    q = np.asarray(q, dtype=np.float64)
    nb, s2, hq, d = q.shape
    B = s2 // 2
    hkv = k_new.shape[2]
    group = hq // hkv
    out = np.zeros_like(q)
    kc = np.array(k_cache, dtype=np.float64, copy=True)
    vc = np.array(v_cache, dtype=np.float64, copy=True)
    for b in range(nb):
        n, p = int(cache_len[b]), int(pending[b])
        slots = list(range(p)) + list(range(B, 2 * B))  # valid slots in position order
        for g in range(hkv):
            kc[b, g, n:n + p, :] = k_new[b, :p, g, :]
            vc[b, g, n:n + p, :] = v_new[b, :p, g, :]
        for h in range(hq):
            g = h // group
            keys = np.concatenate([k_cache[b, g, :n, :], k_new[b, slots, g, :]], axis=0)
            vals = np.concatenate([v_cache[b, g, :n, :], v_new[b, slots, g, :]], axis=0)
            nq = len(slots)
            visible = np.ones((nq, n + nq), dtype=bool)
            for j in range(nq):
                visible[j, n + j + 1:] = False
            scores = scale * (q[b, slots, h, :] @ keys.T)
            out[b, slots, h, :], _ = _softmax_attend(scores, visible, vals)
    return out, kc, vc


def accept_deferred(logits, tau: float, cache_len, pending, gate: str = "prob"):
    """Acceptance step of the deferred-KV sampler: the same tokens, confidences
    and commit counts as accept(), but no K/V is copied; the cursor advances by
    the previous step's count (the rows the decode step just wrote) and the new
    count becomes the pending count of the next step.

    Returns (tokens, conf, n_new, cache_len') with cache_len' = cache_len + pending.
    """
    tokens, conf, n = accept(logits, tau, gate)
    return tokens, conf, n, np.asarray(cache_len, dtype=np.int64) + np.asarray(pending, dtype=np.int64)


# --------------------------------------------------------------------------
# Confidence-threshold acceptance ([blog] "Inference"; [paper] gap (4);
# [news] "at least one token")
# --------------------------------------------------------------------------

def accept_rows(logits, gate: str = "prob"):
    """Per proposal position: greedy token and its confidence.

    logits: [..., V] float64 (finite).  m = max_v l_v; token = the smallest v
    with l_v = m.  With gate "prob" the confidence is the top-1 probability
    1 / sum_v exp(l_v - m) = softmax(l)[token] at temperature 1 ([blog]
    "Inference").  With gate "margin" it is the top token's lead over the rest,
    read as p1 - p2: softmax(l)[token] minus the largest softmax(l)[v] over the
    other v (0 when two tokens tie at the max; p1 when V == 1).
    """
    assert gate in ("prob", "margin")
    x = np.asarray(logits, dtype=np.float64)
    assert np.all(np.isfinite(x)), "logits must be finite"
    flat = x.reshape(-1, x.shape[-1])
    tokens = np.empty(flat.shape[0], dtype=np.int64)
    conf = np.empty(flat.shape[0], dtype=np.float64)
    for r in range(flat.shape[0]):
        row = flat[r]
        m = row.max()
        tok = int(np.flatnonzero(row == m)[0])
        tokens[r] = tok
        if gate == "prob":
            conf[r] = 1.0 / np.exp(row - m).sum()
        else:
            p = np.exp(row - m)
            p /= p.sum()
            others = np.delete(p, tok)
            conf[r] = p[tok] - (others.max() if others.size else 0.0)
    return tokens.reshape(x.shape[:-1]), conf.reshape(x.shape[:-1])


def commit_count(conf_row, tau: float) -> int:
    """Left-to-right commit rule for one sequence.

    Walk the B proposals in order and stop at the first whose confidence is
    below tau; at least one token is always committed, so n = max(1, prefix).
    """
    n = 0
    for c in conf_row:
        if c >= tau:
            n += 1
        else:
            break
    return max(n, 1)


def accept(logits, tau: float, gate: str = "prob", batch_min: bool = False):
    """tokens [b, B], conf [b, B], n_commit [b] for logits [b, B, V] (gate: see accept_rows).

    batch_min: the paper's original sampler, whose block-level cache advanced at
    the batch-minimum acceptance ([blog] "Inference"): every sequence commits the
    smallest of the per-sequence counts.
    """
    tokens, conf = accept_rows(logits, gate)
    n = np.array([commit_count(conf[b], tau) for b in range(conf.shape[0])], dtype=np.int64)
    if batch_min:
        n = np.full_like(n, n.min())
    return tokens, conf, n


def lm_head_logits(hidden, weight):
    """Logits of the LM head for the proposal positions: logits[..., v] =
    sum_k hidden[..., k] * weight[v, k] (fp64), with weight in the [V, hidden]
    layout of the head's linear map.  The MARS blog post ("Where it stands
    against the alternatives") names this 152k-vocabulary projection as the
    drafter's cost; the acceptance step reads its output."""
    return np.asarray(hidden, dtype=np.float64) @ np.asarray(weight, dtype=np.float64).T


def lm_head_accept(hidden, weight, tau: float):
    """The LM head followed by the acceptance step, as one definition: the
    tokens, confidences and commit counts of accept() (top-1 probability gate)
    on lm_head_logits(hidden, weight).  hidden: [b, B, K]; weight: [V, K]."""
    return accept(lm_head_logits(hidden, weight), tau)


def append_kv(k_cache, v_cache, cache_len, k_new, v_new, n_commit):
    """Block-level KV cache append ([paper] contributions; [blog] "Inference").

    For each sequence b, rows 0..n_commit[b]-1 of k_new/v_new ([b, B, Hkv, D])
    are written at cache positions cache_len[b] + i of k_cache/v_cache
    ([b, Hkv, cap, D]); cache_len[b] then grows by n_commit[b].  Works on
    copies and returns (k_cache, v_cache, cache_len).
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    ln = np.array(cache_len, dtype=np.int64, copy=True)
    for b in range(kc.shape[0]):
        n = int(n_commit[b])
        for i in range(n):
            kc[b, :, ln[b] + i, :] = k_new[b, i, :, :]
            vc[b, :, ln[b] + i, :] = v_new[b, i, :, :]
        ln[b] += n
    return kc, vc, ln


def near_threshold(conf, tau: float, band: float = 1e-4) -> np.ndarray:
    """Positions whose fp64 confidence lies within ``band`` of tau.

    A commit decision at such a position may legitimately differ between an
    fp32 kernel and this fp64 oracle; parity reports them instead of failing.
    """
    return np.abs(np.asarray(conf, dtype=np.float64) - tau) < band
