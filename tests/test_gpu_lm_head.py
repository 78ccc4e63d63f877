"""mars_lm_head_accept (the LM head fused with the acceptance step) on the GPU
against the fp64 oracle (oracle.lm_head_accept: logits = hidden . weight^T, then
the top-1 probability gate, the left-to-right commit rule and the append).

Tolerances.  The kernel's logits are tensor-core fp32 sums of exact bf16 x bf16
products, K of them (3584 at the 7B width).  The accumulation's rounding error
grows with K: about K * 2^-24 times the size of the partial sums, i.e. up to
~1e-4 absolute for logits of a few units here (measured: conf within 1.3e-4
relative of fp64 at K = 3584).  The top-1 probability, a smooth function of the
logit differences, is held to 1e-3 relative; the argmax is bit-exact except on
rows whose two largest fp64 logits are closer than 1e-3 (ten times that error),
which are reported; commit counts are bit-exact unless the first differing
pass/fail decision has an fp64 confidence within 1e-3 of tau (reported).
Appended cache rows are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import token_decoding_gb300 as mars
from token_decoding_gb300 import synth
from tests.gpu_util import bits_of, dev_bf16

pytestmark = pytest.mark.gpu

CONF_REL = 1e-3
TIE_GAP = 1e-3
TAU_BAND = 1e-3


def head_inputs(batch, B, K, V, seed, spike_rows=0, spike=12.0):
    """hidden ~ N(0, 1); weight ~ N(0, 1) * 2 / sqrt(K) (logits ~ N(0, 4)).  For the
    first `spike_rows` rows a distinct vocabulary row is aligned with the row's
    hidden state, so that row's logit there is about `spike` (confident rows)."""
    g = synth.rng_for("lm_head", seed)
    h = g.standard_normal((batch, B, K), dtype=np.float32)
    w = g.standard_normal((V, K), dtype=np.float32) * np.float32(2.0 / np.sqrt(K))
    rows = h.reshape(-1, K)
    for r in range(min(spike_rows, rows.shape[0])):
        t = int(g.integers(0, V))
        w[t] = rows[r] * np.float32(spike / float(rows[r] @ rows[r]))
    return synth.Bf16.from_float(h), synth.Bf16.from_float(w)


def kv_for(batch, B, hkv, D, cap, seed):
    g = np.random.default_rng(seed)
    mk = lambda shape: synth.Bf16.from_float(g.standard_normal(shape, dtype=np.float32))  # noqa: E731
    return mk((batch, B, hkv, D)), mk((batch, B, hkv, D)), mk((batch, hkv, cap, D)), mk((batch, hkv, cap, D))


def oracle_chunked(h64, w64, tau, chunk=8192):
    """oracle.lm_head_logits over vocabulary chunks (bounded host memory), then the
    oracle's acceptance on the assembled logits."""
    V = w64.shape[0]
    logits = np.concatenate([oracle.lm_head_logits(h64, w64[v:v + chunk]) for v in range(0, V, chunk)], axis=-1)
    tok, conf, n = oracle.accept(logits, tau)
    return tok, conf, n, logits


def run_case(batch, B, K, V, tau, seed, spike_rows=0, hkv=2, D=64, cap=48, lens=None):
    h, w = head_inputs(batch, B, K, V, seed, spike_rows)
    kn, vn, kc, vc = kv_for(batch, B, hkv, D, cap, seed + 1)
    lens = np.zeros(batch, dtype=np.int32) if lens is None else np.asarray(lens, dtype=np.int32)
    d_kc, d_vc = dev_bf16(kc), dev_bf16(vc)
    d_len = torch.from_numpy(lens.copy()).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tok, conf, n = mars.lm_head_accept(dev_bf16(h), dev_bf16(w), tau, dev_bf16(kn), dev_bf16(vn), d_kc, d_vc, d_len,
                                       status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    tok, conf, n = tok.cpu().numpy(), conf.cpu().numpy().astype(np.float64), n.cpu().numpy()
    t_o, c_o, n_o, logits = oracle_chunked(h.f64, w.f64, tau)
    # argmax: exact except near ties of the fp64 logits
    top2 = np.sort(logits, axis=-1)[..., -2:] if V > 1 else np.concatenate([logits, logits - np.inf], -1)
    gap = top2[..., 1] - top2[..., 0]
    ties = []
    for b in range(batch):
        for i in range(B):
            if tok[b, i] != t_o[b, i]:
                assert gap[b, i] < TIE_GAP, (b, i, tok[b, i], t_o[b, i], gap[b, i])
                ties.append((b, i))
    ok = np.ones_like(tok, dtype=bool)
    for b, i in ties:
        ok[b, i] = False
    rel = np.abs(conf - c_o) / c_o
    assert float(rel[ok].max()) < CONF_REL, float(rel[ok].max())
    # commit counts: exact unless the first differing decision is within the band
    report = []
    for b in range(batch):
        if int(n[b]) == int(n_o[b]):
            continue
        diff = np.flatnonzero((conf[b].astype(np.float32) >= np.float32(tau)) != (c_o[b] >= tau))
        assert diff.size > 0 and abs(c_o[b, diff[0]] - tau) < TAU_BAND, (b, n[b], n_o[b])
        report.append((b, int(diff[0])))
    kc_o, vc_o, len_o = oracle.append_kv(kc.bits, vc.bits, lens, kn.bits, vn.bits, n)
    assert np.array_equal(d_len.cpu().numpy(), len_o)
    assert np.array_equal(bits_of(d_kc), kc_o) and np.array_equal(bits_of(d_vc), vc_o)
    return n, ties, report


def test_tiny_head():
    n, ties, _ = run_case(1, 4, 64, 1000, 0.5, 1, spike_rows=2)
    assert not ties


@pytest.mark.parametrize("V", [1, 255, 256, 257, 1001, 4099])
def test_ragged_vocabulary(V):
    """V not a multiple of the 256-entry weight tile (and smaller than one tile)."""
    run_case(3, 5, 128, V, 0.3, 10 + V, spike_rows=6)


@pytest.mark.parametrize("tau", [0.0, 0.5, 0.95, 1.0])
def test_commit_counts_across_tau(tau):
    """Spiked rows make confidences span (0, 1): counts from 1 to B occur at tau 0.5."""
    n, _, _ = run_case(8, 8, 256, 8000, tau, 20, spike_rows=40, lens=np.arange(8) * 3)
    if tau == 0.0:
        assert np.all(n == 8)
    if tau == 1.0:
        assert np.all(n == 1)


def test_more_rows_than_one_tile():
    """Several 128-row tiles of hidden states (a ragged last one)."""
    run_case(20, 8, 192, 5000, 0.5, 30, spike_rows=60)


def test_qwen7b_shaped_head_batch1():
    """The Qwen2.5-7B head: hidden 3584, V = 152064, one sequence of B = 4 proposals."""
    n, ties, report = run_case(1, 4, 3584, 152064, 0.9, 40, spike_rows=2, hkv=4, D=128, cap=2100,
                               lens=[2048])
    print(f"near ties {ties}, near-tau {report}")


def test_qwen7b_shaped_head_batch64_rows():
    """512 proposal rows (batch 64, B = 8) against the 7B-sized hidden width, on a
    32768-entry slice of the vocabulary (the oracle's fp64 product stays short)."""
    n, ties, report = run_case(64, 8, 3584, 32768, 0.5, 50, spike_rows=128, hkv=4, D=128, cap=64)
    print(f"near ties {ties}, near-tau {report}")
