"""Sliding-window decode episodes on the GPU against an fp64 oracle replay.

One decode step of MARS ("MARS: Enabling Autoregressive Models Multi-Token
Generation", Fig. 2 right: B placeholders appended after the cursor and filled
by one forward; the authors' blog post, "Inference: a knob, not a mode switch":
commit the leading confident proposals into the block-level KV cache) is
decode attention over the committed cache plus the B placeholders, then the
acceptance rule, then the append.  Here whole episodes run on the GPU with the
cache and the cursor carried on the device from step to step, so every step's
decode attention reads the rows that the previous steps' mars_accept appended.

The replay composes the oracle's pinned pieces in the same order:
oracle.decode_attn -> oracle.accept -> oracle.append_kv, carrying its own fp64
cache and lengths.  At every step the attention output is held to 1e-2, the
tokens and confidences to the accept tolerances, and the commit count must be
bit-exact unless the first differing pass/fail decision sits within 1e-4 of
tau; then the replay adopts the GPU's count (so later steps stay comparable)
and the position is reported.  The caches and lengths are compared bit for bit
at the end of each episode.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import token_decoding_gb300 as mars
from token_decoding_gb300 import synth
from tests.gpu_util import ATTN_TOL, bf16_to_f64, check_accept, dev_bf16, max_abs

pytestmark = pytest.mark.gpu


class Replay:
    """The oracle's side of one episode: fp64 caches, lengths, and the near-tau report."""

    def __init__(self, kc64, vc64, lens):
        self.kc, self.vc = kc64, vc64
        self.lens = np.asarray(lens, dtype=np.int64).copy()
        self.report = []

    def decode(self, q64, kn64, vn64, scale):
        return oracle.decode_attn(q64, kn64, vn64, self.kc, self.vc, self.lens, scale)

    def accept_and_append(self, step, tok, conf, n_gpu, logits64, tau, kn64, vn64):
        n_o, report = check_accept(tok, conf, n_gpu, logits64, tau)
        n_used = np.asarray(n_o, dtype=np.int64).copy()
        for b, pos in report:  # a near-tau decision: follow the GPU from here on
            n_used[b] = int(n_gpu[b])
            self.report.append((step, b, pos))
        self.kc, self.vc, self.lens = oracle.append_kv(self.kc, self.vc, self.lens, kn64, vn64, n_used)
        return n_used


def compare_final(replay, d_kc, d_vc, d_len, rows=None):
    got_len = d_len.cpu().numpy().astype(np.int64)
    kc, vc = bf16_to_f64(d_kc), bf16_to_f64(d_vc)
    if rows is not None:
        got_len, kc, vc = got_len[rows], kc[rows], vc[rows]
    assert np.array_equal(got_len, replay.lens), (got_len, replay.lens)
    # bf16 -> f64 widening is exact, so equal doubles mean equal bits
    assert np.array_equal(kc, replay.kc)
    assert np.array_equal(vc, replay.vc)


def test_batch1_7b_episode_tau_sweep():
    """The Qwen2.5-7B-shaped batch-1 workload: cache 2048, B = 4, 256 steps, at each
    tau in {1.0, 0.95, 0.9, 0.5}; the four episodes share their per-step inputs."""
    s = synth.DECODE_7B_B1
    scale = s.D ** -0.5
    kc0, vc0 = synth.cache_inputs(s, fill_len=s.len_lo)
    lens0 = synth.initial_cache_lens(s)
    max_len = s.cap - s.B
    runs = []
    for tau in s.taus:
        d_kc, d_vc = dev_bf16(kc0), dev_bf16(vc0)
        d_len = torch.from_numpy(lens0.copy()).cuda()
        ws = mars.accept_workspace(s.batch, s.B, s.V, "cuda")
        runs.append((tau, d_kc, d_vc, d_len, ws, Replay(kc0.f64.copy(), vc0.f64.copy(), lens0)))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    worst = 0.0
    commits = {tau: 0 for tau in s.taus}
    for t in range(s.steps):
        q, kn, vn = synth.step_inputs(s, t)
        logits = synth.step_logits(s, t)
        d_q, d_kn, d_vn, d_logits = dev_bf16(q), dev_bf16(kn), dev_bf16(vn), dev_bf16(logits)
        outs = []
        for tau, d_kc, d_vc, d_len, ws, _ in runs:
            o = mars.decode_attn(d_q, d_kn, d_vn, d_kc, d_vc, d_len, max_len, scale=scale, status=status)
            tok, conf, n = mars.accept(d_logits, tau, d_kn, d_vn, d_kc, d_vc, d_len, workspace=ws, status=status)
            outs.append((bf16_to_f64(o), tok.cpu().numpy(), conf.cpu().numpy(), n.cpu().numpy()))
        for (tau, *_, rep), (o, tok, conf, n) in zip(runs, outs):
            err = max_abs(o, rep.decode(q.f64, kn.f64, vn.f64, scale))
            assert err <= ATTN_TOL, (tau, t, err)
            worst = max(worst, err)
            n_used = rep.accept_and_append(t, tok, conf, n, logits.f64, tau, kn.f64, vn.f64)
            commits[tau] += int(n_used.sum())
            if tau == 1.0:
                assert n.tolist() == [1]  # tau = 1 gives back one-token AR decoding
    assert int(status.item()) == 0
    for tau, d_kc, d_vc, d_len, _, rep in runs:
        compare_final(rep, d_kc, d_vc, d_len)
        print(f"tau {tau}: {commits[tau]} tokens in {s.steps} steps, near-tau reports {rep.report}")
    print(f"worst attention |delta| over the episodes: {worst:.3g}")


def spiked_logits_device(batch, B, V, sigma, prob, lo, hi, gen):
    x = torch.randn((batch, B, V), generator=gen, device="cuda", dtype=torch.float32) * sigma
    spiked = torch.rand((batch, B), generator=gen, device="cuda") < prob
    tok = torch.randint(0, V, (batch, B), generator=gen, device="cuda")
    height = lo + (hi - lo) * torch.rand((batch, B), generator=gen, device="cuda")
    x.scatter_add_(2, tok.unsqueeze(-1), (height * spiked).unsqueeze(-1))
    return x.to(torch.bfloat16)


def test_batch64_7b_episode_checked_on_sequences():
    """The Qwen2.5-7B-shaped batch-64 workload (caches 256..4096, B = 8, tau = 0.95,
    128 steps) runs whole on the GPU; the oracle replays three of its sequences
    (the longest, the shortest and sequence 0), whose inputs are drawn on the host
    per sequence.  The other sequences take device-drawn inputs of the same
    recipe: sequences are independent, and those are checked for the cursor
    invariant (every step commits at least one token and cache_len grows by the
    commit count)."""
    s = synth.DECODE_7B_B64
    scale = s.D ** -0.5
    lens0 = synth.initial_cache_lens(s)
    order = np.argsort(-lens0, kind="stable")
    check = sorted({int(order[0]), int(order[-1]), 0})
    gen = torch.Generator(device="cuda")
    gen.manual_seed(77)
    max_len = s.cap - s.B
    d_kc = torch.randn((s.batch, s.Hkv, s.cap, s.D), generator=gen, device="cuda").to(torch.bfloat16)
    d_vc = torch.randn((s.batch, s.Hkv, s.cap, s.D), generator=gen, device="cuda").to(torch.bfloat16)
    kcs, vcs = [], []
    for b in check:
        kc, vc = synth.seq_cache_inputs(s, b, int(lens0[b]))
        d_kc[b:b + 1].copy_(dev_bf16(kc))
        d_vc[b:b + 1].copy_(dev_bf16(vc))
        kcs.append(kc.f64)
        vcs.append(vc.f64)
    rep = Replay(np.concatenate(kcs), np.concatenate(vcs), lens0[check])
    d_len = torch.from_numpy(lens0.copy()).cuda()
    ws = mars.accept_workspace(s.batch, s.B, s.V, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    total = np.zeros(s.batch, dtype=np.int64)
    worst = 0.0
    for t in range(s.steps):
        d_q = torch.randn((s.batch, s.B, s.Hq, s.D), generator=gen, device="cuda").to(torch.bfloat16)
        d_kn = torch.randn((s.batch, s.B, s.Hkv, s.D), generator=gen, device="cuda").to(torch.bfloat16)
        d_vn = torch.randn((s.batch, s.B, s.Hkv, s.D), generator=gen, device="cuda").to(torch.bfloat16)
        d_logits = spiked_logits_device(s.batch, s.B, s.V, s.base_sigma, s.spike_prob, s.spike_lo, s.spike_hi, gen)
        host = [synth.seq_step_inputs(s, t, b) + (synth.seq_step_logits(s, t, b),) for b in check]
        for b, (q, kn, vn, lg) in zip(check, host):
            d_q[b:b + 1].copy_(dev_bf16(q))
            d_kn[b:b + 1].copy_(dev_bf16(kn))
            d_vn[b:b + 1].copy_(dev_bf16(vn))
            d_logits[b:b + 1].copy_(dev_bf16(lg))
        o = mars.decode_attn(d_q, d_kn, d_vn, d_kc, d_vc, d_len, max_len, scale=scale, status=status)
        tok, conf, n = mars.accept(d_logits, s.taus[0], d_kn, d_vn, d_kc, d_vc, d_len, workspace=ws, status=status)
        o64, tok, conf, n = bf16_to_f64(o[check]), tok.cpu().numpy(), conf.cpu().numpy(), n.cpu().numpy()
        assert np.all(n >= 1) and np.all(n <= s.B)
        total += n
        q64 = np.concatenate([h[0].f64 for h in host])
        kn64 = np.concatenate([h[1].f64 for h in host])
        vn64 = np.concatenate([h[2].f64 for h in host])
        lg64 = np.concatenate([h[3].f64 for h in host])
        err = max_abs(o64, rep.decode(q64, kn64, vn64, scale))
        assert err <= ATTN_TOL, (t, err)
        worst = max(worst, err)
        rep.accept_and_append(t, tok[check], conf[check], n[check], lg64, s.taus[0], kn64, vn64)
    assert int(status.item()) == 0
    assert np.array_equal(d_len.cpu().numpy().astype(np.int64), lens0 + total)
    compare_final(rep, d_kc, d_vc, d_len, rows=check)
    print(f"sequences {check}: near-tau reports {rep.report}; worst attention |delta| {worst:.3g}; "
          f"tokens per step over the batch {total.sum() / s.steps:.2f}")


COVERAGE = dataclasses.replace(
    synth.DECODE_7B_B64, name="coverage-episode-b4-B8-V32000", batch=4, V=32000, cap=700 + 48 * 8, len_lo=0,
    len_hi=700, steps=48, spike_prob=0.8, spike_lo=12.0, spike_hi=30.0, taus=(0.5,))


def test_multi_commit_episode():
    """Spikes of height U[12, 30] make confidences span (0, 1), so steps commit 1..B
    tokens and later steps read multi-row appends (B = 8, 28/4 heads, D = 128)."""
    s = COVERAGE
    scale = s.D ** -0.5
    lens0 = np.array([0, 37, 300, 700], dtype=np.int32)
    kc, vc = synth.cache_inputs(s, fill_len=700)
    d_kc, d_vc = dev_bf16(kc), dev_bf16(vc)
    d_len = torch.from_numpy(lens0.copy()).cuda()
    rep = Replay(kc.f64.copy(), vc.f64.copy(), lens0)
    ws = mars.accept_workspace(s.batch, s.B, s.V, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    seen = set()
    for t in range(s.steps):
        q, kn, vn = synth.step_inputs(s, t)
        logits = synth.step_logits(s, t)
        d_kn, d_vn = dev_bf16(kn), dev_bf16(vn)
        o = mars.decode_attn(dev_bf16(q), d_kn, d_vn, d_kc, d_vc, d_len, s.cap - s.B, scale=scale, status=status)
        tok, conf, n = mars.accept(dev_bf16(logits), s.taus[0], d_kn, d_vn, d_kc, d_vc, d_len, workspace=ws,
                                   status=status)
        assert max_abs(bf16_to_f64(o), rep.decode(q.f64, kn.f64, vn.f64, scale)) <= ATTN_TOL, t
        n_used = rep.accept_and_append(t, tok.cpu().numpy(), conf.cpu().numpy(), n.cpu().numpy(), logits.f64,
                                       s.taus[0], kn.f64, vn.f64)
        seen.update(n_used.tolist())
    assert int(status.item()) == 0
    compare_final(rep, d_kc, d_vc, d_len)
    assert len(seen) >= 4, seen
    print(f"commit counts seen {sorted(seen)}; near-tau reports {rep.report}")
