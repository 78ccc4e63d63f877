"""mars_accept_margin on the GPU against the fp64 oracle: the margin gate
conf = p1 - p2 ([blog] "Inference": the top token's lead over the rest), computed
in the same single pass over the logits, with the same commit rule and append."""
import numpy as np
import pytest
import torch

import oracle
import token_decoding_gb300 as mars
from token_decoding_gb300 import synth
from tests.gpu_util import bits_of, check_accept, dev_bf16

pytestmark = pytest.mark.gpu


def run(logits, tau, kn, vn, kc, vc, lens):
    d_kc, d_vc = dev_bf16(kc), dev_bf16(vc)
    d_len = torch.from_numpy(np.asarray(lens, dtype=np.int32)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tok, conf, n = mars.accept(dev_bf16(logits), tau, dev_bf16(kn), dev_bf16(vn), d_kc, d_vc, d_len,
                               status=status, gate="margin")
    torch.cuda.synchronize()
    return (tok.cpu().numpy(), conf.cpu().numpy(), n.cpu().numpy(), bits_of(d_kc), bits_of(d_vc),
            d_len.cpu().numpy(), int(status.item()))


def kv_for(batch, B, hkv, D, cap, seed):
    g = np.random.default_rng(seed)
    mk = lambda shape: synth.Bf16.from_float(g.standard_normal(shape, dtype=np.float32))  # noqa: E731
    return mk((batch, B, hkv, D)), mk((batch, B, hkv, D)), mk((batch, hkv, cap, D)), mk((batch, hkv, cap, D))


def check_full(logits, tau, lens, hkv=2, D=64, cap=None, seed=0):
    batch, B, _ = logits.shape
    cap = int(max(lens)) + B if cap is None else cap
    kn, vn, kc, vc = kv_for(batch, B, hkv, D, cap, seed)
    tok, conf, n, kc2, vc2, lens2, status = run(logits, tau, kn, vn, kc, vc, lens)
    assert status == 0
    _, report = check_accept(tok, conf, n, logits.f64, tau, gate="margin")
    kc_o, vc_o, len_o = oracle.append_kv(kc.bits, vc.bits, lens, kn.bits, vn.bits, n)
    assert np.array_equal(lens2, len_o)
    assert np.array_equal(kc2, kc_o) and np.array_equal(vc2, vc_o)
    return conf, n, report


@pytest.mark.parametrize("tau", [1.0, 0.5, 0.1, 0.0])
def test_tiny_decode_step(tau):
    s = synth.TINY_DECODE
    logits = synth.step_logits(s, 0)
    check_full(logits, tau, [60], hkv=s.Hkv, D=s.D)


def test_batch1_7b_vocab():
    s = synth.DECODE_7B_B1
    logits = synth.step_logits(s, 3)
    check_full(logits, 0.5, [2048], hkv=s.Hkv, D=s.D)


def test_batch64_7b_vocab():
    s = synth.DECODE_7B_B64
    logits = synth.step_logits(s, 1)
    lens = synth.initial_cache_lens(s)
    check_full(logits, 0.95, lens, hkv=s.Hkv, D=s.D, cap=int(lens.max()) + s.B)


def test_margins_span_the_unit_interval_and_commit_many():
    """Spikes of varied height give margins across (0, 1), so commit counts 1..B occur."""
    g = np.random.default_rng(11)
    batch, B, V = 24, 8, 5000
    x = g.standard_normal((batch, B, V), dtype=np.float32)
    for b in range(batch):
        for i in range(B):
            x[b, i, g.integers(0, V)] += g.uniform(5.0, 16.0)
    logits = synth.Bf16.from_float(x)
    conf, n, _ = check_full(logits, 0.2, np.full(batch, 10), seed=12)
    assert conf.min() < 0.05 and conf.max() > 0.95
    assert len(set(n.tolist())) >= 4 and n.max() >= 5


def test_ties_and_runner_up_across_slices():
    """The runner-up is found wherever it lies: in the max's 16 KB slice, in another
    slice, or in the unaligned head and tail; an exact tie gives a margin of 0."""
    V = 8192 * 3 + 5
    x = np.full((1, 6, V), -4.0, dtype=np.float32)
    x[0, 0, [100, 20000]] = 5.0           # tie across slices -> margin 0, token 100
    x[0, 1, 3] = 6.0
    x[0, 1, 24000] = 5.5                   # runner-up in the last slice
    x[0, 2, V - 1] = 6.0
    x[0, 2, 0] = 5.75                      # max in the tail, runner-up in the head
    x[0, 3, 8191] = 7.0
    x[0, 3, 8192] = 7.0                    # tie on a slice boundary -> margin 0, token 8191
    x[0, 4, 77] = 3.0                      # plain single spike
    x[0, 5, :] = 1.0                       # all equal -> margin 0, token 0
    logits = synth.Bf16.from_float(x)
    conf, n, _ = check_full(logits, 0.0, [0], seed=13)
    assert conf[0, 0] == 0.0 and conf[0, 3] == 0.0 and conf[0, 5] == 0.0


@pytest.mark.parametrize("V", [1, 2, 7, 8, 9, 8191, 8193, 16384 + 3])
def test_ragged_vocab(V):
    g = np.random.default_rng(V)
    logits = synth.Bf16.from_float(g.standard_normal((3, 4, V), dtype=np.float32) * 3)
    conf, _, _ = check_full(logits, 0.2, [5, 0, 17], seed=V)
    if V == 1:
        assert np.all(conf == 1.0)


def run_batch_min(logits, tau, kn, vn, kc, vc, lens, gate="prob"):
    d_kc, d_vc = dev_bf16(kc), dev_bf16(vc)
    d_len = torch.from_numpy(np.asarray(lens, dtype=np.int32)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tok, conf, n = mars.accept(dev_bf16(logits), tau, dev_bf16(kn), dev_bf16(vn), d_kc, d_vc, d_len,
                               status=status, gate=gate, batch_min=True)
    torch.cuda.synchronize()
    return (tok.cpu().numpy(), conf.cpu().numpy(), n.cpu().numpy(), bits_of(d_kc), bits_of(d_vc),
            d_len.cpu().numpy(), int(status.item()))


@pytest.mark.parametrize("gate", ["prob", "margin"])
def test_batch_minimum_mode(gate):
    """The paper's original sampler: every sequence commits the batch-minimum count."""
    g = np.random.default_rng(21)
    batch, B, V, hkv, D = 16, 8, 3000, 2, 64
    x = g.standard_normal((batch, B, V), dtype=np.float32)
    for b in range(batch):
        for i in range(B):
            x[b, i, g.integers(0, V)] += g.uniform(6.0, 16.0)
    x[:, :2, 5] += 30.0  # the first two positions always pass: the minimum is at least 2
    logits = synth.Bf16.from_float(x)
    lens = g.integers(0, 50, size=batch).astype(np.int32)
    kn, vn, kc, vc = kv_for(batch, B, hkv, D, 64, 22)
    tok, conf, n, kc2, vc2, lens2, status = run_batch_min(logits, 0.2, kn, vn, kc, vc, lens, gate)
    assert status == 0
    t_o, c_o, n_o = oracle.accept(logits.f64, 0.2, gate, batch_min=True)
    assert np.array_equal(tok, t_o)
    _, _, n_each = oracle.accept(logits.f64, 0.2, gate)
    assert len(set(n_each.tolist())) > 1  # the per-sequence counts differ, so the mode matters
    assert np.all(n == n[0]) and np.array_equal(n, n_o) and n[0] >= 2, (n, n_o)
    kc_o, vc_o, len_o = oracle.append_kv(kc.bits, vc.bits, lens, kn.bits, vn.bits, n_o)
    assert np.array_equal(lens2, len_o) and np.array_equal(kc2, kc_o) and np.array_equal(vc2, vc_o)


def test_batch_minimum_mode_capacity():
    """A sequence without room for the batch-minimum count reports and keeps its cache."""
    g = np.random.default_rng(23)
    batch, B, V, hkv, D, cap = 4, 4, 500, 1, 64, 16
    x = g.standard_normal((batch, B, V), dtype=np.float32)
    x[:, :, 7] += 20.0  # every position confident: counts are B everywhere
    logits = synth.Bf16.from_float(x)
    lens = np.array([0, 5, 14, 12], dtype=np.int32)  # 14 + 4 > 16
    kn, vn, kc, vc = kv_for(batch, B, hkv, D, cap, 24)
    tok, conf, n, kc2, vc2, lens2, status = run_batch_min(logits, 0.5, kn, vn, kc, vc, lens)
    assert status & mars.MARS_DEV_CAPACITY
    assert list(n) == [4, 4, 0, 4]
    n_eff = np.array([4, 4, 0, 4])
    kc_o, vc_o, len_o = oracle.append_kv(kc.bits, vc.bits, lens, kn.bits, vn.bits, n_eff)
    assert np.array_equal(lens2, len_o) and np.array_equal(kc2, kc_o) and np.array_equal(vc2, vc_o)
