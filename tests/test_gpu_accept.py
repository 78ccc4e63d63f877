"""mars_accept on the GPU against the fp64 oracle (top-1 probability, argmax,
left-to-right commit with at-least-one, block-level KV append)."""
import numpy as np
import pytest
import torch

import oracle
import token_decoding_gb300 as mars
from token_decoding_gb300 import synth
from tests.gpu_util import bits_of, check_accept, dev_bf16

pytestmark = pytest.mark.gpu


def run_accept(logits, tau, kn, vn, kc, vc, lens, cap=None, workspace=None):
    """logits / kn / vn / kc / vc are synth.Bf16 or uint16 bit arrays; lens int32 numpy."""
    d_logits = dev_bf16(logits)
    d_kn, d_vn = dev_bf16(kn), dev_bf16(vn)
    d_kc, d_vc = dev_bf16(kc), dev_bf16(vc)
    d_len = torch.from_numpy(np.asarray(lens, dtype=np.int32)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tok, conf, n = mars.accept(d_logits, tau, d_kn, d_vn, d_kc, d_vc, d_len, workspace=workspace, status=status)
    torch.cuda.synchronize()
    return (tok.cpu().numpy(), conf.cpu().numpy(), n.cpu().numpy(), bits_of(d_kc), bits_of(d_vc),
            d_len.cpu().numpy(), int(status.item()))


def kv_for(batch, B, hkv, D, cap, seed):
    g = np.random.default_rng(seed)
    kn = synth.Bf16.from_float(g.standard_normal((batch, B, hkv, D), dtype=np.float32))
    vn = synth.Bf16.from_float(g.standard_normal((batch, B, hkv, D), dtype=np.float32))
    kc = synth.Bf16.from_float(g.standard_normal((batch, hkv, cap, D), dtype=np.float32))
    vc = synth.Bf16.from_float(g.standard_normal((batch, hkv, cap, D), dtype=np.float32))
    return kn, vn, kc, vc


def check_full(logits, tau, kn, vn, kc, vc, lens):
    tok, conf, n, kc2, vc2, lens2, status = run_accept(logits, tau, kn, vn, kc, vc, lens)
    assert status == 0
    _, report = check_accept(tok, conf, n, logits.f64, tau)
    # the cache must hold exactly the rows the kernel committed, everything else untouched
    kc_o, vc_o, len_o = oracle.append_kv(kc.bits, vc.bits, lens, kn.bits, vn.bits, n)
    assert np.array_equal(lens2, len_o)
    assert np.array_equal(kc2, kc_o) and np.array_equal(vc2, vc_o)
    return n, report


@pytest.mark.parametrize("tau", [1.0, 0.9, 0.0])
def test_tiny_decode_step(tau):
    shape = synth.TINY_DECODE
    logits = synth.step_logits(shape, 0)
    kn, vn, kc, vc = kv_for(1, shape.B, shape.Hkv, shape.D, shape.cap, 1)
    n, _ = check_full(logits, tau, kn, vn, kc, vc, np.array([60], dtype=np.int32))
    if tau == 1.0:
        assert n[0] == 1
    if tau == 0.0:
        assert n[0] == shape.B


@pytest.mark.parametrize("tau", [1.0, 0.95, 0.9, 0.5])
def test_batch1_7b_shapes(tau):
    shape = synth.DECODE_7B_B1
    logits = synth.step_logits(shape, 3)
    kn, vn, kc, vc = kv_for(1, shape.B, shape.Hkv, shape.D, 2048 + 64, 2)
    check_full(logits, tau, kn, vn, kc, vc, np.array([2048], dtype=np.int32))


def test_batch64_7b_shapes():
    shape = synth.DECODE_7B_B64
    logits = synth.step_logits(shape, 0)
    lens = synth.initial_cache_lens(shape)
    kn, vn, kc, vc = kv_for(shape.batch, shape.B, shape.Hkv, shape.D, 4096 + 16, 3)
    n, report = check_full(logits, 0.95, kn, vn, kc, vc, lens)
    print("near-threshold positions:", report)


@pytest.mark.parametrize("tau", [0.9, 0.5, 0.2])
def test_multi_commit_coverage(tau):
    """Spikes of height U[12, 30] make confidences span (0, 1): commit counts 1..B occur."""
    g = synth.rng_for("coverage", tau)
    logits = synth.spiked_logits(32, 8, 152064, 2.0, 0.8, 12.0, 30.0, g)
    kn, vn, kc, vc = kv_for(32, 8, 4, 128, 300, 4)
    lens = np.random.default_rng(5).integers(0, 290, size=32).astype(np.int32)
    n, _ = check_full(logits, tau, kn, vn, kc, vc, lens)
    assert len(set(n.tolist())) > 2


@pytest.mark.parametrize("V", [1, 7, 13, 1001, 4099, 152065])
def test_ragged_vocab(V):
    """V not a multiple of 8: rows start at every 2-byte offset mod 16."""
    g = np.random.default_rng(V)
    logits = synth.Bf16.from_float(g.standard_normal((3, 5, V), dtype=np.float32) * 3)
    kn, vn, kc, vc = kv_for(3, 5, 2, 64, 40, 6)
    check_full(logits, 0.3, kn, vn, kc, vc, np.array([0, 7, 30], dtype=np.int32))


def test_ties_and_split_boundaries():
    """Equal maxima in different CTA slices and inside one 16-byte vector: lowest index wins."""
    V = 152064
    x = np.zeros((2, 4, V), dtype=np.float32)
    x[0, 0, [5, 6, 70000, 151000]] = 4.0        # first two share a vector
    x[0, 1, [150000, 3]] = 2.0
    x[0, 2, :] = 1.0                            # all equal -> token 0
    x[0, 3, [V - 1, V - 2]] = 9.0
    x[1] = np.random.default_rng(7).standard_normal((4, V)).astype(np.float32)
    x[1, :, 100] = 7.0
    x[1, :, 90000] = 7.0
    logits = synth.Bf16.from_float(x)
    kn, vn, kc, vc = kv_for(2, 4, 1, 64, 16, 8)
    tok, conf, n, *_ = run_accept(logits, 0.5, kn, vn, kc, vc, np.array([0, 3], dtype=np.int32))
    assert tok[0].tolist() == [5, 3, 0, V - 2]
    assert tok[1].tolist() == [100] * 4
    check_accept(tok, conf, n, logits.f64, 0.5)


def test_single_position_block():
    g = np.random.default_rng(9)
    logits = synth.Bf16.from_float(g.standard_normal((4, 1, 5000), dtype=np.float32))
    kn, vn, kc, vc = kv_for(4, 1, 2, 128, 8, 10)
    n, _ = check_full(logits, 0.99, kn, vn, kc, vc, np.array([0, 1, 6, 7], dtype=np.int32))
    assert np.all(n == 1)


def test_capacity_overflow_is_reported_and_skipped():
    g = np.random.default_rng(11)
    logits = synth.Bf16.from_float(g.standard_normal((2, 4, 300), dtype=np.float32))
    kn, vn, kc, vc = kv_for(2, 4, 1, 64, 10, 12)
    lens = np.array([4, 9], dtype=np.int32)   # tau = 0 commits 4: 4 + 4 <= 10, 9 + 4 > 10
    tok, conf, n, kc2, vc2, lens2, status = run_accept(logits, 0.0, kn, vn, kc, vc, lens)
    assert status & mars.MARS_DEV_CAPACITY
    assert n.tolist() == [4, 0]
    assert lens2.tolist() == [8, 9]
    assert np.array_equal(kc2[1], kc.bits[1]) and np.array_equal(vc2[1], vc.bits[1])
    kc_o, vc_o, _ = oracle.append_kv(kc.bits[:1], vc.bits[:1], lens[:1], kn.bits[:1], vn.bits[:1], n[:1])
    assert np.array_equal(kc2[:1], kc_o) and np.array_equal(vc2[:1], vc_o)


def test_workspace_is_reusable_across_calls():
    """Tickets reset themselves: two calls in a row on one workspace give the same answer."""
    shape = synth.DECODE_7B_B1
    logits = synth.step_logits(shape, 5)
    ws = mars.accept_workspace(1, shape.B, shape.V, "cuda")
    kn, vn, kc, vc = kv_for(1, shape.B, shape.Hkv, shape.D, 2100, 13)
    r1 = run_accept(logits, 0.5, kn, vn, kc, vc, np.array([100], dtype=np.int32), workspace=ws)
    r2 = run_accept(logits, 0.5, kn, vn, kc, vc, np.array([100], dtype=np.int32), workspace=ws)
    r3 = run_accept(logits, 0.5, kn, vn, kc, vc, np.array([100], dtype=np.int32))  # fresh zeroed workspace
    for a, b, c in zip(r1, r2, r3):
        assert np.array_equal(np.asarray(a), np.asarray(b)) and np.array_equal(np.asarray(a), np.asarray(c))


def test_host_rejects_bad_arguments():
    d = torch.zeros((1, 4, 100), dtype=torch.bfloat16, device="cuda")
    kn = torch.zeros((1, 4, 1, 64), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16, device="cuda")
    ln = torch.zeros(1, dtype=torch.int32, device="cuda")
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(mars.MarsError) as e:
        mars.accept(d, 0.5, kn, kn, kc, kc, ln, workspace=small)
    assert e.value.code == 2


def test_word_outputs_need_only_4_byte_alignment():
    """tokens / conf / n_commit / cache_len may be rows of larger arrays (4-byte aligned)."""
    g = np.random.default_rng(21)
    logits = synth.Bf16.from_float(g.standard_normal((1, 4, 999), dtype=np.float32))
    kn, vn, kc, vc = kv_for(1, 4, 1, 64, 16, 22)
    hist = torch.zeros((5, 1), dtype=torch.int32, device="cuda")
    lens = torch.zeros((3,), dtype=torch.int32, device="cuda")
    conf = torch.zeros((3, 4), dtype=torch.float32, device="cuda")
    toks = torch.zeros((3, 4), dtype=torch.int32, device="cuda")
    lens[1] = 5
    t, c, n = mars.accept(dev_bf16(logits), 0.0, dev_bf16(kn), dev_bf16(vn), dev_bf16(kc), dev_bf16(vc),
                          lens[1:2], tokens=toks[1:2], conf=conf[1:2], n_commit=hist[3])
    torch.cuda.synchronize()
    assert int(hist[3].item()) == 4 and int(lens[1].item()) == 9
    t_o, c_o, _ = oracle.accept(logits.f64, 0.0)
    assert np.array_equal(toks[1].cpu().numpy(), t_o[0])
