"""The deferred-KV sampler on the GPU (mars_decode_attn_deferred and
mars_accept_ex with MARS_ACCEPT_DEFERRED) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import token_decoding_gb300 as mars
from token_decoding_gb300 import synth
from tests.gpu_util import ATTN_TOL, bf16_to_f64, bits_of, check_accept, dev_bf16, max_abs

pytestmark = pytest.mark.gpu


def rand_bf16(shape, seed, sigma=1.0):
    g = np.random.default_rng(seed)
    return synth.Bf16.from_float(g.standard_normal(shape, dtype=np.float32) * np.float32(sigma))


def i32(x):
    return torch.from_numpy(np.asarray(x, dtype=np.int32)).cuda()


def run(q, kn, vn, kc, vc, lens, pend, max_len, scale, status=None):
    d_kc, d_vc = dev_bf16(kc), dev_bf16(vc)
    o = mars.decode_attn_deferred(dev_bf16(q), dev_bf16(kn), dev_bf16(vn), d_kc, d_vc, i32(lens), i32(pend),
                                  max_len, scale=scale, status=status)
    torch.cuda.synchronize()
    return bf16_to_f64(o), bits_of(o), bits_of(d_kc), bits_of(d_vc)


def check_cache(kc_bits_in, kn_bits, kc_bits_out, lens, pend, bs):
    """Rows [len, len + pending) hold the pending K rows bit for bit; every other row is untouched."""
    for b in bs:
        want = kc_bits_in[b].copy()
        n, p = int(lens[b]), int(pend[b])
        want[:, n:n + p, :] = np.transpose(kn_bits[b, :p], (1, 0, 2))
        assert np.array_equal(kc_bits_out[b], want), b


def case(batch, B, hq, hkv, D, cap, lens, pend, seed, max_len=None, sample=None, nan_invalid=False):
    S = 2 * B
    q = rand_bf16((batch, S, hq, D), seed)
    kn, vn = rand_bf16((batch, S, hkv, D), seed + 1), rand_bf16((batch, S, hkv, D), seed + 2)
    kc, vc = rand_bf16((batch, hkv, cap, D), seed + 3), rand_bf16((batch, hkv, cap, D), seed + 4)
    lens, pend = np.asarray(lens, dtype=np.int32), np.asarray(pend, dtype=np.int32)
    if nan_invalid:
        nan = np.uint16(0x7FC0)
        for b in range(batch):
            p = int(pend[b])
            q.bits[b, p:B], kn.bits[b, p:B], vn.bits[b, p:B] = nan, nan, nan
        q, kn, vn = (synth.Bf16(t.bits, synth.bf16_bits_to_f64(t.bits)) for t in (q, kn, vn))
    scale = D ** -0.5
    got, got_bits, kc_out, vc_out = run(q, kn, vn, kc, vc, lens, pend, cap if max_len is None else max_len, scale)
    bs = np.arange(batch) if sample is None else np.asarray(sample)
    want, _, _ = oracle.decode_attn_deferred(q.f64[bs], kn.f64[bs], vn.f64[bs], kc.f64[bs], vc.f64[bs], lens[bs],
                                             pend[bs], scale)
    for j, b in enumerate(bs):
        valid = [c for c in range(S) if c < pend[b] or c >= B]
        invalid = [c for c in range(S) if c not in valid]
        err = max_abs(got[b, valid], want[j, valid])
        assert err <= ATTN_TOL, (b, err)
        assert np.all(got_bits[b, invalid] == 0), b  # +0.0 exactly
    check_cache(kc.bits, kn.bits, kc_out, lens, pend, bs)
    check_cache(vc.bits, vn.bits, vc_out, lens, pend, bs)


def test_tiny_deferred_step():
    s = synth.TINY_DECODE
    case(1, s.B, s.Hq, s.Hkv, s.D, s.cap, [60], [3], 1100)


@pytest.mark.parametrize("p", [0, 1, 4, 8])
def test_batch1_7b_shapes(p):
    s = synth.DECODE_7B_B64
    case(1, s.B, s.Hq, s.Hkv, s.D, 2048 + 64, [2048], [p], 1200 + p)


def test_batch64_7b_shapes_sampled():
    """The full batch-64 step (B = 8, so 16 slots, 7 heads of 16 rows: 112 of 128 MMA rows)."""
    s = synth.DECODE_7B_B64
    lens = synth.initial_cache_lens(s)
    pend = np.random.default_rng(13).integers(0, s.B + 1, size=s.batch)
    order = np.argsort(-lens, kind="stable")
    sample = sorted(set(order[:3].tolist() + order[-3:].tolist() + [0, 17, 40, 63]))
    case(s.batch, s.B, s.Hq, s.Hkv, s.D, 4096 + 16, lens, pend, 1300, max_len=4096, sample=sample)


@pytest.mark.parametrize("lens,pend", [([0, 0], [0, 3]), ([62, 63], [3, 4]), ([64, 65], [4, 1]),
                                       ([127, 190], [2, 4])])
def test_cursor_around_tiles(lens, pend):
    """Pending rows that straddle a 64-key tile boundary, empty caches, nothing pending."""
    case(2, 4, 8, 2, 128, 256, lens, pend, 1400 + lens[1])


@pytest.mark.parametrize("B", [1, 2, 3, 5, 8])
def test_block_sizes(B):
    rng = np.random.default_rng(B)
    pend = rng.integers(0, B + 1, size=3)
    case(3, B, 14, 2, 64, 320, [0, 100, 290], pend, 1500 + B)


@pytest.mark.parametrize("hq,hkv,D", [(4, 4, 64), (12, 3, 128), (32, 2, 128), (16, 1, 64)])
def test_head_layouts(hq, hkv, D):
    """Includes groups wider than one 128-row unit (16 heads x 16 slots), split into head chunks."""
    case(2, 8, hq, hkv, D, 540, [513, 7], [5, 8], 1600 + hq)


def test_invalid_slots_hold_nan():
    """Invalid pending slots carry NaN in q, k and v: valid rows are unchanged and invalid rows are zero."""
    case(4, 4, 8, 2, 64, 200, [10, 70, 0, 130], [0, 2, 1, 3], 1700, nan_invalid=True)
    case(2, 8, 28, 4, 128, 400, [300, 1], [1, 7], 1701, nan_invalid=True)


def test_all_pending_zero_matches_plain_step():
    """pending = 0: the mask slots compute the plain decode step."""
    B, hq, hkv, D, cap = 4, 8, 2, 128, 300
    q = rand_bf16((3, 2 * B, hq, D), 1800)
    kn, vn = rand_bf16((3, 2 * B, hkv, D), 1801), rand_bf16((3, 2 * B, hkv, D), 1802)
    kc, vc = rand_bf16((3, hkv, cap, D), 1803), rand_bf16((3, hkv, cap, D), 1804)
    lens = np.array([5, 200, 64], dtype=np.int32)
    _, got_bits, _, _ = run(q, kn, vn, kc, vc, lens, [0, 0, 0], cap, D ** -0.5)
    plain = mars.decode_attn(dev_bf16(q.bits[:, B:]), dev_bf16(kn.bits[:, B:]), dev_bf16(vn.bits[:, B:]),
                             dev_bf16(kc), dev_bf16(vc), i32(lens), cap, scale=D ** -0.5)
    torch.cuda.synchronize()
    # the same keys in the same tiles, the new ones in other columns of the new-key tile
    assert max_abs(synth.bf16_bits_to_f64(got_bits[:, B:]), bf16_to_f64(plain)) <= ATTN_TOL / 2
    assert np.all(got_bits[:, :B] == 0)


def test_bad_pending_and_capacity_status():
    B, hq, hkv, D, cap = 4, 4, 1, 64, 100
    q = rand_bf16((3, 2 * B, hq, D), 1900)
    kn, vn = rand_bf16((3, 2 * B, hkv, D), 1901), rand_bf16((3, 2 * B, hkv, D), 1902)
    kc, vc = rand_bf16((3, hkv, cap, D), 1903), rand_bf16((3, hkv, cap, D), 1904)
    lens, pend = np.array([10, 98, 20], dtype=np.int32), np.array([B + 1, 3, 2], dtype=np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got, got_bits, kc_out, vc_out = run(q, kn, vn, kc, vc, lens, pend, cap, D ** -0.5, status=status)
    assert int(status.item()) == mars.MARS_DEV_LEN_RANGE | mars.MARS_DEV_CAPACITY
    assert np.all(got_bits[:2] == 0)
    assert np.array_equal(kc_out[:2], kc.bits[:2]) and np.array_equal(vc_out[:2], vc.bits[:2])
    want, _, _ = oracle.decode_attn_deferred(q.f64[2:], kn.f64[2:], vn.f64[2:], kc.f64[2:], vc.f64[2:], lens[2:],
                                             pend[2:], D ** -0.5)
    valid = [0, 1] + list(range(B, 2 * B))
    assert max_abs(got[2, valid], want[0, valid]) <= ATTN_TOL


def test_rejects_block_size_above_8():
    B = 9
    q = torch.zeros((1, 2 * B, 4, 64), dtype=torch.bfloat16, device="cuda")
    kn = torch.zeros((1, 2 * B, 1, 64), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 1, 64, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mars.MarsError):
        mars.decode_attn_deferred(q, kn, kn, kc, kc.clone(), i32([0]), i32([0]), 0)


# ---------------------------------------------------------------- acceptance step


def spiked(batch, B, V, seed):
    g = np.random.default_rng(seed)
    return synth.spiked_logits(batch, B, V, 1.0, 0.6, 8.0, 16.0, g)


@pytest.mark.parametrize("gate", ["prob", "margin"])
def test_accept_deferred_advances_cursor_by_pending(gate):
    batch, B, V, cap, tau = 16, 8, 3001, 200, 0.6
    x = spiked(batch, B, V, 2000)
    rng = np.random.default_rng(2001)
    lens = rng.integers(0, 150, size=batch).astype(np.int32)
    pend = rng.integers(0, B + 1, size=batch).astype(np.int32)
    d_len, d_n = i32(lens), i32(pend)
    tok, conf, n = mars.accept_deferred(dev_bf16(x), tau, d_len, d_n, cap, gate=gate)
    torch.cuda.synchronize()
    n_o, report = check_accept(tok.cpu().numpy(), conf.cpu().numpy(), n.cpu().numpy(), x.f64, tau, gate)
    _, _, n_or, len_or = oracle.accept_deferred(x.f64, tau, lens, pend, gate)
    assert np.array_equal(d_len.cpu().numpy(), len_or)
    assert not report and np.array_equal(n.cpu().numpy(), n_or)


def test_accept_deferred_batch_min():
    batch, B, V, cap, tau = 8, 4, 1000, 64, 0.3
    x = spiked(batch, B, V, 2100)
    x.bits[:, :2] = synth.Bf16.from_float(np.where(np.arange(V) == 5, 30.0, 0.0).astype(np.float32)).bits
    x = synth.Bf16(x.bits, synth.bf16_bits_to_f64(x.bits))
    lens = np.arange(batch, dtype=np.int32) * 3
    pend = np.array([1, 2, 3, 4, 0, 1, 2, 3], dtype=np.int32)
    d_len, d_n = i32(lens), i32(pend)
    tok, conf, n = mars.accept_deferred(dev_bf16(x), tau, d_len, d_n, cap, batch_min=True)
    torch.cuda.synchronize()
    t_o, c_o, n_o = oracle.accept(x.f64, tau, "prob", batch_min=True)
    assert np.array_equal(tok.cpu().numpy(), t_o)
    assert np.array_equal(n.cpu().numpy(), n_o) and int(n_o[0]) >= 2
    assert np.array_equal(d_len.cpu().numpy(), lens + pend)


def test_accept_deferred_capacity():
    """cursor + new count past cap: commit 0 after advancing; a bad pending count keeps the cursor."""
    B, V, cap = 4, 500, 16
    x = synth.Bf16.from_float(np.tile(np.where(np.arange(V) == 3, 40.0, 0.0).astype(np.float32), (4, B, 1)))
    lens = np.array([0, 10, 14, 12], dtype=np.int32)
    pend = np.array([4, 3, 3, 9], dtype=np.int32)  # 13 + 4 > cap; 14 + 3 > cap; 9 > B
    d_len, d_n = i32(lens), i32(pend)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, _, n = mars.accept_deferred(dev_bf16(x), 0.5, d_len, d_n, cap, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == mars.MARS_DEV_CAPACITY
    assert n.cpu().tolist() == [4, 0, 0, 0]
    assert d_len.cpu().tolist() == [4, 13, 14, 12]  # advanced, advanced, kept, kept


# ---------------------------------------------------------------- several steps


def test_deferred_loop_matches_oracle():
    """Five steps of decode + accept with the cursor, the pending count and the
    cache carried on the device, against the oracle carrying the same state."""
    batch, B, hq, hkv, D, V, cap, tau = 6, 4, 8, 2, 64, 700, 256, 0.5
    rng = np.random.default_rng(2200)
    lens = rng.integers(0, 120, size=batch).astype(np.int32)
    pend = np.zeros(batch, dtype=np.int32)
    kc, vc = rand_bf16((batch, hkv, cap, D), 2201), rand_bf16((batch, hkv, cap, D), 2202)
    d_kc, d_vc, d_len, d_n = dev_bf16(kc), dev_bf16(vc), i32(lens), i32(pend)
    kc64, vc64 = kc.f64, vc.f64
    ws = mars.accept_workspace(batch, B, V, "cuda")
    for step in range(5):
        seed = 2300 + 10 * step
        q = rand_bf16((batch, 2 * B, hq, D), seed)
        kn, vn = rand_bf16((batch, 2 * B, hkv, D), seed + 1), rand_bf16((batch, 2 * B, hkv, D), seed + 2)
        x = spiked(batch, B, V, seed + 3)
        o = mars.decode_attn_deferred(dev_bf16(q), dev_bf16(kn), dev_bf16(vn), d_kc, d_vc, d_len, d_n, cap - 2 * B)
        tok, conf, n = mars.accept_deferred(dev_bf16(x), tau, d_len, d_n, cap, workspace=ws)
        torch.cuda.synchronize()
        o_o, kc64, vc64 = oracle.decode_attn_deferred(q.f64, kn.f64, vn.f64, kc64, vc64, lens, pend, D ** -0.5)
        t_o, c_o, n_o, lens = oracle.accept_deferred(x.f64, tau, lens, pend, "prob")
        got = bf16_to_f64(o)
        for b in range(batch):
            valid = [c for c in range(2 * B) if c < pend[b] or c >= B]
            assert max_abs(got[b, valid], o_o[b, valid]) <= ATTN_TOL, (step, b)
        assert np.array_equal(tok.cpu().numpy(), t_o)
        assert np.array_equal(n.cpu().numpy(), n_o), step
        assert np.array_equal(d_len.cpu().numpy(), lens), step
        pend = n_o.astype(np.int32)
        assert np.array_equal(bf16_to_f64(d_kc), kc64) and np.array_equal(bf16_to_f64(d_vc), vc64), step
