"""mars_decode_attn on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import token_decoding_gb300 as mars
from token_decoding_gb300 import synth
from tests.gpu_util import ATTN_TOL, bf16_to_f64, dev_bf16, max_abs

pytestmark = pytest.mark.gpu


def rand_bf16(shape, seed, sigma=1.0):
    g = np.random.default_rng(seed)
    return synth.Bf16.from_float(g.standard_normal(shape, dtype=np.float32) * np.float32(sigma))


def run_decode(q, kn, vn, kc, vc, lens, max_len, scale, status=None):
    d_len = torch.from_numpy(np.asarray(lens, dtype=np.int32)).cuda()
    o = mars.decode_attn(dev_bf16(q), dev_bf16(kn), dev_bf16(vn), dev_bf16(kc), dev_bf16(vc), d_len, max_len,
                         scale=scale, status=status)
    torch.cuda.synchronize()
    return bf16_to_f64(o)


def case(batch, B, hq, hkv, D, cap, lens, seed, max_len=None, sample=None):
    q = rand_bf16((batch, B, hq, D), seed)
    kn, vn = rand_bf16((batch, B, hkv, D), seed + 1), rand_bf16((batch, B, hkv, D), seed + 2)
    kc, vc = rand_bf16((batch, hkv, cap, D), seed + 3), rand_bf16((batch, hkv, cap, D), seed + 4)
    lens = np.asarray(lens, dtype=np.int32)
    scale = D ** -0.5
    got = run_decode(q, kn, vn, kc, vc, lens, cap if max_len is None else max_len, scale)
    bs = np.arange(batch) if sample is None else np.asarray(sample)
    want = oracle.decode_attn(q.f64[bs], kn.f64[bs], vn.f64[bs], kc.f64[bs], vc.f64[bs], lens[bs], scale)
    err = max_abs(got[bs], want)
    assert err <= ATTN_TOL, err
    return err


def test_tiny_decode_step():
    s = synth.TINY_DECODE
    case(1, s.B, s.Hq, s.Hkv, s.D, s.cap, [60], 100)


def test_batch1_7b_shapes():
    s = synth.DECODE_7B_B1
    case(1, s.B, s.Hq, s.Hkv, s.D, 2048 + 64, [2048], 200)


def test_batch64_7b_shapes_sampled():
    s = synth.DECODE_7B_B64
    lens = synth.initial_cache_lens(s)
    order = np.argsort(-lens, kind="stable")
    sample = sorted(set(order[:3].tolist() + order[-3:].tolist() + [0, 17, 40, 63]))
    case(s.batch, s.B, s.Hq, s.Hkv, s.D, 4096 + 16, lens, 300, max_len=4096, sample=sample)


@pytest.mark.parametrize("lens", [[0, 1], [63, 64], [65, 127], [128, 200]])
def test_cache_lengths_around_tiles(lens):
    case(2, 4, 8, 2, 128, 256, lens, 400)


@pytest.mark.parametrize("B", [1, 2, 3, 8, 16])
def test_block_sizes(B):
    case(3, B, 14, 2, 64, 300, [0, 100, 290], 500 + B)


@pytest.mark.parametrize("hq,hkv,D", [(4, 4, 64), (12, 3, 128), (32, 2, 128), (16, 1, 64)])
def test_head_layouts(hq, hkv, D):
    """Includes units wider than 128 rows (16 heads x 16 positions) split into head chunks."""
    B = 16 if hq // hkv >= 16 else 4
    case(2, B, hq, hkv, D, 520, [513, 7], 600 + hq)


def test_many_sequences_unsorted_order():
    """More sequences than the heavy-first ranking handles: plain index order."""
    rng = np.random.default_rng(7)
    lens = rng.integers(0, 100, size=300)
    case(300, 4, 4, 1, 64, 112, lens, 700, sample=[0, 1, 150, 299])


@pytest.mark.parametrize("batch,B,hq,hkv,D,lens", [
    (3, 4, 28, 4, 128, [0, 700, 2040]),   # 28 rows: owners 14 and 15 hold no rows
    (2, 4, 14, 2, 64, [1, 1999]),          # D = 64, one sequence with a single cache key
    (1, 1, 17, 1, 64, [1100]),             # 17 rows (odd), one position
    (2, 2, 16, 1, 128, [64, 1024]),        # 32 rows, cache lengths on tile boundaries
])
def test_wide_cluster_small_units(batch, B, hq, hkv, D, lens):
    """Small units (<= 32 rows) with few units and a long max_len run as 16-CTA
    clusters where the device schedules them: ranks past a short sequence's tiles hold
    no keys and ranks past the rows own none."""
    case(batch, B, hq, hkv, D, 2048 + 64, lens, 750 + hq + D, max_len=2048)


def test_max_len_equals_cap():
    case(1, 4, 7, 1, 128, 1000, [1000], 800, max_len=1000)


def test_cache_len_out_of_range_is_reported():
    q = rand_bf16((2, 4, 4, 64), 900)
    kn, vn = rand_bf16((2, 4, 2, 64), 901), rand_bf16((2, 4, 2, 64), 902)
    kc, vc = rand_bf16((2, 2, 64, 64), 903), rand_bf16((2, 2, 64, 64), 904)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_decode(q, kn, vn, kc, vc, [10, 50], 40, 0.125, status=status)
    assert int(status.item()) & mars.MARS_DEV_LEN_RANGE
    assert np.all(got[1] == 0)
    want = oracle.decode_attn(q.f64[:1], kn.f64[:1], vn.f64[:1], kc.f64[:1], vc.f64[:1], [10], 0.125)
    assert max_abs(got[:1], want) <= ATTN_TOL


def test_deterministic_across_calls():
    s = synth.DECODE_7B_B1
    q = rand_bf16((1, 4, 28, 128), 1000)
    kn, vn = rand_bf16((1, 4, 4, 128), 1001), rand_bf16((1, 4, 4, 128), 1002)
    kc, vc = rand_bf16((1, 4, 2100, 128), 1003), rand_bf16((1, 4, 2100, 128), 1004)
    a = run_decode(q, kn, vn, kc, vc, [2048], 2100, 128 ** -0.5)
    b = run_decode(q, kn, vn, kc, vc, [2048], 2100, 128 ** -0.5)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("D", [64, 128])
def test_cache_beyond_len_holds_nan(D):
    """What the cache holds at or past cache_len (here NaN) never reaches the output."""
    batch, B, hq, hkv, cap = 2, 4, 8, 2, 256
    lens = np.asarray([70, 129], dtype=np.int32)
    q = rand_bf16((batch, B, hq, D), 1100)
    kn, vn = rand_bf16((batch, B, hkv, D), 1101), rand_bf16((batch, B, hkv, D), 1102)
    kc, vc = rand_bf16((batch, hkv, cap, D), 1103), rand_bf16((batch, hkv, cap, D), 1104)
    for t in (kc, vc):
        for b in range(batch):
            t.bits[b, :, lens[b]:, :] = 0x7FC0  # bf16 quiet NaN
            t.f64[b, :, lens[b]:, :] = np.nan
    scale = D ** -0.5
    got = run_decode(q, kn, vn, kc, vc, lens, cap, scale)
    assert np.all(np.isfinite(got))
    want = oracle.decode_attn(q.f64, kn.f64, vn.f64, kc.f64, vc.f64, lens, scale)
    assert max_abs(got, want) <= ATTN_TOL
