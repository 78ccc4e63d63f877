"""mars_train_attn on the GPU against the fp64 oracle (Eq. 2 mask over [x ; x~])."""
import numpy as np
import pytest
import torch

import oracle
import token_decoding_gb300 as mars
from token_decoding_gb300 import synth
from tests.gpu_util import ATTN_TOL, bf16_to_f64, dev_bf16, max_abs

pytestmark = pytest.mark.gpu


def rand_bf16(shape, seed):
    g = np.random.default_rng(seed)
    return synth.Bf16.from_float(g.standard_normal(shape, dtype=np.float32))


def run_train(q, k, v, L, B, scale, want_lse=True):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = mars.train_attn(dev_bf16(q), dev_bf16(k), dev_bf16(v), L, B, scale=scale, want_lse=want_lse,
                             status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return bf16_to_f64(o), lse.cpu().numpy().astype(np.float64)


def case(batch, L, B, hq, hkv, D, seed, rows=None):
    q = rand_bf16((batch, 2 * L, hq, D), seed)
    k, v = rand_bf16((batch, 2 * L, hkv, D), seed + 1), rand_bf16((batch, 2 * L, hkv, D), seed + 2)
    scale = D ** -0.5
    o, lse = run_train(q, k, v, L, B, scale)
    o_ref, lse_ref = oracle.train_attn(q.f64, k.f64, v.f64, L, B, scale, rows=rows)
    sel = slice(None) if rows is None else np.asarray(rows)
    err = max_abs(o[:, sel], o_ref)
    assert err <= ATTN_TOL, err
    lerr = max_abs(lse[:, :, sel], lse_ref)
    assert lerr <= 1e-3, lerr
    return err


def test_tiny_training_step():
    s = synth.TINY_TRAIN
    q, k, v = synth.train_inputs(s)
    o, lse = run_train(q, k, v, s.L, s.B, s.D ** -0.5)
    o_ref, lse_ref = oracle.train_attn(q.f64, k.f64, v.f64, s.L, s.B, s.D ** -0.5)
    assert max_abs(o, o_ref) <= ATTN_TOL
    assert max_abs(lse, lse_ref) <= 1e-3


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("L,B", [(300, 4), (256, 8), (130, 3), (131, 5), (200, 6), (64, 1)])
def test_several_tiles_and_ragged_ends(L, B, D):
    case(2, L, B, 4, 2, D, 10 * L + B)


@pytest.mark.parametrize("L,B", [(300, 1), (300, 2), (257, 16), (384, 32), (200, 8)])
def test_own_block_tile_d64(L, B):
    """Block sizes that divide 32 with several query tiles at D = 64: the noisy query
    tiles after the first take the own-block path (only the warp's 32 columns of
    their last key tile are read); ragged last tiles included."""
    case(2, L, B, 6, 2, 64, 13 * L + B)


@pytest.mark.parametrize("L,B", [(10, 16), (100, 100), (129, 128), (260, 200), (128, 128), (1, 1), (5, 2)])
def test_degenerate_blocks(L, B):
    case(1, L, B, 2, 1, 64, 7 * L + B)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (28, 4), (14, 2), (8, 1)])
def test_head_layouts(hq, hkv):
    case(1, 200, 4, hq, hkv, 128 if hq == 28 else 64, hq * 31 + hkv)


def _full_shape(s):
    """Every row of every (sequence, head) slice against the oracle."""
    q, k, v = synth.train_inputs(s)
    o, lse = run_train(q, k, v, s.L, s.B, s.D ** -0.5)
    assert np.all(np.isfinite(o))
    G = s.Hq // s.Hkv
    worst = 0.0
    for b in range(s.batch):
        for g in range(s.Hkv):  # one KV group at a time keeps the oracle's memory small
            hs = slice(g * G, (g + 1) * G)
            o_ref, lse_ref = oracle.train_attn(q.f64[b:b + 1, :, hs], k.f64[b:b + 1, :, g:g + 1],
                                               v.f64[b:b + 1, :, g:g + 1], s.L, s.B, s.D ** -0.5)
            err = max_abs(o[b:b + 1, :, hs], o_ref)
            assert err <= ATTN_TOL, (b, g, err)
            assert max_abs(lse[b:b + 1, hs], lse_ref) <= 1e-3, (b, g)
            worst = max(worst, err)
    print(f"{s.name}: worst |delta| over all rows {worst:.3g}")


def test_qwen05b_shaped_training_all_rows():
    _full_shape(synth.TRAIN_05B)


def test_qwen7b_shaped_training_all_rows():
    _full_shape(synth.TRAIN_7B)


def test_noisy_blocks_match_decode_kernel():
    """Noisy block k of the training forward is a decode step over cache = clean
    K/V of blocks < k and new = that block's placeholders (both kernels on GPU)."""
    L, B, hq, hkv, D = 192, 8, 8, 2, 128
    q = rand_bf16((1, 2 * L, hq, D), 50)
    k, v = rand_bf16((1, 2 * L, hkv, D), 51), rand_bf16((1, 2 * L, hkv, D), 52)
    scale = D ** -0.5
    o_train, _ = run_train(q, k, v, L, B, scale)
    dq, dk, dv = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    kc = dk[0, :L].permute(1, 0, 2).unsqueeze(0).contiguous()   # [1, Hkv, L, D]
    vc = dv[0, :L].permute(1, 0, 2).unsqueeze(0).contiguous()
    for kb in (0, 1, 5, L // B - 1):
        n = kb * B
        rows = slice(L + n, L + n + B)
        lens = torch.tensor([n], dtype=torch.int32, device="cuda")
        o_dec = mars.decode_attn(dq[:, rows].contiguous(), dk[:, rows].contiguous(), dv[:, rows].contiguous(),
                                 kc, vc, lens, L, scale=scale)
        torch.cuda.synchronize()
        assert max_abs(bf16_to_f64(o_dec), o_train[:, rows]) <= ATTN_TOL


def test_deterministic():
    q = rand_bf16((1, 512, 4, 64), 60)
    k, v = rand_bf16((1, 512, 2, 64), 61), rand_bf16((1, 512, 2, 64), 62)
    a, _ = run_train(q, k, v, 256, 4, 0.125)
    b, _ = run_train(q, k, v, 256, 4, 0.125)
    assert np.array_equal(a, b)
