"""mars_train_attn_bwd on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import token_decoding_gb300 as mars
from token_decoding_gb300 import synth
from tests.gpu_util import bf16_to_f64, dev_bf16

pytestmark = pytest.mark.gpu

# The outputs are bf16 (relative rounding 2^-9 ~ 2e-3) and P, dS are rounded to
# bf16 before the tensor-core products (relative 2^-9 per term, partly averaging
# over the sum): every gradient element is held to 1% of the largest magnitude of
# its tensor plus 1e-3 (measured on these shapes: at most 0.44%).
REL_TOL = 1e-2
ABS_TOL = 1e-3


def rand_bf16(shape, seed, sigma=1.0):
    g = np.random.default_rng(seed)
    return synth.Bf16.from_float(g.standard_normal(shape, dtype=np.float32) * np.float32(sigma))


def run(q, k, v, do, L, B, scale):
    dq_, dk_, dv_ = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    ddo = dev_bf16(do)
    o, lse = mars.train_attn(dq_, dk_, dv_, L, B, scale=scale, want_lse=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dq, dk, dv = mars.train_attn_bwd(dq_, dk_, dv_, o, ddo, lse, L, B, scale=scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return bf16_to_f64(dq), bf16_to_f64(dk), bf16_to_f64(dv)


def check(got, want, name):
    bound = REL_TOL * float(np.max(np.abs(want))) + ABS_TOL
    err = float(np.max(np.abs(got - want)))
    assert err <= bound, (name, err, bound)
    return err


def case(nb, L, B, hq, hkv, d, seed, heads=None):
    q = rand_bf16((nb, 2 * L, hq, d), seed)
    k, v = rand_bf16((nb, 2 * L, hkv, d), seed + 1), rand_bf16((nb, 2 * L, hkv, d), seed + 2)
    do = rand_bf16((nb, 2 * L, hq, d), seed + 3)
    scale = d ** -0.5
    dq, dk, dv = run(q, k, v, do, L, B, scale)
    if heads is None:
        want = oracle.train_attn_bwd(q.f64, k.f64, v.f64, do.f64, L, B, scale)
        got = (dq, dk, dv)
    else:  # one KV group of one sequence: its query heads only touch their KV head
        b, g = heads
        G = hq // hkv
        hs = slice(g * G, (g + 1) * G)
        want = oracle.train_attn_bwd(q.f64[b:b + 1, :, hs], k.f64[b:b + 1, :, g:g + 1], v.f64[b:b + 1, :, g:g + 1],
                                     do.f64[b:b + 1, :, hs], L, B, scale)
        got = (dq[b:b + 1, :, hs], dk[b:b + 1, :, g:g + 1], dv[b:b + 1, :, g:g + 1])
    return [check(x, w, n) for x, w, n in zip(got, want, ("dq", "dk", "dv"))]


def test_tiny():
    case(1, 64, 4, 1, 1, 64, 3000)


@pytest.mark.parametrize("D", [64, 128])
def test_ragged_and_gqa(D):
    """L not a multiple of B or of the 128-row tile; two query heads per KV head."""
    case(2, 200, 3, 4, 2, D, 3100 + D)


def test_several_tiles_d128():
    case(1, 300, 8, 2, 1, 128, 3200)


def test_block_ge_L():
    case(1, 50, 64, 2, 2, 64, 3300)


def test_group_of_seven_d128():
    case(1, 256, 4, 7, 1, 128, 3400)


def _shape_groups(s, seed, groups):
    """The full-size backward once on the GPU, then (sequence, KV group) slices
    against the oracle: a group's query heads only touch their own KV head."""
    q = rand_bf16((s.batch, 2 * s.L, s.Hq, s.D), seed)
    k, v = rand_bf16((s.batch, 2 * s.L, s.Hkv, s.D), seed + 1), rand_bf16((s.batch, 2 * s.L, s.Hkv, s.D), seed + 2)
    do = rand_bf16((s.batch, 2 * s.L, s.Hq, s.D), seed + 3)
    scale = s.D ** -0.5
    dq, dk, dv = run(q, k, v, do, s.L, s.B, scale)
    G = s.Hq // s.Hkv
    for b, g in groups:
        hs = slice(g * G, (g + 1) * G)
        want = oracle.train_attn_bwd(q.f64[b:b + 1, :, hs], k.f64[b:b + 1, :, g:g + 1], v.f64[b:b + 1, :, g:g + 1],
                                     do.f64[b:b + 1, :, hs], s.L, s.B, scale)
        got = (dq[b:b + 1, :, hs], dk[b:b + 1, :, g:g + 1], dv[b:b + 1, :, g:g + 1])
        for x, w, n in zip(got, want, ("dq", "dk", "dv")):
            check(x, w, f"{n} b{b} g{g}")


def test_qwen05b_shape_every_group():
    s = synth.TRAIN_05B
    _shape_groups(s, 3500, [(b, g) for b in range(s.batch) for g in range(s.Hkv)])


def test_qwen7b_shape_every_group():
    """Every (sequence, KV group) of the 7B shape.  Its dK/dV units split a group's
    seven query heads into 1 to 5 chunks depending on the key tile (5 for the first
    clean tile, 1 from the 14th and for every noisy one), so uneven chunks, whole
    groups written directly and the chunk reduction all meet the oracle here."""
    s = synth.TRAIN_7B
    _shape_groups(s, 3600, [(b, g) for b in range(s.batch) for g in range(s.Hkv)])


def test_deterministic():
    q = rand_bf16((1, 256, 2, 64), 3700)
    k, v = rand_bf16((1, 256, 1, 64), 3701), rand_bf16((1, 256, 1, 64), 3702)
    do = rand_bf16((1, 256, 2, 64), 3703)
    a = run(q, k, v, do, 128, 4, 0.125)
    b = run(q, k, v, do, 128, 4, 0.125)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
