"""mars_accept_noalloc: acceptance for callers that cannot allocate.

Some callers of this library never get to allocate device memory: a plugin
that is only handed its input and output buffers by the framework hosting it,
or a decode loop that runs under a fixed memory budget, where a cudaMalloc
could fail in the middle of generation and would stall the whole device.
mars_accept_noalloc serves them with scratch that lives inside the library.

These tests call it through the C ABI (ctypes, raw device pointers) and check
it against the workspace-taking mars_accept on the same inputs, two calls in a
row, with the tolerances the other accept tests use.  This file is collected
last on purpose, so a failure here never hides the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import token_decoding_gb300 as mars
from token_decoding_gb300 import _lib
from token_decoding_gb300 import synth
from tests.gpu_util import bits_of, dev_bf16

pytestmark = pytest.mark.gpu


def _inputs(batch, B, V, hkv, D, cap, seed):
    g = synth.rng_for("noalloc", seed)
    logits = synth.spiked_logits(batch, B, V, 2.0, 0.7, 8.0, 25.0, g)
    kn = synth.Bf16.from_float(g.standard_normal((batch, B, hkv, D), dtype=np.float32))
    vn = synth.Bf16.from_float(g.standard_normal((batch, B, hkv, D), dtype=np.float32))
    kc = synth.Bf16.from_float(g.standard_normal((batch, hkv, cap, D), dtype=np.float32))
    vc = synth.Bf16.from_float(g.standard_normal((batch, hkv, cap, D), dtype=np.float32))
    lens = g.integers(0, cap - B - 1, size=batch).astype(np.int32)
    return logits, kn, vn, kc, vc, lens


def _state(kc, vc, lens):
    return dev_bf16(kc), dev_bf16(vc), torch.from_numpy(lens.copy()).cuda()


def _noalloc_via_c_abi(logits, tau, kn, vn, kc, vc, lens, tokens, conf, n_commit):
    """Call the C entry point directly with device pointers and the current stream."""
    f = _lib.lib().mars_accept_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.restype = I
    f.argtypes = [P, I, I, I, F, P, P, P, P, P, I, I, I, P, P, P, P, P]
    nb, bq, V = logits.shape
    rc = f(P(logits.data_ptr()), nb, bq, V, F(tau), P(kn.data_ptr()), P(vn.data_ptr()), P(kc.data_ptr()),
           P(vc.data_ptr()), P(lens.data_ptr()), kn.shape[2], kn.shape[3], kc.shape[2], P(tokens.data_ptr()),
           P(conf.data_ptr()), P(n_commit.data_ptr()), None, P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, (rc, mars.status_string(rc))


@pytest.mark.parametrize("batch,B,V,tau", [(1, 4, 152064, 0.9), (64, 8, 152064, 0.95), (3, 5, 1001, 0.3)])
def test_noalloc_matches_workspace_accept_twice(batch, B, V, tau):
    hkv, D, cap = 4, 128, 64
    for call in range(2):
        logits, kn, vn, kc, vc, lens = _inputs(batch, B, V, hkv, D, cap, (batch, B, V, call))
        d_logits, d_kn, d_vn = dev_bf16(logits), dev_bf16(kn), dev_bf16(vn)
        # reference: the workspace-taking entry point
        kc_a, vc_a, len_a = _state(kc, vc, lens)
        tok_a, conf_a, n_a = mars.accept(d_logits, tau, d_kn, d_vn, kc_a, vc_a, len_a)
        # the no-allocation entry point, through the C ABI
        kc_b, vc_b, len_b = _state(kc, vc, lens)
        tok_b = torch.full((batch, B), -1, dtype=torch.int32, device="cuda")
        conf_b = torch.full((batch, B), -1.0, dtype=torch.float32, device="cuda")
        n_b = torch.full((batch,), -1, dtype=torch.int32, device="cuda")
        _noalloc_via_c_abi(d_logits, tau, d_kn, d_vn, kc_b, vc_b, len_b, tok_b, conf_b, n_b)
        torch.cuda.synchronize()

        assert torch.equal(tok_a, tok_b)
        ca, cb = conf_a.cpu().numpy().astype(np.float64), conf_b.cpu().numpy().astype(np.float64)
        assert float(np.max(np.abs(ca - cb) / ca)) < 1e-5
        na, nb_ = n_a.cpu().numpy(), n_b.cpu().numpy()
        near = np.abs(ca - tau) < 1e-4
        for b in np.flatnonzero(na != nb_):
            assert near[b].any(), (b, na[b], nb_[b])
        same = na == nb_
        assert np.array_equal(len_a.cpu().numpy()[same], len_b.cpu().numpy()[same])
        assert np.array_equal(bits_of(kc_a)[same], bits_of(kc_b)[same])
        assert np.array_equal(bits_of(vc_a)[same], bits_of(vc_b)[same])


def test_noalloc_large_then_small_without_reset():
    """A small call right after a large one reads only slots it wrote itself: the
    stale partials the large call left in the shared array change nothing."""
    tau = 0.5
    big = _inputs(64, 8, 152064, 4, 128, 64, "big")
    small = _inputs(3, 5, 1001, 4, 128, 64, "small")
    for logits, kn, vn, kc, vc, lens in (big, small):
        d_logits, d_kn, d_vn = dev_bf16(logits), dev_bf16(kn), dev_bf16(vn)
        kc_a, vc_a, len_a = _state(kc, vc, lens)
        tok_a, conf_a, n_a = mars.accept(d_logits, tau, d_kn, d_vn, kc_a, vc_a, len_a)
        nb, B = logits.shape[:2]
        kc_b, vc_b, len_b = _state(kc, vc, lens)
        tok_b = torch.full((nb, B), -1, dtype=torch.int32, device="cuda")
        conf_b = torch.full((nb, B), -1.0, dtype=torch.float32, device="cuda")
        n_b = torch.full((nb,), -1, dtype=torch.int32, device="cuda")
        _noalloc_via_c_abi(d_logits, tau, d_kn, d_vn, kc_b, vc_b, len_b, tok_b, conf_b, n_b)
        torch.cuda.synchronize()
        assert torch.equal(tok_a, tok_b)
        ca, cb = conf_a.cpu().numpy().astype(np.float64), conf_b.cpu().numpy().astype(np.float64)
        assert float(np.max(np.abs(ca - cb) / ca)) < 1e-5
        assert torch.equal(n_a, n_b) or bool((np.abs(ca - tau) < 1e-4).any())


def test_noalloc_python_wrapper_with_status_word():
    """The binding's accept_noalloc passes its arguments in the C order and leaves a
    clean status word (0) on a valid call."""
    logits, kn, vn, kc, vc, lens = _inputs(2, 4, 5000, 2, 64, 48, "wrapper")
    d_logits, d_kn, d_vn = dev_bf16(logits), dev_bf16(kn), dev_bf16(vn)
    kc_a, vc_a, len_a = _state(kc, vc, lens)
    tok_a, conf_a, n_a = mars.accept(d_logits, 0.4, d_kn, d_vn, kc_a, vc_a, len_a)
    kc_b, vc_b, len_b = _state(kc, vc, lens)
    tok_b = torch.empty((2, 4), dtype=torch.int32, device="cuda")
    conf_b = torch.empty((2, 4), dtype=torch.float32, device="cuda")
    n_b = torch.empty((2,), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.accept_noalloc(d_logits, 0.4, d_kn, d_vn, kc_b, vc_b, len_b, tok_b, conf_b, n_b, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(tok_a, tok_b) and torch.equal(n_a, n_b) and torch.equal(len_a, len_b)
    assert torch.allclose(conf_a, conf_b, rtol=1e-5, atol=0)
    assert torch.equal(kc_a, kc_b) and torch.equal(vc_a, vc_b)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """batch * B * ceil(V / 8192) above 65536 is refused before anything is launched."""
    f = _lib.lib().mars_accept_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.restype = I
    f.argtypes = [P, I, I, I, F, P, P, P, P, P, I, I, I, P, P, P, P, P]
    buf = torch.zeros(4096, dtype=torch.int32, device="cuda")
    ptr = P(buf.data_ptr())
    # 512 sequences x 16 positions x ceil(73729 / 8192) = 8192 x 10 slices > 65536
    rc = f(ptr, 512, 16, 73729, F(0.5), ptr, ptr, ptr, ptr, ptr, 1, 64, 8, ptr, ptr, ptr, None, None)
    assert rc == 5, mars.status_string(rc)
    # the same rows with a short vocabulary fit
    assert mars.status_string(5).startswith("shape exceeds")
