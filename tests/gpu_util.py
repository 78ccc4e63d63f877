"""Helpers for the GPU parity tests: move seeded inputs to the device and compare."""
import numpy as np
import torch


def dev_bf16(x, device="cuda"):
    """A synth.Bf16 (or uint16 bit array) as a contiguous bf16 CUDA tensor."""
    bits = x.bits if hasattr(x, "bits") else x
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def bf16_to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def bits_of(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def max_abs(a, b):
    return float(np.max(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64))))


ATTN_TOL = 1e-2  # max |delta| for bf16 outputs with fp32 accumulation


def check_accept(tokens, conf, n_commit, logits64, tau, gate="prob"):
    """Compare a GPU accept result with the fp64 oracle.

    Tokens must match exactly; conf to 1e-5 relative (top-1 probability) or
    2e-6 absolute (margin p1 - p2, which is 0 on ties).  A commit count may
    differ only where the first position whose pass/fail decision differs has
    an fp64 confidence within 1e-4 of tau; such positions are returned as a
    report (b, position) instead of failing.
    """
    import oracle

    t_o, c_o, n_o = oracle.accept(logits64, tau, gate)
    assert np.array_equal(tokens, t_o), np.argwhere(tokens != t_o)[:8]
    if gate == "prob":
        rel = np.abs(conf.astype(np.float64) - c_o) / c_o
        assert float(rel.max()) < 1e-5, float(rel.max())
    else:
        err = np.abs(conf.astype(np.float64) - c_o)
        assert float(err.max()) < 2e-6, float(err.max())
    near = oracle.near_threshold(c_o, tau)
    report = []
    for b in range(n_o.shape[0]):
        if int(n_commit[b]) == int(n_o[b]):
            continue
        gpu_pass = conf[b].astype(np.float32) >= np.float32(tau)
        or_pass = c_o[b] >= tau
        diff = np.flatnonzero(gpu_pass != or_pass)
        assert diff.size > 0, (b, n_commit[b], n_o[b])
        first = int(diff[0])
        assert near[b, first], (b, first, c_o[b, first], tau)
        report.append((b, first))
    return n_o, report
