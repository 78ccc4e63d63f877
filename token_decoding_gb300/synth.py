"""Seeded synthetic inputs shared by the tests, the bench and the oracle legs.

This module only draws random numbers and rounds them to bf16: it holds none
of the method's arithmetic.  Every array comes out twice, as bf16 bit
patterns (``uint16``, what the CUDA library reads) and as the exactly widened
float64 values (what the oracle reads), so both sides see identical inputs.

Randomness is numpy's PCG64 seeded from (master seed, workload, step), which
is reproducible across x86 and Arm hosts.

The shapes follow the Qwen2.5-0.5B / 7B workloads that the MARS pages run on
("MARS: Enabling Autoregressive Models Multi-Token Generation", Sec. 4 setup;
the authors' blog post, "Where it stands against the alternatives": a
152k-vocabulary LM head).  The benchmark datasets themselves are not used:
q/k/v are N(0, 1), and logits are scaled N(0, 1) noise with one spiked token
at a random subset of positions, which is what makes some positions
confident and others not.
"""

from __future__ import annotations

import dataclasses
import zlib

import numpy as np

MASTER_SEED = 0


# --------------------------------------------------------------------------
# bf16 helpers (input preparation only)
# --------------------------------------------------------------------------

def to_bf16_bits(x) -> np.ndarray:
    """Round float values to bf16 (round-to-nearest-even); returns uint16 bits."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    return r


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@dataclasses.dataclass
class Bf16:
    """One bf16 tensor: bit patterns and their exact float64 values."""

    bits: np.ndarray
    f64: np.ndarray

    @classmethod
    def from_float(cls, x) -> "Bf16":
        bits = to_bf16_bits(x)
        return cls(bits=bits, f64=bf16_bits_to_f64(bits))

    @property
    def shape(self):
        return self.bits.shape


def rng_for(*key) -> np.random.Generator:
    """A PCG64 generator seeded from the master seed and a tuple of labels."""
    h = zlib.crc32(repr((MASTER_SEED,) + tuple(key)).encode())
    return np.random.default_rng([MASTER_SEED, h])


# --------------------------------------------------------------------------
# Workload shapes
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class TrainShape:
    name: str
    batch: int
    L: int
    B: int
    Hq: int
    Hkv: int
    D: int

    @property
    def useful_flops(self) -> int:
        """Multiply-adds x 2 over the L(L+1) visible (query, key) pairs, QK and PV."""
        return 4 * self.D * self.Hq * self.batch * self.L * (self.L + 1)


@dataclasses.dataclass(frozen=True)
class DecodeShape:
    name: str
    batch: int
    B: int
    Hq: int
    Hkv: int
    D: int
    V: int
    cap: int
    len_lo: int
    len_hi: int
    steps: int
    spike_prob: float
    spike_lo: float
    spike_hi: float
    base_sigma: float
    taus: tuple


# Tiny step: 1 sequence, L=64, B=4, 1/1 heads, D=64; decode over a 60-token cache.
TINY_TRAIN = TrainShape("tiny-train-L64-B4-h1-d64", 1, 64, 4, 1, 1, 64)
TINY_DECODE = DecodeShape("tiny-decode-len60-B4-V1000", 1, 4, 1, 1, 64, 1000,
                          cap=128, len_lo=60, len_hi=60, steps=1,
                          spike_prob=0.5, spike_lo=8.0, spike_hi=8.0, base_sigma=3.0,
                          taus=(1.0, 0.9, 0.0))
# Qwen2.5-0.5B-shaped training-mask attention.
TRAIN_05B = TrainShape("qwen2.5-0.5b-train-b4-L1024-B4-h14/2-d64", 4, 1024, 4, 14, 2, 64)
# Qwen2.5-7B-shaped training-mask attention.
TRAIN_7B = TrainShape("qwen2.5-7b-train-b2-L2048-B8-h28/4-d128", 2, 2048, 8, 28, 4, 128)
# Qwen2.5-7B-shaped decode at batch 1, 256 sliding-window steps.
DECODE_7B_B1 = DecodeShape("qwen2.5-7b-decode-b1-len2048-B4-V152064", 1, 4, 28, 4, 128, 152064,
                           cap=2048 + 256 * 4, len_lo=2048, len_hi=2048, steps=256,
                           spike_prob=0.6, spike_lo=10.0, spike_hi=10.0, base_sigma=2.0,
                           taus=(1.0, 0.95, 0.9, 0.5))
# Qwen2.5-7B-shaped batched decode: 64 sequences, varlen caches, 128 steps.
DECODE_7B_B64 = DecodeShape("qwen2.5-7b-decode-b64-len256..4096-B8-V152064", 64, 8, 28, 4, 128, 152064,
                            cap=4096 + 128 * 8, len_lo=256, len_hi=4096, steps=128,
                            spike_prob=0.5, spike_lo=4.0, spike_hi=12.0, base_sigma=2.0,
                            taus=(0.95,))


# --------------------------------------------------------------------------
# Generators
# --------------------------------------------------------------------------

def train_inputs(shape: TrainShape, seed_key=0):
    """q [b, 2L, Hq, D], k, v [b, 2L, Hkv, D], all bf16 ~ N(0, 1)."""
    g = rng_for("train", shape.name, seed_key)
    n2 = 2 * shape.L
    q = Bf16.from_float(g.standard_normal((shape.batch, n2, shape.Hq, shape.D), dtype=np.float32))
    k = Bf16.from_float(g.standard_normal((shape.batch, n2, shape.Hkv, shape.D), dtype=np.float32))
    v = Bf16.from_float(g.standard_normal((shape.batch, n2, shape.Hkv, shape.D), dtype=np.float32))
    return q, k, v


def initial_cache_lens(shape: DecodeShape, seed_key=0) -> np.ndarray:
    """Committed cache length per sequence, uniform in [len_lo, len_hi]."""
    g = rng_for("cache_len", shape.name, seed_key)
    return g.integers(shape.len_lo, shape.len_hi + 1, size=shape.batch).astype(np.int32)


def cache_inputs(shape: DecodeShape, seed_key=0, fill_len=None):
    """k_cache, v_cache [b, Hkv, cap, D] bf16 ~ N(0, 1).

    Only the first ``fill_len`` positions are drawn (the rest stay zero);
    positions beyond a sequence's committed length are never read.
    """
    g = rng_for("cache", shape.name, seed_key)
    fill = shape.cap if fill_len is None else int(fill_len)
    kc = np.zeros((shape.batch, shape.Hkv, shape.cap, shape.D), dtype=np.float32)
    vc = np.zeros_like(kc)
    kc[:, :, :fill, :] = g.standard_normal((shape.batch, shape.Hkv, fill, shape.D), dtype=np.float32)
    vc[:, :, :fill, :] = g.standard_normal((shape.batch, shape.Hkv, fill, shape.D), dtype=np.float32)
    return Bf16.from_float(kc), Bf16.from_float(vc)


def step_inputs(shape: DecodeShape, step: int, seed_key=0):
    """Per-step q [b, B, Hq, D], k_new, v_new [b, B, Hkv, D] bf16 ~ N(0, 1)."""
    g = rng_for("step", shape.name, seed_key, step)
    q = Bf16.from_float(g.standard_normal((shape.batch, shape.B, shape.Hq, shape.D), dtype=np.float32))
    kn = Bf16.from_float(g.standard_normal((shape.batch, shape.B, shape.Hkv, shape.D), dtype=np.float32))
    vn = Bf16.from_float(g.standard_normal((shape.batch, shape.B, shape.Hkv, shape.D), dtype=np.float32))
    return q, kn, vn


def spiked_logits(batch, B, V, base_sigma, spike_prob, spike_lo, spike_hi, g,
                  exact_spike_count=None):
    """logits [batch, B, V] = base_sigma * N(0, 1), plus a spike on one uniform
    token at a random subset of positions.

    With ``exact_spike_count`` set, exactly that many of the B positions of
    each sequence are spiked; otherwise each position is spiked with
    probability ``spike_prob``.  Spike heights are uniform in
    [spike_lo, spike_hi].
    """
    x = g.standard_normal((batch, B, V), dtype=np.float32) * np.float32(base_sigma)
    for b in range(batch):
        if exact_spike_count is not None:
            pos = g.choice(B, size=exact_spike_count, replace=False)
            spiked = np.zeros(B, dtype=bool)
            spiked[pos] = True
        else:
            spiked = g.random(B) < spike_prob
        for i in range(B):
            if spiked[i]:
                tok = g.integers(0, V)
                x[b, i, tok] += np.float32(g.uniform(spike_lo, spike_hi))
    return Bf16.from_float(x)


def step_logits(shape: DecodeShape, step: int, seed_key=0, spike_lo=None, spike_hi=None):
    """This step's logits [b, B, V] for a decode workload."""
    g = rng_for("logits", shape.name, seed_key, step)
    lo = shape.spike_lo if spike_lo is None else spike_lo
    hi = shape.spike_hi if spike_hi is None else spike_hi
    exact = None
    if shape is TINY_DECODE:
        # half of the positions, chosen at random: exactly B / 2 of them.
        exact = shape.B // 2
    return spiked_logits(shape.batch, shape.B, shape.V, shape.base_sigma, shape.spike_prob,
                         lo, hi, g, exact_spike_count=exact)


# --------------------------------------------------------------------------
# Per-sequence draws (sliding-window episodes checked on a subset of sequences)
# --------------------------------------------------------------------------
# Sequences of a decode batch are independent, so an episode can be checked on
# a few of them: these generators draw one sequence's arrays from a seed of its
# own (workload, sequence, step), so that the sequences under check never need
# the whole batch drawn on the host.

def seq_cache_inputs(shape: DecodeShape, b: int, fill_len: int, seed_key=0):
    """k_cache, v_cache [1, Hkv, cap, D] of sequence b; rows past fill_len are zero."""
    g = rng_for("seq_cache", shape.name, seed_key, b)
    kc = np.zeros((1, shape.Hkv, shape.cap, shape.D), dtype=np.float32)
    vc = np.zeros_like(kc)
    kc[:, :, :fill_len, :] = g.standard_normal((1, shape.Hkv, fill_len, shape.D), dtype=np.float32)
    vc[:, :, :fill_len, :] = g.standard_normal((1, shape.Hkv, fill_len, shape.D), dtype=np.float32)
    return Bf16.from_float(kc), Bf16.from_float(vc)


def seq_step_inputs(shape: DecodeShape, step: int, b: int, seed_key=0):
    """This step's q [1, B, Hq, D], k_new, v_new [1, B, Hkv, D] of sequence b."""
    g = rng_for("seq_step", shape.name, seed_key, step, b)
    q = Bf16.from_float(g.standard_normal((1, shape.B, shape.Hq, shape.D), dtype=np.float32))
    kn = Bf16.from_float(g.standard_normal((1, shape.B, shape.Hkv, shape.D), dtype=np.float32))
    vn = Bf16.from_float(g.standard_normal((1, shape.B, shape.Hkv, shape.D), dtype=np.float32))
    return q, kn, vn


def seq_step_logits(shape: DecodeShape, step: int, b: int, seed_key=0, spike_lo=None, spike_hi=None,
                    spike_prob=None):
    """This step's logits [1, B, V] of sequence b (the workload's spike recipe unless overridden)."""
    g = rng_for("seq_logits", shape.name, seed_key, step, b)
    lo = shape.spike_lo if spike_lo is None else spike_lo
    hi = shape.spike_hi if spike_hi is None else spike_hi
    prob = shape.spike_prob if spike_prob is None else spike_prob
    return spiked_logits(1, shape.B, shape.V, shape.base_sigma, prob, lo, hi, g)
