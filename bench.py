"""Benchmark of the MARS hot path on GB300 (one JSON line on rank 0).

One step runs every stage of the path on synthetic Qwen2.5-shaped inputs:
  * one decode step at batch 1 (cache 2048, B=4): decode attention + accept
  * mars_train_attn on the Qwen2.5-7B-shaped batch (b2, L=2048, B=8, 28/4, D=128)
  * mars_train_attn on the Qwen2.5-0.5B-shaped training batch (b4, L=1024,
    B=4, 14/2 heads, D=64)                          -> headline value, TFLOP/s
  * one sliding-window decode step at batch 64 (varlen caches 256..4096, B=8,
    28/4 heads, D=128, V=152064): mars_decode_attn then mars_accept (+ KV append)
Each decode step is launched as one CUDA graph per step, as a decode loop runs;
the training kernels are plain launches.  CUDA events on the launching stream
bracket every kernel and graph; inputs rotate over enough buffers that each
kernel's working set exceeds twice the L2, so nothing is served from a warm L2
between iterations.  The decode kernels' own rates come from graphs of
back-to-back launches of one kernel.

--impl reference times the fp64 CPU oracle (the reference arm: the plain CPU implementation)
on bounded samples of the same workload.
"""

from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "train-mask attn TFLOP/s; decode attn+accept GB/s & steps/s; % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 126 * 1024 * 1024
DECODE_TAU = 0.95
CONFIG = {
    "workload": ("mars step: train-mask attn Qwen2.5-0.5B shape (b4 L1024 B4 14/2 d64; headline value) + "
                 "train-mask attn Qwen2.5-7B shape (b2 L2048 B8 28/4 d128) + batched decode step "
                 "(b64, cache 256..4096, B8, 28/4 d128, V152064: decode attn + accept/append, tau 0.95) + "
                 "batch-1 decode step (cache 2048, B4, V152064)"),
    "l2": "inputs rotate over buffer sets so each kernel's working set is >= 2x L2",
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_sources_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "token_decoding_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic():
    """Per-launch DRAM bytes from the committed ncu capture, if the kernels are unchanged since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return {}
    if t.get("kernel_sources_sha") != kernel_sources_sha():
        return {}
    return t.get("traffic_bytes_per_launch", {})


# --------------------------------------------------------------------------
# distributed plumbing (replicas only: the path has no exchange step)
# --------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist, world):
    if world > 1:
        dist.barrier()


def max_over_ranks(dist, world, value, device):
    if world == 1:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, world, value, device):
    if world == 1:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons; only the samples whose
    timestamps fall inside the timed window (host wall clock) are reported."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile

        fd, self.path = tempfile.mkstemp(prefix="mars_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.PERIOD_MS)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return
        # the window opens only once the sampler is producing lines
        t0 = time.time()
        while time.time() - t0 < 10 and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    def stop(self, window):
        """window = (start, end) as datetime.datetime on the host clock."""
        import datetime

        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        outside = 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                    mhz, max_mhz = float(parts[2]), float(parts[3])
                except ValueError:
                    continue
                if not window[0] <= ts <= window[1]:
                    outside += 1
                    continue
                sm.append(mhz)
                smax.append(max_mhz)
                for name, val in zip(names, parts[6:10]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0, "samples_outside": outside,
                    "reasons": ["no samples in the timed window"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "period_ms": self.PERIOD_MS, "reasons": sorted(reasons)}


# --------------------------------------------------------------------------
# the GPU arm
# --------------------------------------------------------------------------

def roofline(bound, achieved, peak, unit, traffic):
    return {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic}


def spiked_logits_gpu(batch, B, V, sigma, prob, lo, hi, gen, device):
    import torch

    x = torch.randn((batch, B, V), generator=gen, device=device, dtype=torch.float32) * sigma
    spiked = torch.rand((batch, B), generator=gen, device=device) < prob
    tok = torch.randint(0, V, (batch, B), generator=gen, device=device)
    height = lo + (hi - lo) * torch.rand((batch, B), generator=gen, device=device)
    x.scatter_add_(2, tok.unsqueeze(-1), (height * spiked).unsqueeze(-1))
    return x.to(torch.bfloat16)


class TrainWork:
    def __init__(self, shape, device, gen, min_bytes):
        import torch

        s = shape
        self.s = s
        per = (2 * s.batch * 2 * s.L * (s.Hq + s.Hkv) * s.D) * 2   # q + o + k + v bytes
        self.nsets = max(1, -(-min_bytes // per))
        self.sets = []
        for _ in range(self.nsets):
            q = torch.randn((s.batch, 2 * s.L, s.Hq, s.D), generator=gen, device=device).to(torch.bfloat16)
            k = torch.randn((s.batch, 2 * s.L, s.Hkv, s.D), generator=gen, device=device).to(torch.bfloat16)
            v = torch.randn((s.batch, 2 * s.L, s.Hkv, s.D), generator=gen, device=device).to(torch.bfloat16)
            self.sets.append((q, k, v, torch.empty_like(q)))
        self.flops = s.useful_flops

    def run(self, mars, step):
        q, k, v, o = self.sets[step % self.nsets]
        mars.train_attn(q, k, v, self.s.L, self.s.B, o=o)


class DecodeWork:
    """One sliding-window decode step (decode attention, then accept + append)."""

    def __init__(self, shape, device, gen, min_bytes, steps_per_episode):
        import torch
        from token_decoding_gb300 import synth

        import token_decoding_gb300 as mars

        s = shape
        self.s = s
        lens0 = synth.initial_cache_lens(s)
        self.lens0_host = lens0.astype(np.int64)
        cache_bytes = int(lens0.sum()) * s.Hkv * s.D * 2 * 2
        per = cache_bytes + s.batch * s.B * s.V * 2
        self.nsets = max(1, -(-min_bytes // per))
        self.sets = []
        for _ in range(self.nsets):
            kc = torch.randn((s.batch, s.Hkv, s.cap, s.D), generator=gen, device=device).to(torch.bfloat16)
            vc = torch.randn((s.batch, s.Hkv, s.cap, s.D), generator=gen, device=device).to(torch.bfloat16)
            lens = torch.from_numpy(lens0.copy()).to(device)
            logits = spiked_logits_gpu(s.batch, s.B, s.V, s.base_sigma, s.spike_prob, s.spike_lo, s.spike_hi,
                                       gen, device)
            ws = mars.accept_workspace(s.batch, s.B, s.V, device)
            self.sets.append({"kc": kc, "vc": vc, "lens": lens, "logits": logits, "ws": ws})
        self.lens0 = torch.from_numpy(lens0.copy()).to(device)
        self.q = torch.randn((s.batch, s.B, s.Hq, s.D), generator=gen, device=device).to(torch.bfloat16)
        self.kn = torch.randn((s.batch, s.B, s.Hkv, s.D), generator=gen, device=device).to(torch.bfloat16)
        self.vn = torch.randn((s.batch, s.B, s.Hkv, s.D), generator=gen, device=device).to(torch.bfloat16)
        self.o = torch.empty_like(self.q)
        self.tokens = torch.empty((s.batch, s.B), dtype=torch.int32, device=device)
        self.conf = torch.empty((s.batch, s.B), dtype=torch.float32, device=device)
        self.episode = steps_per_episode
        self.max_len = s.cap - s.B

    def reset(self):
        """Start a new episode: every buffer set goes back to the initial cache lengths."""
        for st in self.sets:
            st["lens"].copy_(self.lens0)

    def run_decode(self, mars, step):
        st = self.sets[step % self.nsets]
        mars.decode_attn(self.q, self.kn, self.vn, st["kc"], st["vc"], st["lens"], self.max_len, o=self.o)

    def run_accept(self, mars, step, n_out, gate="prob", tau=DECODE_TAU):
        st = self.sets[step % self.nsets]
        mars.accept(st["logits"], tau, self.kn, self.vn, st["kc"], st["vc"], st["lens"], workspace=st["ws"],
                    tokens=self.tokens, conf=self.conf, n_commit=n_out, gate=gate)

    def byte_counts(self, records):
        """Algorithmic bytes of decode and accept per executed step, from the commit history."""
        s = self.s
        lens = {i: self.lens0_host.copy() for i in range(self.nsets)}
        dec, acc = [], []
        small = s.batch * s.B * (2 * s.Hkv + 2 * s.Hq) * s.D * 2
        for kind, set_idx, n in records:
            if kind == "reset":
                lens = {i: self.lens0_host.copy() for i in range(self.nsets)}
                continue
            L = lens[set_idx]
            dec.append(int(L.sum()) * s.Hkv * s.D * 2 * 2 + small)
            ncommit = n.astype(np.int64)
            acc.append(s.batch * s.B * s.V * 2 + int(ncommit.sum()) * s.Hkv * s.D * 2 * 2 * 2
                       + s.batch * s.B * 8 + s.batch * 8)
            lens[set_idx] = L + ncommit
        return dec, acc


def run_gpu(args, rank, world, local):
    import torch

    import token_decoding_gb300 as mars
    from token_decoding_gb300 import build as mars_build
    from token_decoding_gb300 import synth

    if not os.path.exists(mars._lib.LIB_PATH):
        mars_build.build()
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    dist = init_dist(world, "nccl")
    peaks, peak_src = load_peaks()
    gen = torch.Generator(device=device)
    gen.manual_seed(1234 + rank)
    min_bytes = 2 * L2_BYTES

    train05 = TrainWork(synth.TRAIN_05B, device, gen, min_bytes)
    train7 = TrainWork(synth.TRAIN_7B, device, gen, min_bytes)
    dec64 = DecodeWork(synth.DECODE_7B_B64, device, gen, min_bytes, steps_per_episode=synth.DECODE_7B_B64.steps)
    dec1 = DecodeWork(synth.DECODE_7B_B1, device, gen, min_bytes, steps_per_episode=synth.DECODE_7B_B1.steps)
    total = args.warmup + args.steps
    ncommit64 = torch.zeros((total, dec64.s.batch), dtype=torch.int32, device=device)
    ncommit1 = torch.zeros((total, dec1.s.batch), dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream()
    # One step: the batch-1 decode step, the two training shapes, then the batch-64
    # decode step.  Each decode step (decode attention + accept) is launched as one
    # CUDA graph per step, as a decode loop runs; the training kernels are plain
    # launches.  The host's launch calls stay ahead of the GPU, so no host gap lands
    # inside the events around a kernel or a graph.
    names = ["decode_step_b1", "train_7b", "train_05b", "decode_step_b64"]
    kernels = ["train_7b", "train_05b"]
    records64, records1 = [], []
    b1_graphs, b64_graphs = {}, {}

    def b1_calls(i):
        dec1.run_decode(mars, i)
        dec1.run_accept(mars, i, ncommit1[i])

    def b64_calls(i):
        dec64.run_decode(mars, i)
        dec64.run_accept(mars, i, ncommit64[i])

    def step(i, ev):
        if i % dec64.episode == 0:
            dec64.reset()
            records64.append(("reset", 0, None))
        if i % dec1.episode == 0:
            dec1.reset()
            records1.append(("reset", 0, None))
        if ev is not None:
            ev[0].record(stream)
        if i in b1_graphs:
            b1_graphs[i].replay()
        else:
            b1_calls(i)
        records1.append(("step", i % dec1.nsets, i))
        if ev is not None:
            ev[1].record(stream)
        train7.run(mars, i)
        if ev is not None:
            ev[2].record(stream)
        train05.run(mars, i)
        if ev is not None:
            ev[3].record(stream)
        if i in b64_graphs:
            b64_graphs[i].replay()
        else:
            b64_calls(i)
        records64.append(("step", i % dec64.nsets, i))
        if ev is not None:
            ev[4].record(stream)

    for i in range(args.warmup):
        step(i, None)
    torch.cuda.synchronize()
    # the decode steps of every timed step, captured ahead of the timed region
    pool = torch.cuda.graph_pool_handle()
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        for i in range(args.warmup, args.warmup + args.steps):
            for graphs, calls in ((b1_graphs, b1_calls), (b64_graphs, b64_calls)):
                g = torch.cuda.CUDAGraph()
                g.capture_begin(pool=pool)
                calls(i)
                g.capture_end()
                graphs[i] = g
    stream.wait_stream(cap)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    barrier(dist, world)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    win0 = datetime.datetime.now()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        step(args.warmup + k, events[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(dist, world)
    total_ms = t_start.elapsed_time(t_end)
    per_kernel_ms = {n: [events[k][j].elapsed_time(events[k][j + 1]) for k in range(args.steps)]
                     for j, n in enumerate(names)}
    total_ms = max_over_ranks(dist, world, total_ms, device)

    # algorithmic work of the timed steps
    n64 = ncommit64.cpu().numpy()
    n1 = ncommit1.cpu().numpy()

    def resolve(records, hist):
        out = []
        for kind, set_idx, i in records:
            out.append((kind, set_idx, None if kind == "reset" else hist[i]))
        return out

    dec64_b, acc64_b = dec64.byte_counts(resolve(records64, n64))
    dec1_b, acc1_b = dec1.byte_counts(resolve(records1, n1))
    timed = slice(args.warmup, args.warmup + args.steps)
    work = {
        "train_05b": ("tensor", [train05.flops] * args.steps, "TFLOP/s", 1e-12),
        "train_7b": ("tensor", [train7.flops] * args.steps, "TFLOP/s", 1e-12),
    }
    traffic = ncu_traffic()
    parts = {}
    for n in kernels:
        bound, units, unit, scale = work[n]
        ms = sum(per_kernel_ms[n])
        achieved = sum(units) * scale / (ms * 1e-3)
        peak = peaks["bf16_tflops"] if bound == "tensor" else peaks["hbm_gbs"]
        parts[n] = {
            "avg_us": round(ms / args.steps * 1e3, 3),
            "roofline": roofline(bound, achieved, peak, unit, traffic.get(n)),
        }
        if bound == "tensor":
            parts[n]["frac_of_sustained"] = round(achieved / peaks["bf16_tflops_sustained"], 4)
    for tag, ms, byts, hist in (
            ("b64", sum(per_kernel_ms["decode_step_b64"]), sum(dec64_b[timed]) + sum(acc64_b[timed]), n64),
            ("b1", sum(per_kernel_ms["decode_step_b1"]), sum(dec1_b[timed]) + sum(acc1_b[timed]), n1)):
        parts[f"decode_step_{tag}"] = {
            "steps_per_s": round(args.steps / (ms * 1e-3), 1),
            "GB_per_s": round(byts / (ms * 1e-3) / 1e9, 1),
            "frac_of_hbm": round(byts / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "tokens_per_step": round(float(hist[timed].sum(axis=1).mean()), 3),
        }
    for tag in ("b1", "b64"):
        parts[f"decode_step_{tag}"]["in_step"] = "one CUDA graph per step (decode attention + accept)"
    # The training shapes also as planned for them: back-to-back launches between two
    # CUDA events (inputs rotating over the same >= 2x L2 buffer sets), median of 5.
    for n, w in (("train_05b", train05), ("train_7b", train7)):
        reps = []
        for _ in range(5):
            b0 = torch.cuda.Event(enable_timing=True)
            b1 = torch.cuda.Event(enable_timing=True)
            b0.record(stream)
            for i in range(200):
                w.run(mars, i)
            b1.record(stream)
            torch.cuda.synchronize()
            reps.append(b0.elapsed_time(b1) / 200)
        us = statistics.median(reps) * 1e3
        ach = w.flops / (us * 1e-6) * 1e-12
        parts[n]["back_to_back"] = {"avg_us": round(us, 3), "launches": 200, "median_of": 5,
                                    "achieved": round(ach, 2), "frac": round(ach / peaks["bf16_tflops"], 4)}
    # The decode kernels' own device rates: a CUDA graph of back-to-back launches of
    # one kernel over the rotating buffer sets (64 at batch 64, 256 at batch 1), each
    # launch's set-up overlapping the previous one's tail as in a decode loop.
    for n, kind, work_, nl in (("decode_attn_b64", "decode", dec64, 64), ("accept_b64", "accept", dec64, 64),
                               ("decode_attn_b1", "decode", dec1, 256), ("accept_b1", "accept", dec1, 256)):
        us, byts = run_graph_kernel(mars, work_, kind, n_launches=nl)
        parts[n] = {"avg_us": round(us, 3), "timing": f"{nl} back-to-back launches in one CUDA graph",
                    "roofline": roofline("hbm", byts / (us * 1e-6) / 1e9, peaks["hbm_gbs"], "GB/s", traffic.get(n))}
    dominant = max(kernels, key=lambda n: sum(per_kernel_ms[n]))

    # headline: training-mask attention TFLOP/s on the Qwen2.5-0.5B-shaped batch
    t05_ms = max_over_ranks(dist, world, sum(per_kernel_ms["train_05b"]), device)
    value = sum_over_ranks(dist, world, train05.flops * args.steps, device) / (t05_ms * 1e-3) / 1e12

    # end to end through the public API with pinned host buffers
    e2e = run_e2e(args, mars, train05, device, stream, dist, world)
    if not args.no_graph:
        parts["decode_step_b1"].update(run_graph(mars, dec1, device, peaks["hbm_gbs"]))
        parts["decode_step_b64"].update(run_graph(mars, dec64, device, peaks["hbm_gbs"]))
        # the batch-1 workload's four thresholds, each a 256-step episode in one graph
        parts["decode_step_b1"]["tau_sweep"] = {
            str(tau): run_graph(mars, dec1, device, peaks["hbm_gbs"], tau=tau) for tau in dec1.s.taus}
    # variants of the accept row, timed on their own after the step loop: the margin
    # gate and the batch-minimum cache mode (the paper's original sampler)
    parts["accept_margin_b64"] = run_accept_variant(args, mars, dec64, device, peaks["hbm_gbs"], traffic,
                                                    "accept_margin_b64", gate="margin")
    parts["accept_batchmin_b64"] = run_accept_variant(args, mars, dec64, device, peaks["hbm_gbs"], traffic,
                                                      "accept_batchmin_b64", batch_min=True)
    # the deferred-KV sampler (decode over 2B slots with the fused commit, then the
    # acceptance that only moves the cursor), timed the same way
    parts.update(run_deferred_variant(args, mars, dec64, device, peaks["hbm_gbs"], traffic, gen))
    # the backward of the training-mask attention on both training shapes
    parts["train_bwd_05b"] = run_train_bwd(args, mars, train05, peaks["bf16_tflops"], traffic, "train_bwd_05b")
    parts["train_bwd_7b"] = run_train_bwd(args, mars, train7, peaks["bf16_tflops"], traffic, "train_bwd_7b")
    # the LM head of the proposals fused with the acceptance (Qwen2.5-7B head)
    parts.update(run_lm_head(args, mars, device, peaks, traffic, gen))

    # the clock record spans every timed phase above (step loop, back-to-back
    # training launches, e2e, graph episodes, variants, backward)
    clk = clocks.stop((win0, datetime.datetime.now()))

    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v/caches, spiked N(0,1)*2 logits; Qwen2.5-0.5B/7B shapes)",
        "config": dict(CONFIG, parallelism="replicas" if world > 1 else "single GPU", peaks=peak_src,
                       step_timing="CUDA events between the step's launches (the batch-1 decode step is one "
                                   "CUDA graph per step)"),
        "roofline": parts[dominant]["roofline"],
        "roofline_kernel": dominant,
        "parts": parts,
        "e2e": e2e,
        "clocks": clk,
        "gpu_launches": 8 * args.steps,  # 2 train, 2 decode, 2 x (accept stream + finish); decode pairs in graphs
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
        for name, cb in cpu_baselines_per_part(args.cpu_seconds).items():
            parts[name]["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_e2e(args, mars, work, device, stream, dist, world):
    """Headline metric end to end: pinned host inputs -> device -> kernel -> host.

    Every step copies its q, k, v in from pinned host memory and its o back out,
    all inside the timed region. Copies run on their own streams (one per
    direction, so the two copy engines work at once) into two device buffer
    sets, so the inputs of step i+1 and the output of step i-1 move while step
    i computes -- the way a training loop prefetches its next batch.
    """
    import torch

    s = work.s
    hq = [t.cpu().pin_memory() for t in work.sets[0][:3]]
    ho = [torch.empty(work.sets[0][3].shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    bufs = [[torch.empty_like(t) for t in work.sets[0]] for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        j = i % 2
        q, k, v, o = bufs[j]
        s_in.wait_event(ev_done[j])          # step i-2 no longer reads these inputs
        with torch.cuda.stream(s_in):
            for dst, src in zip((q, k, v), hq):
                dst.copy_(src, non_blocking=True)
        ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        stream.wait_event(ev_out[j])         # step i-2's output has left o
        mars.train_attn(q, k, v, s.L, s.B, o=o)
        ev_done[j].record(stream)
        s_out.wait_event(ev_done[j])
        with torch.cuda.stream(s_out):
            ho[j].copy_(o, non_blocking=True)
        ev_out[j].record(s_out)

    def drain():
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    for j in range(2):
        ev_done[j].record(stream)
        ev_out[j].record(stream)
    for i in range(3):
        step(i)
    drain()
    torch.cuda.synchronize()
    barrier(dist, world)
    steps = max(1, args.steps)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(steps):
        step(i)
    drain()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(dist, world, e0.elapsed_time(e1), device)
    h2d = sum(t.numel() * t.element_size() for t in hq)
    d2h = ho[0].numel() * ho[0].element_size()
    val = work.flops * steps * world / (ms * 1e-3) / 1e12
    return {"value": round(val, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "copies on their own streams, double-buffered across steps"}


def run_accept_variant(args, mars, work, device, hbm_peak, traffic, name, gate="prob", batch_min=False):
    """An accept variant on the batch-64 decode workload: min(steps, 64) calls after a
    cache reset (so the appends stay inside the cache), CUDA events on the stream."""
    import torch

    s = work.s
    n = max(1, min(args.steps, 64))
    stream = torch.cuda.current_stream()
    n_out = torch.zeros((n + args.warmup, s.batch), dtype=torch.int32, device=device)

    def call(i):
        st = work.sets[i % work.nsets]
        mars.accept(st["logits"], DECODE_TAU, work.kn, work.vn, st["kc"], st["vc"], st["lens"], workspace=st["ws"],
                    tokens=work.tokens, conf=work.conf, n_commit=n_out[i], gate=gate, batch_min=batch_min)

    work.reset()
    for i in range(args.warmup):
        call(i)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(args.warmup, args.warmup + n):
        call(i)
    ev[1].record(stream)
    torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1])
    committed = int(n_out[args.warmup:].sum().item())
    bytes_ = n * (s.batch * s.B * s.V * 2 + s.batch * s.B * 8 + s.batch * 8) + committed * s.Hkv * s.D * 2 * 2 * 2
    achieved = bytes_ / (ms * 1e-3) / 1e9
    work.reset()
    return {"avg_us": round(ms / n * 1e3, 3), "calls": n,
            "roofline": roofline("hbm", achieved, hbm_peak, "GB/s", traffic.get(name))}


def run_deferred_variant(args, mars, work, device, hbm_peak, traffic, gen):
    """The deferred-KV sampler on the batch-64 decode workload: min(steps, 64) steps
    after a cache reset, each step the deferred decode step (2B slots: the previous
    step's committed tokens, then B placeholders) and the deferred acceptance, every
    launch bracketed by CUDA events on the stream."""
    import torch

    s = work.s
    n = max(1, min(args.steps, 64))
    total = args.warmup + n
    stream = torch.cuda.current_stream()
    q2 = torch.randn((s.batch, 2 * s.B, s.Hq, s.D), generator=gen, device=device).to(torch.bfloat16)
    kn2 = torch.randn((s.batch, 2 * s.B, s.Hkv, s.D), generator=gen, device=device).to(torch.bfloat16)
    vn2 = torch.randn((s.batch, 2 * s.B, s.Hkv, s.D), generator=gen, device=device).to(torch.bfloat16)
    o2 = torch.empty_like(q2)
    pend = [torch.zeros((s.batch,), dtype=torch.int32, device=device) for _ in range(work.nsets)]
    hist_len = torch.zeros((total, s.batch), dtype=torch.int32, device=device)
    hist_p = torch.zeros((total, s.batch), dtype=torch.int32, device=device)
    hist_n = torch.zeros((total, s.batch), dtype=torch.int32, device=device)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]

    def call(i, e=None):
        st, p = work.sets[i % work.nsets], pend[i % work.nsets]
        hist_len[i].copy_(st["lens"])
        hist_p[i].copy_(p)
        if e is not None:
            e[0].record(stream)
        mars.decode_attn_deferred(q2, kn2, vn2, st["kc"], st["vc"], st["lens"], p, work.max_len, o=o2)
        if e is not None:
            e[1].record(stream)
        mars.accept_deferred(st["logits"], DECODE_TAU, st["lens"], p, s.cap, workspace=st["ws"],
                             tokens=work.tokens, conf=work.conf)
        if e is not None:
            e[2].record(stream)
        hist_n[i].copy_(p)  # this step's count (the next step's pending)

    work.reset()
    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize()
    for i in range(n):
        call(args.warmup + i, ev[i])
    torch.cuda.synchronize()
    dec_ms = sum(e[0].elapsed_time(e[1]) for e in ev)
    acc_ms = sum(e[1].elapsed_time(e[2]) for e in ev)
    lens = hist_len[args.warmup:].to(torch.int64).sum(dim=1).cpu().numpy()
    pends = hist_p[args.warmup:].to(torch.int64).sum(dim=1).cpu().numpy()
    kv_row = s.Hkv * s.D * 2 * 2  # K and V bytes of one cache row
    dec_bytes = int((lens * kv_row).sum()) + n * s.batch * 2 * s.B * (2 * s.Hkv + 2 * s.Hq) * s.D * 2 \
        + int((pends * kv_row).sum())
    acc_bytes = n * (s.batch * s.B * s.V * 2 + s.batch * s.B * 8 + s.batch * 16)
    committed = float(hist_n[args.warmup:].to(torch.float64).sum(dim=1).mean().item())
    work.reset()
    dec_gbs = dec_bytes / (dec_ms * 1e-3) / 1e9
    acc_gbs = acc_bytes / (acc_ms * 1e-3) / 1e9
    return {
        "decode_attn_deferred_b64": {"avg_us": round(dec_ms / n * 1e3, 3), "calls": n,
                                     "roofline": roofline("hbm", dec_gbs, hbm_peak, "GB/s",
                                                          traffic.get("decode_attn_deferred_b64"))},
        "accept_deferred_b64": {"avg_us": round(acc_ms / n * 1e3, 3), "calls": n,
                                "roofline": roofline("hbm", acc_gbs, hbm_peak, "GB/s",
                                                     traffic.get("accept_deferred_b64"))},
        "deferred_step_b64": {"steps_per_s": round(n / ((dec_ms + acc_ms) * 1e-3), 1),
                              "tokens_per_step": round(committed, 3)},
    }


def run_train_bwd(args, mars, work, peak, traffic, name):
    """mars_train_attn_bwd on a training shape: min(steps, 20) calls over the rotating
    input sets (their o and lse from one forward each), CUDA events on the stream.
    Useful FLOPs = 2.5 x the forward's: five products (S, dP, dV, dK, dQ) over the
    visible pairs; the kernels also recompute S and dP for dQ, which is not counted."""
    import torch

    s = work.s
    n = max(1, min(args.steps, 20))
    stream = torch.cuda.current_stream()
    prep = []
    for q, k, v, _ in work.sets:
        o_, lse = mars.train_attn(q, k, v, s.L, s.B, want_lse=True)
        do = torch.randn(q.shape, device=q.device, dtype=torch.float32).to(torch.bfloat16)
        prep.append((q, k, v, o_, do, lse, torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)))
    ws = torch.empty(mars._lib.train_attn_bwd_workspace_size(s.batch, s.L, s.Hq, s.Hkv, s.D), dtype=torch.uint8,
                     device=prep[0][0].device)

    def call(i):
        q, k, v, o_, do, lse, dq, dk, dv = prep[i % len(prep)]
        mars.train_attn_bwd(q, k, v, o_, do, lse, s.L, s.B, dq=dq, dk=dk, dv=dv, workspace=ws)

    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        call(i)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    achieved = 2.5 * work.flops / (ms * 1e-3) / 1e12
    return {"avg_us": round(ms * 1e3, 3), "calls": n, "useful_tflop_per_call": round(2.5 * work.flops / 1e12, 4),
            "roofline": roofline("tensor", achieved, peak, "TFLOP/s", traffic.get(name))}


def run_lm_head(args, mars, device, peaks, traffic, gen):
    """mars_lm_head_accept with the Qwen2.5-7B head (hidden 3584, V 152064; synthetic
    weight ~ N(0, 4 / hidden)) for the batch-64 (512 proposal rows) and batch-1 (4
    rows) decode shapes: min(steps, 20) calls after warm-up, CUDA events on the
    stream.  Batch 64 is bound by the tensor cores (2 M K V useful FLOPs per call),
    batch 1 by reading the weight from HBM (2 V K bytes per call)."""
    import torch

    from token_decoding_gb300 import synth

    K, V = 3584, synth.DECODE_7B_B64.V
    w = (torch.randn((V, K), generator=gen, device=device) * (2.0 / K ** 0.5)).to(torch.bfloat16)
    n = max(1, min(args.steps, 20))
    stream = torch.cuda.current_stream()
    out = {}
    for name, shape in (("lm_head_accept_b64", synth.DECODE_7B_B64), ("lm_head_accept_b1", synth.DECODE_7B_B1)):
        s = shape
        cap = 64 + (n + args.warmup) * s.B
        h = torch.randn((s.batch, s.B, K), generator=gen, device=device).to(torch.bfloat16)
        kn = torch.randn((s.batch, s.B, s.Hkv, s.D), generator=gen, device=device).to(torch.bfloat16)
        kc = torch.zeros((s.batch, s.Hkv, cap, s.D), dtype=torch.bfloat16, device=device)
        vc = torch.zeros_like(kc)
        lens = torch.zeros((s.batch,), dtype=torch.int32, device=device)
        ws = mars.lm_head_accept_workspace(s.batch, s.B, V, device)
        tok = torch.empty((s.batch, s.B), dtype=torch.int32, device=device)
        conf = torch.empty((s.batch, s.B), dtype=torch.float32, device=device)
        nc = torch.empty((s.batch,), dtype=torch.int32, device=device)

        def call():
            mars.lm_head_accept(h, w, DECODE_TAU, kn, kn, kc, vc, lens, workspace=ws, tokens=tok, conf=conf,
                                n_commit=nc)

        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / n
        rows = s.batch * s.B
        flops = 2 * rows * K * V
        if s.batch > 1:
            ach = flops / (us * 1e-6) / 1e12
            rl = roofline("tensor", ach, peaks["bf16_tflops"], "TFLOP/s", traffic.get(name))
        else:
            ach = 2 * V * K / (us * 1e-6) / 1e9
            rl = roofline("hbm", ach, peaks["hbm_gbs"], "GB/s", traffic.get(name))
        out[name] = {"avg_us": round(us, 3), "calls": n, "rows": rows, "hidden": K, "V": V,
                     "tflop_per_call": round(flops / 1e12, 4), "roofline": rl}
        del h, kn, kc, vc, ws
    del w
    torch.cuda.empty_cache()
    return out


def run_graph(mars, work, device, hbm_peak, tau=DECODE_TAU):
    """A whole decode episode (decode attention + accept per step: 256 steps at batch 1,
    128 at batch 64) captured as one CUDA graph; device-side steps/s, tokens per
    step and the algorithmic GB/s of the episode."""
    import torch

    n_steps = work.s.steps
    stream = torch.cuda.Stream(device=device)
    n_out = torch.zeros((n_steps, work.s.batch), dtype=torch.int32, device=device)
    with torch.cuda.stream(stream):
        work.reset()
        for i in range(2):
            work.run_decode(mars, i)
            work.run_accept(mars, i, n_out[i], tau=tau)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(n_steps):
                work.run_decode(mars, i)
                work.run_accept(mars, i, n_out[i], tau=tau)
        reps = 3
        work.reset()
        graph.replay()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        ms = 0.0
        for _ in range(reps):
            work.reset()
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            stream.synchronize()
            ms += e0.elapsed_time(e1)
    hist = n_out.cpu().numpy()
    records = [("reset", 0, None)] + [("step", i % work.nsets, hist[i]) for i in range(n_steps)]
    dec_b, acc_b = work.byte_counts(records)
    work.reset()
    gbs = reps * (sum(dec_b) + sum(acc_b)) / (ms * 1e-3) / 1e9
    return {"graph_steps_per_s": round(reps * n_steps / (ms * 1e-3), 1), "graph_GB_per_s": round(gbs, 1),
            "graph_frac_of_hbm": round(gbs / hbm_peak, 4), "graph_us_per_step": round(ms * 1e3 / (reps * n_steps), 3),
            "tokens_per_step": round(float(hist.sum(axis=1).mean()), 3)}


def run_graph_kernel(mars, work, kind, n_launches=256, reps=3):
    """n_launches of one kernel (decode attention, or accept + append) over the
    rotating buffer sets, captured in one CUDA graph; returns (device us per launch,
    algorithmic bytes per launch)."""
    import torch

    s = work.s
    stream = torch.cuda.Stream(device=work.q.device)
    n_out = torch.zeros((n_launches, s.batch), dtype=torch.int32, device=work.q.device)

    def body():
        for i in range(n_launches):
            if kind == "decode":
                work.run_decode(mars, i)
            else:
                work.run_accept(mars, i, n_out[i])

    with torch.cuda.stream(stream):
        work.reset()
        body()
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            body()
        ms = 0.0
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        for _ in range(reps + 1):
            work.reset()
            stream.synchronize()
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            stream.synchronize()
            ms_rep = e0.elapsed_time(e1)
            if _ > 0:  # the first replay warms up
                ms += ms_rep
    hist = n_out.cpu().numpy()
    work.reset()
    kv_row = s.Hkv * s.D * 2 * 2
    small = s.batch * s.B * (2 * s.Hkv + 2 * s.Hq) * s.D * 2
    if kind == "decode":
        byts = int(work.lens0_host.sum()) * kv_row + small  # decode reads the reset lengths every launch
    else:
        byts = s.batch * s.B * s.V * 2 + float(hist.sum(axis=1).mean()) * 2 * kv_row + s.batch * s.B * 8 + s.batch * 8
    return ms * 1e3 / (reps * n_launches), byts


# --------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# --------------------------------------------------------------------------

def oracle_train_sample(budget_s, shape=None):
    """Time the fp64 oracle on whole (batch, head) slices of a training batch (the
    0.5B-shaped one by default) until about budget_s seconds have passed; returns
    (useful TFLOP/s, description, seconds)."""
    import oracle
    from token_decoding_gb300 import synth

    s = synth.TRAIN_05B if shape is None else shape
    q, k, v = synth.train_inputs(s)
    per_head = 4 * s.D * s.L * (s.L + 1)
    done = 0
    el = 0.0
    heads = 0
    while True:
        b, h = divmod(heads % (s.batch * s.Hq), s.Hq)
        g = h // (s.Hq // s.Hkv)
        t0 = time.perf_counter()
        oracle.train_attn(q.f64[b:b + 1, :, h:h + 1], k.f64[b:b + 1, :, g:g + 1], v.f64[b:b + 1, :, g:g + 1],
                          s.L, s.B, s.D ** -0.5)
        el += time.perf_counter() - t0
        done += per_head
        heads += 1
        if el >= budget_s:
            break
    return done / el / 1e12, f"{heads} (batch, head) slices of {s.name}, fp64 numpy, dense 2L x 2L masked", el


def oracle_decode_sample(budget_s, shape, tau=DECODE_TAU):
    """Time the fp64 oracle's sliding-window step (decode attention, acceptance,
    KV append) on the decode workload `shape` until about budget_s seconds of
    oracle time have passed.  Sequences are independent, so the sample is whole
    steps of single sequences (in index order, up to 8 steps each from its own
    initial cache length, so the sample spreads over the batch's lengths); the
    batch's steps/s is one over (mean time per sequence-step x batch).
    Input drawing is not timed.  Returns (steps/s, description, seconds)."""
    import oracle
    from token_decoding_gb300 import synth

    s = shape
    lens0 = synth.initial_cache_lens(s)
    el = 0.0
    seq_steps = 0
    seqs = 0
    scale = s.D ** -0.5
    per_seq = s.steps if s.batch == 1 else min(s.steps, 8)  # spread the sample over the batch's lengths
    while el < budget_s and seqs < s.batch:
        b = seqs
        kc, vc = synth.seq_cache_inputs(s, b, int(lens0[b]))
        kc64, vc64, lens = kc.f64, vc.f64, np.array([lens0[b]], dtype=np.int64)
        for t in range(per_seq):
            q, kn, vn = synth.seq_step_inputs(s, t, b)
            logits = synth.seq_step_logits(s, t, b)
            t0 = time.perf_counter()
            oracle.decode_attn(q.f64, kn.f64, vn.f64, kc64, vc64, lens, scale)
            _, _, n = oracle.accept(logits.f64, tau)
            kc64, vc64, lens = oracle.append_kv(kc64, vc64, lens, kn.f64, vn.f64, n)
            el += time.perf_counter() - t0
            seq_steps += 1
            if el >= budget_s:
                break
        seqs += 1
    per_seq_step = el / seq_steps
    desc = (f"{seq_steps} sequence-steps of {s.name} over {seqs} sequence(s) (oracle decode_attn + accept + "
            f"append_kv, tau {tau}), scaled to the batch of {s.batch}")
    return 1.0 / (per_seq_step * s.batch), desc, el


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(budget_s):
    val, sample, _ = oracle_train_sample(budget_s)
    return {"value": round(val, 6), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": sample + " (numpy BLAS threads: all available cores)"}


def cpu_baselines_per_part(budget_s):
    """The oracle beside every timed configuration: the 7B-shaped training batch
    (TFLOP/s) and both decode workloads (steps/s)."""
    from token_decoding_gb300 import synth

    out = {}
    val, sample, _ = oracle_train_sample(budget_s, synth.TRAIN_7B)
    out["train_7b"] = {"value": round(val, 6), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                       "sample": sample}
    for name, shape in (("decode_step_b1", synth.DECODE_7B_B1), ("decode_step_b64", synth.DECODE_7B_B64)):
        val, sample, _ = oracle_decode_sample(budget_s, shape)
        out[name] = {"value": round(val, 4), "unit": "steps/s", "cores": cpu_cores(), "kind": "oracle",
                     "sample": sample}
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return
    budget = max(0.5, args.cpu_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_train_sample(budget)
    vals, secs = [], 0.0
    desc = ""
    for _ in range(args.steps):
        v, desc, el = oracle_train_sample(budget)
        vals.append(v)
        secs += el
    value = float(np.mean(vals)) if vals else 0.0
    line = {
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs / max(1, args.steps) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(CONFIG, parallelism="single process on the host cores"),
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_profile(args):
    """--profile PART: warm-up + steps launches of one kernel on its workload, nothing else (for ncu)."""
    import torch

    import token_decoding_gb300 as mars
    from token_decoding_gb300 import build as mars_build
    from token_decoding_gb300 import synth

    if not os.path.exists(mars._lib.LIB_PATH):
        mars_build.build()
    device = torch.device("cuda:0")
    gen = torch.Generator(device=device)
    gen.manual_seed(1234)
    part = args.profile
    if part.startswith("lm_head"):
        K, V = 3584, synth.DECODE_7B_B64.V
        shape = synth.DECODE_7B_B64 if part.endswith("b64") else synth.DECODE_7B_B1
        w = (torch.randn((V, K), generator=gen, device=device) * (2.0 / K ** 0.5)).to(torch.bfloat16)
        h = torch.randn((shape.batch, shape.B, K), generator=gen, device=device).to(torch.bfloat16)
        kn = torch.randn((shape.batch, shape.B, shape.Hkv, shape.D), generator=gen, device=device).to(torch.bfloat16)
        kc = torch.zeros((shape.batch, shape.Hkv, 64, shape.D), dtype=torch.bfloat16, device=device)
        lens = torch.zeros((shape.batch,), dtype=torch.int32, device=device)

        def run(i):
            lens.zero_()
            mars.lm_head_accept(h, w, DECODE_TAU, kn, kn, kc, kc, lens)
    elif part.startswith("train_bwd"):
        w = TrainWork(synth.TRAIN_05B if part == "train_bwd_05b" else synth.TRAIN_7B, device, gen, 0)
        s = w.s
        q, k, v, _ = w.sets[0]
        o_, lse = mars.train_attn(q, k, v, s.L, s.B, want_lse=True)
        do = torch.randn(q.shape, generator=gen, device=device).to(torch.bfloat16)
        run = lambda i: mars.train_attn_bwd(q, k, v, o_, do, lse, s.L, s.B)  # noqa: E731
    elif part.startswith("train"):
        w = TrainWork(synth.TRAIN_05B if part == "train_05b" else synth.TRAIN_7B, device, gen, 0)
        run = lambda i: w.run(mars, i)  # noqa: E731
    else:
        shape = synth.DECODE_7B_B64 if part.endswith("b64") else synth.DECODE_7B_B1
        w = DecodeWork(shape, device, gen, 0, steps_per_episode=shape.steps)
        n_out = torch.zeros((shape.batch,), dtype=torch.int32, device=device)
        s = shape
        if "deferred" in part:
            # a fixed pending count per sequence (uniform in [0, B]), restored before each call
            pend0 = torch.randint(0, s.B + 1, (s.batch,), generator=gen, device=device, dtype=torch.int32)
        if part == "decode_attn_deferred_b64":
            q2 = torch.randn((s.batch, 2 * s.B, s.Hq, s.D), generator=gen, device=device).to(torch.bfloat16)
            kn2 = torch.randn((s.batch, 2 * s.B, s.Hkv, s.D), generator=gen, device=device).to(torch.bfloat16)
            vn2 = torch.randn((s.batch, 2 * s.B, s.Hkv, s.D), generator=gen, device=device).to(torch.bfloat16)
            o2 = torch.empty_like(q2)

            def run(i):
                st = w.sets[i % w.nsets]
                mars.decode_attn_deferred(q2, kn2, vn2, st["kc"], st["vc"], st["lens"], pend0, w.max_len, o=o2)
        elif part == "accept_deferred_b64":
            def run(i):
                w.reset()
                n_out.copy_(pend0)
                st = w.sets[i % w.nsets]
                mars.accept_deferred(st["logits"], DECODE_TAU, st["lens"], n_out, s.cap, workspace=st["ws"],
                                     tokens=w.tokens, conf=w.conf)
        elif part.startswith("decode"):
            run = lambda i: w.run_decode(mars, i)  # noqa: E731
        else:
            gate = "margin" if "margin" in part else "prob"

            def run(i):
                w.reset()
                w.run_accept(mars, i, n_out, gate)
    for i in range(args.warmup + args.steps):
        run(i)
    torch.cuda.synchronize()
    print("profiled", part, args.warmup + args.steps, "launches")


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None,
                   help="timed steps (default: 1000 for the GPU arm, about half a second of GPU time; 10 for "
                        "--impl reference)")
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["mars", "reference"], default="mars")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph decode episodes (batch 1 and 64)")
    p.add_argument("--profile", choices=["train_05b", "train_7b", "decode_attn_b64", "accept_b64", "decode_attn_b1",
                                         "accept_b1", "accept_margin_b64", "decode_attn_deferred_b64",
                                         "accept_deferred_b64", "train_bwd_05b", "train_bwd_7b",
                                         "lm_head_accept_b64", "lm_head_accept_b1"],
                   help="only launch this kernel, warm-up + steps times, and print no JSON (for ncu)")
    args = p.parse_args()
    if args.steps is None:
        args.steps = 10 if args.impl == "reference" else (3 if args.profile else 1000)
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    if args.profile:
        run_profile(args)
        return
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_gpu(args, rank, world, local)


if __name__ == "__main__":
    main()
