#!/usr/bin/env python
"""Benchmark of one denoising step over a 256-position canvas on GB300.

A step is one pass of the whole hot path over one canvas:
  canvas attention (bidirectional, GQA, over prefix cache + canvas)
  -> fused vocabulary step (logits, softmax, argmax, confidence,
     self-conditioning) -> threshold re-noise,
plus, once per canvas (every `steps` of the workload), the canvas
initialisation and the incremental KV append of the finished canvas.

Prints ONE JSON line (rank 0). `value` is denoising steps/s over the whole
job (all ranks; replicas: each rank denoises its own canvas). Inputs are
seeded synthetic tensors resident in HBM; the embedding table (1.48 GB at
the headline size) is larger than L2, so no separate L2 flush is needed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on the host cores
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from canvas_denoising_gb300.configs import HEADLINE, WORKLOADS  # noqa: E402



def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch every kernel from Python instead of a CUDA graph")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def replica_seed(base_seed: int, rank: int) -> int:
    """Replicas: every rank denoises its own canvas, seeded by its rank."""
    return base_seed + rank


def max_over_ranks(value: float, device=None) -> float:
    """Slowest rank's time (the job finishes when the last replica does)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, steps: int, ms: float) -> float:
    """Whole-job steps/s: every rank ran `steps` steps; time is the slowest rank's."""
    return world * steps / (ms / 1e3)


def metric_name():
    return "denoise steps/s & canvas tok/s (256-pos, V=262144); % of bf16/HBM roofline"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.lines = []
        self.dev = device_index

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        uuid = getattr(torch.cuda.get_device_properties(self.dev), "uuid", None)
        if uuid is not None:
            s = str(uuid)
            cmd += ["-i", s if s.startswith("GPU-") else "GPU-" + s]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.th.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- workload state on the GPU
class Canvas:
    """Everything one rank needs for the denoising loop, resident in HBM."""

    N_INPUTS = 4  # distinct per-step (H, Q, K_c, V_c) sets cycled through

    def __init__(self, w, seed, device):
        from canvas_denoising_gb300 import binding as B
        from canvas_denoising_gb300 import synth
        self.B, self.w = B, w
        dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
        self.dt = dt
        self.seed = seed
        self.emb = synth.embedding(w.V, w.d, seed, dtype=dt, device=device)
        self.tgt = synth.targets(w.C, w.V, seed, device=device)
        self.P = w.prefix
        self.cap = w.prefix + w.C
        self.k, self.v = synth.kv_prefix(w.Hkv, self.cap, w.hd, w.prefix, seed, dtype=dt, device=device)
        self.inputs = []
        for s in range(self.N_INPUTS):
            h = synth.hidden(self.emb, self.tgt, w.alpha, seed, step=s, dtype=dt)
            q, kn, vn = synth.canvas_qkv(w.C, w.Hq, w.Hkv, w.hd, seed, step=s, dtype=dt, device=device)
            self.inputs.append((h, q, kn, vn))
        self.tokens = torch.empty(w.C, dtype=torch.int32, device=device)
        self.renoised = torch.empty(w.C, dtype=torch.uint8, device=device)
        self.out = torch.empty((w.C, w.Hq, w.hd), dtype=dt, device=device)
        self.lse_attn = torch.empty((w.Hq, w.C), dtype=torch.float32, device=device)
        self.argmax = torch.empty(w.C, dtype=torch.int32, device=device)
        self.conf = torch.empty(w.C, dtype=torch.float32, device=device)
        self.lse = torch.empty(w.C, dtype=torch.float32, device=device)
        self.selfcond = torch.empty((w.C, w.d), dtype=dt, device=device)
        dcode = B.DG_F32 if dt == torch.float32 else B.DG_BF16
        na = B.canvas_attn_workspace_size(w.C, w.Hq, w.Hkv, w.hd, self.P, dcode)
        nv = B.vocab_step_workspace_size(w.C, w.V, w.d, dcode)
        self.ws_attn = torch.empty(max(na, 256), dtype=torch.uint8, device=device)
        self.ws_vocab = torch.empty(max(nv, 256), dtype=torch.uint8, device=device)
        self.launches_per_step = None
        self.vocab_kernels = vocab_kernels_per_call(B, w, dt)

    def step(self, s, stream, ev=None, inputs=None):
        """One denoising iteration; per-canvas work at the canvas boundaries."""
        B, w = self.B, self.w
        h, q, kn, vn = inputs if inputs is not None else self.inputs[s % self.N_INPUTS]
        j = s % w.steps
        n = 0
        if j == 0:
            B.canvas_init(self.tokens, w.V, self.seed, self.P, stream=stream)
            n += 1
        if ev is not None and ev[2] is not None:
            ev[2].record(stream)
        B.canvas_attn(q, self.k, self.v, self.P, kn, vn, out=self.out, lse=self.lse_attn, workspace=self.ws_attn,
                      stream=stream)
        # one attention kernel, plus (with key splits) a counter reset kernel ahead of it at
        # head_dim 128 (DG_ATTN_COOP=1: a memset instead) or a combine kernel after it otherwise
        split = self.ws_attn.numel() > 256
        n += 2 if split and not (w.hd == 128 and os.environ.get("DG_ATTN_COOP") == "1") else 1
        if ev is not None and ev[3] is not None:
            ev[3].record(stream)
        if ev is not None and ev[0] is not None:
            ev[0].record(stream)
        # vocabulary step with the threshold re-noise fused into its last kernel
        B.vocab_step_renoise(h, self.emb, self.tokens, w.thresholds[0], self.seed, j, self.P, argmax=self.argmax,
                             conf=self.conf, lse=self.lse, selfcond=self.selfcond, renoised=self.renoised,
                             workspace=self.ws_vocab, stream=stream)
        if ev is not None and ev[1] is not None:
            ev[1].record(stream)
        n += self.vocab_kernels
        if j == w.steps - 1:
            # finished canvas -> cache rows [P, P+C); the next canvas restarts at the same prefix
            B.kv_append(self.k, self.v, self.P, kn, vn, stream=stream)
            n += 1
        return n


ATTN_TIMING = ("right after the timed region, host ahead, each call = counter reset + attention kernel: "
               "avg_launch_ms_l2_flushed over 20 calls each timed alone after a 256 MiB write that evicts L2, "
               "events around the call; avg_launch_ms_l2_warm over 50 calls back to back, K/V staying in L2. "
               "avg_launch_ms is the one the timed steps see: flushed where the vocabulary table is larger "
               "than L2 (the vocabulary step streams it through L2 before each attention call), warm where it "
               "fits")


def per_call_l2_flushed(stream, flush_buf, fn, n, before=None):
    """Mean device time of fn(i) over n calls, each after a write of flush_buf (larger than L2), with
    events around the call only and the host held ahead (a GPU sleep queued first)."""
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        if before is not None:
            before()
        fn(0)
        torch.cuda._sleep(20_000_000)
        for i in range(n):
            flush_buf.fill_(i & 0xFF)
            pairs[i][0].record(stream)
            fn(i)
            pairs[i][1].record(stream)
    stream.synchronize()
    return sum(a.elapsed_time(b) for a, b in pairs) / n


def vocab_kernels_per_call(B, w, dt) -> int:
    """Kernels one vocabulary step (with the fused re-noise) launches: the bf16 paired form resets
    its flags with a kernel (DG_VOCAB_COOP=1: a memset) ahead of the paired kernel and the combine;
    the single-SM form has a memset, its kernel and the combine; fp32 a kernel and the re-noise."""
    if dt == torch.float32:
        return 2
    pairs = B.vocab_step_plan(w.C, w.V, w.d)["cluster_pairs"] > 0
    return 3 if pairs and os.environ.get("DG_VOCAB_COOP") != "1" else 2


def run_graphed_blocks(args, world, rank, local, w, dev, seed):
    """Block diffusion (workloads with several canvases): one CUDA graph per
    canvas with the cache length on the device, replayed while the prefix
    grows by C per canvas; after the last block the length is reset to the
    first prefix (a torch fill of one int64) and the cycle repeats."""
    from canvas_denoising_gb300 import binding as B
    from canvas_denoising_gb300 import synth
    from canvas_denoising_gb300.driver import GraphedBlockDiffusion
    dt = torch.bfloat16
    emb = synth.embedding(w.V, w.d, seed, dtype=dt, device=dev)
    tgt = synth.targets(w.C, w.V, seed, device=dev)
    k, v = synth.kv_prefix(w.Hkv, w.cap, w.hd, w.prefix, seed, dtype=dt, device=dev)
    k[:, w.prefix:].zero_()  # rows past the prefix are read (and masked) by the device-length attention
    v[:, w.prefix:].zero_()
    stream = torch.cuda.Stream(device=dev)
    gb = GraphedBlockDiffusion(emb, k, v, w.prefix, w.C, w.Hq, w.thresholds[0], seed, w.steps, stream)
    per = []
    for s in range(w.steps + 1):
        q, kn, vn = synth.canvas_qkv(w.C, w.Hq, w.Hkv, w.hd, seed, step=s % 4, dtype=dt, device=dev)
        h = synth.hidden(emb, tgt, w.alpha, seed, step=s % 4, dtype=dt)
        per.append((q, kn, vn, h))
    gb.load_block(torch.stack([p[0] for p in per[:w.steps]]), torch.stack([p[1] for p in per]),
                  torch.stack([p[2] for p in per]), torch.stack([p[3] for p in per[:w.steps]]))
    gb.capture()
    stream.synchronize()

    def canvas(b):
        if b % w.blocks == 0:
            with torch.cuda.stream(stream):
                gb.len_dev.fill_(w.prefix)
        gb.run_block()

    n_warm = max(1, -(-args.warmup // w.steps))
    for b in range(n_warm):
        canvas(b)
    stream.synchronize()
    if B.device_status(stream) != 0:
        raise SystemExit("device status error after warm-up")
    replays = max(1, args.steps // w.steps)
    K = replays * w.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for b in range(replays):
            canvas(b)
        t1.record(stream)
    stream.synchronize()
    clk = clocks.stop()
    ms = max_over_ranks(t0.elapsed_time(t1), dev)
    status = B.device_status(stream)
    # per-call device durations right after the timed region, host ahead (a GPU sleep queued
    # first), at the prefix the last replay ended with
    P_last = w.prefix + ((replays - 1) % w.blocks) * w.C

    def per_call(fn, n):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            gb.len_dev.fill_(P_last)
            fn(0)
            torch.cuda._sleep(20_000_000)
            a0.record(stream)
            for i in range(n):
                fn(i)
            a1.record(stream)
        stream.synchronize()
        return a0.elapsed_time(a1) / n

    o = gb.out
    vocab_call = lambda i: B.vocab_step_renoise_devpos(
        gb.h[0], gb.emb, gb.tokens, gb.threshold, gb.seed, i, gb.len_dev, o.argmax, o.conf, o.lse, o.selfcond,
        o.renoised, gb.ws_vocab, stream=stream)
    attn_call = lambda i: B.canvas_attn_devlen(gb.q[0], gb.k_cache, gb.v_cache, gb.len_dev, gb.prefix_max,
                                               gb.kc[0], gb.vc[0], out=o.attn_out, lse=o.attn_lse,
                                               workspace=gb.ws_attn, stream=stream)
    vocab_ms = per_call(vocab_call, 20)
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    attn_ms_cold = per_call_l2_flushed(stream, flush_buf, attn_call, 20, before=lambda: gb.len_dev.fill_(P_last))
    del flush_buf
    attn_ms_warm = per_call(attn_call, 50)
    attn_ms = attn_ms_warm if fits_in_l2(w) else attn_ms_cold
    vocab_ms_sus = per_call(vocab_call, 600)  # sustained, as in the timed loop (last: it heats the GPU)
    pk = peaks()
    flops = 4.0 * w.C * w.V * w.d
    aflops = 4.0 * w.C * (P_last + w.C) * w.hd * w.Hq
    steps_per_s = job_rate(world, K, ms)
    return {
        "metric": metric_name(), "value": round(steps_per_s, 3), "unit": "steps/s", "n_gpus": world, "steps": K,
        "warmup": n_warm * w.steps, "ms_per_step": round(ms / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "canvas_tok_per_s": round(steps_per_s * w.C, 1),
        "config": {"workload": w.name, "canvas": w.C, "vocab": w.V, "d_model": w.d, "q_heads": w.Hq,
                   "kv_heads": w.Hkv, "head_dim": w.hd, "kv_prefix": f"{w.prefix}->{w.prefix + w.blocks * w.C}",
                   "blocks": w.blocks, "steps_per_canvas": w.steps, "threshold": w.thresholds[0], "alpha": w.alpha,
                   "parallelism": f"replicas{world}", "cuda_graph": "one per canvas, device-side cache length",
                   "l2": "inputs larger than L2 (embedding table %.2f GB), no flush" % (w.V * w.d * 2 / 1e9)},
        "roofline": {"kernel": f"dg_vocab_step_renoise_devpos ({vocab_kernel(w)} + vocab_combine)", "bound": "tensor",
                     "achieved": round(flops / (vocab_ms / 1e3) / 1e12, 1), "peak": pk["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(flops / (vocab_ms / 1e3) / 1e12 / pk["bf16_tflops"], 4),
                     # same vocabulary-step shapes as the headline workload, so its capture applies
                     "traffic": committed_traffic(vocab_kernel(w), "v262k_d2816_p4k"),
                     "peak_source": f"{pk['source']} bf16 burst",
                     "algorithmic_flops_per_launch": flops, "avg_launch_ms": round(vocab_ms, 4),
                     "avg_launch_ms_sustained": round(vocab_ms_sus, 4),
                     "frac_sustained": (round(flops / (vocab_ms_sus / 1e3) / 1e12 / pk["bf16_tflops_sustained"], 4)
                                        if pk.get("bf16_tflops_sustained") else None)},
        "roofline_attention": {"kernel": f"dg_canvas_attn_devlen (attn_fwd_tc) at prefix {P_last}", "bound": "tensor",
                               "achieved": round(aflops / (attn_ms / 1e3) / 1e12, 1), "peak": pk["bf16_tflops"],
                               "unit": "TFLOP/s",
                               "frac": round(aflops / (attn_ms / 1e3) / 1e12 / pk["bf16_tflops"], 4),
                               "traffic": None, "algorithmic_flops_per_launch": aflops,
                               "avg_launch_ms": round(attn_ms, 4), "avg_launch_ms_l2_warm": round(attn_ms_warm, 4),
                               "avg_launch_ms_l2_flushed": round(attn_ms_cold, 4),
                               "timing": ATTN_TIMING},
        # attention at the mean prefix over the canvases (prefix + b*C for canvas b)
        "roofline_step": step_roofline(flops + 4.0 * w.C * (w.prefix + (w.blocks - 1) * w.C / 2 + w.C) * w.hd * w.Hq,
                                       ms / K, pk),
        "gpu_launches": replays * gb.launches * world, "cuda_graph": True, "clocks": clk, "device_status": status,
        "e2e": None,
    }


def run_ours(args, world, rank, local):
    from canvas_denoising_gb300 import binding as B
    from canvas_denoising_gb300 import build as build_mod
    w = WORKLOADS[args.workload]
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    if not os.path.exists(build_mod.LIB):
        raise SystemExit("libdgcanvas is not built: run `python -c 'import __graft_entry__ as g; g.build()'` first")
    B.load()
    seed = replica_seed(w.seed, rank)
    if w.blocks > 1 and not args.no_graph:
        line = run_graphed_blocks(args, world, rank, local, w, dev, seed)
        if world > 1:
            torch.distributed.destroy_process_group()
        return line if rank == 0 else None
    cv = Canvas(w, seed, dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for s in range(args.warmup):
            cv.step(s, stream)
    stream.synchronize()
    if B.device_status(stream) != 0:
        raise SystemExit("device status error after warm-up")

    K = args.steps
    spc = w.steps  # one CUDA graph = one canvas: init, `spc` steps, append
    graph, g_launches = None, 0
    if not args.no_graph:
        graph, g_launches = capture_canvas_graph(cv, stream, spc)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    launches = 0
    # the timed region is graph replays (plus eager steps for a remainder); per-call durations are
    # measured right after it (below), since event nodes inside a graph misreport their interval
    # and eager steps can include host launch gaps
    replays = K // spc if graph is not None else 0
    eager = K - replays * spc
    evs = [None] * eager
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(replays):
            graph.replay()
            launches += g_launches
        for s in range(eager):
            launches += cv.step(s, stream, ev=evs[s])
        t1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    ms = t0.elapsed_time(t1)
    status = B.device_status(stream)
    ms = max_over_ranks(ms, dev)
    # Per-call device durations: back-to-back calls right after the timed region, on the same
    # stream, with the host held ahead of the GPU (a GPU sleep is queued first) so that no host
    # launch gap falls between the events: 20 vocabulary calls, 50 attention calls.
    h0, q0, kn0, vn0 = cv.inputs[0]

    def per_call(fn, n):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            fn(0)
            torch.cuda._sleep(20_000_000)
            a0.record(stream)
            for i in range(n):
                fn(i)
            a1.record(stream)
        stream.synchronize()
        return a0.elapsed_time(a1) / n

    vocab_call = lambda i: B.vocab_step_renoise(
        h0, cv.emb, cv.tokens, w.thresholds[0], cv.seed, i, cv.P, argmax=cv.argmax, conf=cv.conf, lse=cv.lse,
        selfcond=cv.selfcond, renoised=cv.renoised, workspace=cv.ws_vocab, stream=stream)
    attn_call = lambda i: B.canvas_attn(q0, cv.k, cv.v, cv.P, kn0, vn0, out=cv.out, lse=cv.lse_attn,
                                        workspace=cv.ws_attn, stream=stream)
    vocab_ms = per_call(vocab_call, 20)
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    attn_ms_cold = per_call_l2_flushed(stream, flush_buf, attn_call, 20)
    attn_ms_warm = per_call(attn_call, 50)
    attn_ms = attn_ms_warm if fits_in_l2(w) else attn_ms_cold

    # Workloads whose operands fit in L2 (the 32k-vocabulary one: E is 64 MiB) run warm above; the same
    # calls and whole steps are also timed with L2 flushed before each one (a 256 MiB write), events
    # around the call only.
    flushed = None
    if fits_in_l2(w):
        def per_call_flushed(fn, n):
            return per_call_l2_flushed(stream, flush_buf, fn, n)

        flushed = {
            "vocab_ms": per_call_flushed(lambda i: B.vocab_step_renoise(
                h0, cv.emb, cv.tokens, w.thresholds[0], cv.seed, i, cv.P, argmax=cv.argmax, conf=cv.conf,
                lse=cv.lse, selfcond=cv.selfcond, renoised=cv.renoised, workspace=cv.ws_vocab, stream=stream), 20),
            "attn_ms": per_call_flushed(lambda i: B.canvas_attn(q0, cv.k, cv.v, cv.P, kn0, vn0, out=cv.out,
                                                                lse=cv.lse_attn, workspace=cv.ws_attn,
                                                                stream=stream), 20),
            "step_ms": per_call_flushed(lambda i: cv.step(i, stream), 2 * w.steps),
        }
    del flush_buf

    # ---- end to end through the public API: per-step inputs from pinned host memory, result back.
    # As a pipelined caller would: the next step's inputs are copied on a second stream into the
    # other of two device buffers while the current step computes; each step's result (tokens,
    # self-conditioning vector) is staged on the device and read back on the copy stream.
    e2e = None
    if not args.no_e2e:
        Ke = min(K, 200)
        host_in = [tuple(x.cpu().pin_memory() for x in cv.inputs[i]) for i in range(cv.N_INPUTS)]
        dev_in = [tuple(torch.empty_like(x) for x in cv.inputs[0]) for _ in range(2)]
        stage = [(torch.empty_like(cv.tokens), torch.empty_like(cv.selfcond)) for _ in range(2)]
        host_tok = torch.empty(w.C, dtype=torch.int32).pin_memory()
        host_sc = torch.empty((w.C, w.d), dtype=cv.dt).pin_memory()
        h2d = sum(x.numel() * x.element_size() for x in host_in[0])
        d2h = host_tok.numel() * 4 + host_sc.numel() * host_sc.element_size()
        cs = torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event()
        in_ready, in_free, out_ready, out_read = ([ev(), ev()] for _ in range(4))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def load(step, b):
            for dst, src in zip(dev_in[b], host_in[step % cv.N_INPUTS]):
                dst.copy_(src, non_blocking=True)
            in_ready[b].record(cs)

        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        cs.wait_event(e0)
        with torch.cuda.stream(cs):
            load(0, 0)
        for s in range(Ke):
            b = s % 2
            if s + 1 < Ke:
                with torch.cuda.stream(cs):
                    if s >= 1:
                        cs.wait_event(in_free[1 - b])  # step s-1 is done reading that buffer
                    load(s + 1, 1 - b)
            with torch.cuda.stream(stream):
                stream.wait_event(in_ready[b])
                if s >= 2:
                    stream.wait_event(out_read[b])  # the staging buffer's previous read-back is done
                cv.step(s, stream, inputs=dev_in[b])
                in_free[b].record(stream)
                stage[b][0].copy_(cv.tokens, non_blocking=True)
                stage[b][1].copy_(cv.selfcond, non_blocking=True)
                out_ready[b].record(stream)
            with torch.cuda.stream(cs):
                cs.wait_event(out_ready[b])
                host_tok.copy_(stage[b][0], non_blocking=True)
                host_sc.copy_(stage[b][1], non_blocking=True)
                out_read[b].record(cs)
        stream.wait_stream(cs)
        e1.record(stream)
        stream.synchronize()
        ems = e0.elapsed_time(e1)
        ems = max_over_ranks(ems, dev)
        e2e = {"value": round(job_rate(world, Ke, ems), 3), "unit": "steps/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": Ke,
               "pipelining": "inputs double-buffered on a copy stream; results staged on device, read back there"}

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return None
    # the vocabulary call sustained (after every other timing, so that the heat it leaves slows none
    # of them): 600 back-to-back calls, ~0.3 s under the power cap as in the timed loop, the time
    # that the sustained peak applies to
    vocab_ms_sus = per_call(vocab_call, 600)
    pk = peaks()
    flops = 4.0 * w.C * w.V * w.d
    achieved = flops / (vocab_ms / 1e3) / 1e12
    traffic = committed_traffic(vocab_kernel(w), args.workload)
    roof = {"kernel": f"dg_vocab_step_renoise ({vocab_kernel(w)} + vocab_combine)", "bound": "tensor",
            "achieved": round(achieved, 1), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
            "frac": round(achieved / pk["bf16_tflops"], 4), "traffic": traffic,
            "peak_source": f"{pk['source']} bf16 burst", "algorithmic_flops_per_launch": flops,
            "avg_launch_ms": round(vocab_ms, 4),
            "timing": "20 back-to-back calls right after the timed region (flag reset + 2 kernels each), host ahead"}
    roof["avg_launch_ms_sustained"] = round(vocab_ms_sus, 4)
    if pk.get("bf16_tflops_sustained"):
        # 600 back-to-back calls under the power cap against the peak cuBLAS sustains in a long loop
        roof["peak_sustained"] = pk["bf16_tflops_sustained"]
        roof["frac_sustained"] = round(flops / (vocab_ms_sus / 1e3) / 1e12 / pk["bf16_tflops_sustained"], 4)
    # the step's other contraction: canvas attention (one launch per step)
    aflops = 4.0 * w.C * (w.prefix + w.C) * w.hd * w.Hq
    a_ach = aflops / (attn_ms / 1e3) / 1e12
    roof_attn = {"kernel": "dg_canvas_attn (attn_fwd_tc)", "bound": "tensor", "achieved": round(a_ach, 1),
                 "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": round(a_ach / pk["bf16_tflops"], 4),
                 "traffic": committed_traffic("attn_fwd_tc", args.workload),
                 "peak_source": f"{pk['source']} bf16 burst", "algorithmic_flops_per_launch": aflops,
                 "avg_launch_ms": round(attn_ms, 4), "avg_launch_ms_l2_warm": round(attn_ms_warm, 4),
                 "avg_launch_ms_l2_flushed": round(attn_ms_cold, 4),
                 "timing": ATTN_TIMING}
    steps_per_s = job_rate(world, K, ms)
    line = {
        "metric": metric_name(), "value": round(steps_per_s, 3), "unit": "steps/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "canvas_tok_per_s": round(steps_per_s * w.C, 1),
        "config": workload_config(w, world),
        "roofline": roof,
        "roofline_attention": roof_attn,
        "gpu_launches": launches * world,
        "cuda_graph": bool(replays), 
        "clocks": clk, "device_status": status,
    }
    if e2e is not None:
        line["e2e"] = e2e
    line["roofline_step"] = step_roofline(flops + aflops, ms / K, pk)
    if flushed is not None:
        fl_steps = job_rate(world, 1, flushed["step_ms"])
        line["l2_flushed"] = {
            "value": round(fl_steps, 3), "unit": "steps/s", "ms_per_step": round(flushed["step_ms"], 5),
            "vocab_ms": round(flushed["vocab_ms"], 4),
            "vocab_frac": round(flops / (flushed["vocab_ms"] / 1e3) / 1e12 / pk["bf16_tflops"], 4),
            "attn_ms": round(flushed["attn_ms"], 4),
            "attn_frac": round(aflops / (flushed["attn_ms"] / 1e3) / 1e12 / pk["bf16_tflops"], 4),
            "timing": "each call / eager step after a 256 MiB write that evicts L2; events around the call only"}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, cv)
    if world > 1:
        torch.distributed.destroy_process_group()
    return line


def workload_config(w, world):
    """The `config` object of the JSON line (the same for both arms)."""
    return {"workload": w.name, "canvas": w.C, "vocab": w.V, "d_model": w.d, "q_heads": w.Hq, "kv_heads": w.Hkv,
            "head_dim": w.hd, "kv_prefix": w.prefix, "threshold": w.thresholds[0], "steps_per_canvas": w.steps,
            "alpha": w.alpha, "parallelism": f"replicas{world}", "l2": l2_label(w)}


def capture_canvas_graph(cv, stream, spc):
    """Captures one canvas (init, spc denoising steps, append) as a CUDA graph
    without timing events. Returns (graph, kernel launches per replay), or
    (None, 0) if the capture fails."""
    g = torch.cuda.CUDAGraph()
    n = 0
    try:
        with torch.cuda.graph(g, stream=stream):
            for j in range(spc):
                n += cv.step(j, stream)
    except Exception as e:  # e.g. a launch kind this driver cannot capture: fall back to eager launches
        print(f"CUDA graph capture failed ({e}); timing eager launches", file=sys.stderr)
        torch.cuda.synchronize()
        return None, 0
    stream.synchronize()
    with torch.cuda.stream(stream):
        g.replay()  # one untimed replay
    stream.synchronize()
    return g, n


def step_roofline(step_flops, ms_per_step, pk):
    """The whole step against the bf16 peak: the step's algorithmic FLOPs (vocabulary step + attention)
    over the measured time per step (the timed region, graph replays)."""
    ach = step_flops / (ms_per_step / 1e3) / 1e12
    out = {"bound": "tensor", "achieved": round(ach, 1), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
           "frac": round(ach / pk["bf16_tflops"], 4), "algorithmic_flops_per_step": step_flops}
    if pk.get("bf16_tflops_sustained"):
        out["frac_sustained"] = round(ach / pk["bf16_tflops_sustained"], 4)
    return out


L2_BYTES = 126 * 2**20  # this GPU's L2 (129 MB nominal, ~126 MiB usable)


def fits_in_l2(w):
    """True if the step's large operands (E, the K/V cache) fit in L2 together."""
    el = 2 if w.dtype == "bf16" else 4
    return w.V * w.d * el + 2 * w.Hkv * w.cap * w.hd * el < L2_BYTES


def l2_label(w):
    gb = w.V * w.d * (2 if w.dtype == "bf16" else 4) / 1e9
    if fits_in_l2(w):
        return ("operands fit in L2 (embedding table %.3f GB): steps/s and roofline per-call times with L2 warm; "
                "the same after an L2 flush in l2_flushed" % gb)
    return "inputs larger than L2 (embedding table %.2f GB), no flush" % gb


def vocab_kernel(w):
    """Name of the vocabulary step's main kernel in the library's launch plan:
    vocab_pair (CTA pairs) where two-CTA clusters fit, else vocab_main."""
    from canvas_denoising_gb300 import binding as B
    return "vocab_pair" if B.vocab_step_plan(w.C, w.V, w.d)["cluster_pairs"] else "vocab_main"


def committed_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    from the current source of that kernel (else null)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        tab = json.load(f)
    ent = tab.get(kernel, {}).get(workload)
    if not ent:
        return None
    src = os.path.join(ROOT, "canvas_denoising_gb300", "csrc", ent["source"])
    with open(src, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()[:16]
    return ent["bytes_per_launch"] if digest == ent["source_sha256_16"] else None


# ---------------------------------------------------------------- CPU oracle arm
def _np_inputs(cv, i):
    return tuple(x.float().cpu().numpy() for x in cv.inputs[i])


def cpu_baseline(w, cv):
    """The oracle on whole steps of this workload (all rows, the whole
    vocabulary), the faster of two: ~5-20 s of CPU work at the headline size."""
    emb_np = cv.emb.float().cpu().numpy()
    k_np, v_np = cv.k.float().cpu().numpy(), cv.v.float().cpu().numpy()
    secs = min(oracle_step_parts(w, emb_np, k_np, v_np, _np_inputs(cv, i), w.C, w.V, cv.seed, i) for i in range(2))
    return {"value": round(1.0 / secs, 5), "unit": "steps/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": "two whole steps (attention, vocabulary step on every row, re-noise; float64 numpy), the faster"}


def oracle_step_parts(w, emb_np, k_np, v_np, inputs_np, qa, Vs, seed, step):
    """Runs the oracle on (a sample of) one step and returns its seconds:
    attention for the first `qa` canvas positions (every head), the
    vocabulary step on every canvas row over the first `Vs` vocabulary ids,
    the re-noise in full. qa = C and Vs = V is the whole step."""
    import oracle
    h, q, kn, vn = inputs_np
    t = time.perf_counter()
    oracle.canvas_attention(q[:qa], k_np, v_np, w.prefix, kn, vn)
    r = oracle.vocab_step(h, emb_np[:Vs], want_top2=False)
    oracle.renoise(r["argmax"], r["conf"].astype(np.float32), w.V, w.thresholds[0], seed, step, w.prefix)
    return time.perf_counter() - t


REF_BUDGET_S = float(os.environ.get("DG_REF_BUDGET_S", "150"))  # whole reference run, calibration included


def run_reference(args, world, rank, local):
    """The oracle timed on the host cores. Its cost is dominated by data
    movement that does not shrink in proportion to a sample (E is streamed
    and widened to float64 whatever the number of rows; K/V are gathered per
    head whatever the number of queries), so a sample is scaled by a measured
    ratio, not by its share of the work: one whole step and one sample step
    are timed first; each of the W + K steps then runs the sample, sized so
    that the run takes about REF_BUDGET_S seconds, and its time is scaled by
    that ratio. Both calibration times are the faster of two runs."""
    if rank != 0:
        return None
    w = WORKLOADS[args.workload]
    from canvas_denoising_gb300 import synth
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    emb = synth.embedding(w.V, w.d, w.seed, dtype=dt)
    tgt = synth.targets(w.C, w.V, w.seed)
    k, v = synth.kv_prefix(w.Hkv, w.prefix + w.C, w.hd, w.prefix, w.seed, dtype=dt)
    emb_np, k_np, v_np = emb.float().numpy(), k.float().numpy(), v.float().numpy()
    ins = []
    for s in range(2):
        h = synth.hidden(emb, tgt, w.alpha, w.seed, step=s, dtype=dt)
        q, kn, vn = synth.canvas_qkv(w.C, w.Hq, w.Hkv, w.hd, w.seed, step=s, dtype=dt)
        ins.append(tuple(x.float().numpy() for x in (h, q, kn, vn)))
    # the faster of two whole steps (the first call also pays for cold pages)
    t_full = min(oracle_step_parts(w, emb_np, k_np, v_np, ins[i], w.C, w.V, w.seed, i) for i in range(2))
    n = args.steps + args.warmup
    per_step = min(t_full, (REF_BUDGET_S - 2 * t_full) / max(1, n))
    if per_step >= t_full:
        qa, Vs = w.C, w.V  # the whole step fits the budget
    else:
        # the vocabulary step dominates: keep all rows, cut the vocabulary; a few attention positions
        frac = max(per_step, 1e-3) / t_full
        Vs = max(min(w.V, 256), min(w.V, int(w.V * frac) // 256 * 256))
        qa = max(1, min(w.C, int(w.C * frac)))
    t_cal = min(oracle_step_parts(w, emb_np, k_np, v_np, ins[i], qa, Vs, w.seed, i) for i in range(2))
    scale = t_full / t_cal
    for s in range(args.warmup):
        oracle_step_parts(w, emb_np, k_np, v_np, ins[s % 2], qa, Vs, w.seed, s)
    total = 0.0
    for s in range(args.steps):
        total += scale * oracle_step_parts(w, emb_np, k_np, v_np, ins[s % 2], qa, Vs, w.seed, s)
    val = args.steps / total
    sample = ("whole steps" if (qa, Vs) == (w.C, w.V) else
              f"per step: attention for {qa} of {w.C} canvas positions (every head), the vocabulary step on all "
              f"{w.C} rows over {Vs} of {w.V} ids, the re-noise in full (float64 numpy), scaled x{scale:.3g} = one "
              f"whole step ({t_full:.2f} s) / the same sample ({t_cal:.3f} s), each the faster of two, timed first")
    return {"impl": "reference", "metric": metric_name(), "value": round(val, 6), "unit": "steps/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, world),
            "cpu_baseline": {"value": round(val, 6), "unit": "steps/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(val, 6), "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    world, rank, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, world, rank, local)
    else:
        line = run_ours(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
