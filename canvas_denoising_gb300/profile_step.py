"""Runs one C-ABI call repeatedly at a chosen size and prints its CUDA-event
time: a small, self-contained driver for timing or profiling one kernel.

  python -m canvas_denoising_gb300.profile_step --op vocab --C 256 --V 65536 --d 2816
  python -m canvas_denoising_gb300.profile_step --op attn --C 256 --Hq 16 --Hkv 8 --hd 128 --P 4096
  python -m canvas_denoising_gb300.profile_step --op prefill --C 2048 --P 0      # causal append of a prompt chunk
  python -m canvas_denoising_gb300.profile_step --op selfcond --V 262144 --d 2816
"""
from __future__ import annotations

import argparse
import json

import torch

from . import binding as B
from . import synth


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", choices=["vocab", "attn", "append", "prefill", "renoise", "selfcond", "tokprob", "unmask"],
                    default="vocab")
    ap.add_argument("--C", type=int, default=256)
    ap.add_argument("--V", type=int, default=65536)
    ap.add_argument("--d", type=int, default=2816)
    ap.add_argument("--Hq", type=int, default=16)
    ap.add_argument("--Hkv", type=int, default=8)
    ap.add_argument("--hd", type=int, default=128)
    ap.add_argument("--P", type=int, default=4096)
    ap.add_argument("--alpha", type=float, default=11.0)
    ap.add_argument("--iters", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=1)
    a = ap.parse_args()
    B.load()
    dev = torch.device("cuda", 0)
    s = torch.cuda.Stream()
    if a.op == "vocab":
        emb = synth.embedding(a.V, a.d, 0, device=dev)
        h = synth.hidden(emb, synth.targets(a.C, a.V, 0, device=dev), a.alpha, 0)
        ws = torch.empty(max(256, B.vocab_step_workspace_size(a.C, a.V, a.d)), dtype=torch.uint8, device=dev)
        outs = [torch.empty(a.C, dtype=torch.int32, device=dev), torch.empty(a.C, device=dev),
                torch.empty(a.C, device=dev), torch.empty((a.C, a.d), dtype=torch.bfloat16, device=dev)]
        run = lambda: B.vocab_step(h, emb, *outs, workspace=ws, stream=s)
        flops = 4.0 * a.C * a.V * a.d
        print(json.dumps({"vocab_plan": B.vocab_step_plan(a.C, a.V, a.d)}))
    elif a.op == "prefill":
        # causal block attention of a C-row chunk appended at P (the cache is rewritten each call)
        k, v = synth.kv_prefix(a.Hkv, a.P + a.C, a.hd, a.P, 0, device=dev)
        q, kn, vn = synth.canvas_qkv(a.C, a.Hq, a.Hkv, a.hd, 0, device=dev)
        ws = torch.empty(max(256, B.canvas_attn_workspace_size(a.C, a.Hq, a.Hkv, a.hd, a.P)), dtype=torch.uint8,
                         device=dev)
        out = torch.empty_like(q)
        lse = torch.empty((a.Hq, a.C), device=dev)
        run = lambda: B.kv_append(k, v, a.P, kn, vn, q_new=q, out=out, lse=lse, workspace=ws, stream=s)
        flops = 4.0 * a.hd * a.Hq * (a.C * a.P + a.C * (a.C + 1) / 2)  # visible (query, key) pairs
    elif a.op in ("selfcond", "tokprob"):
        emb = synth.embedding(a.V, a.d, 0, device=dev)
        tok = synth.randint(a.V, (a.C,), 0, "tokens", device=dev).to(torch.int32)
        sc = synth.normal((a.C, a.d), 0, "selfcond", std=0.02, device=dev)
        h = synth.normal((a.C, a.d), 0, "h", device=dev)
        lse = torch.full((a.C,), 10.0, device=dev)
        x = torch.empty((a.C, a.d), dtype=torch.bfloat16, device=dev)
        prob = torch.empty(a.C, device=dev)
        if a.op == "selfcond":
            run = lambda: B.selfcond_input(tok, emb, sc, x=x, stream=s)
        else:
            run = lambda: B.token_prob(h, emb, tok, lse, prob=prob, stream=s)
        flops = 0.0
    elif a.op == "unmask":
        tok = torch.full((a.C,), 7, dtype=torch.int32, device=dev)
        am = torch.zeros(a.C, dtype=torch.int32, device=dev)
        conf = torch.rand(a.C, device=dev)
        run = lambda: B.unmask(tok, am, conf, 7, 0.5, stream=s)
        flops = 0.0
    elif a.op in ("attn", "append"):
        k, v = synth.kv_prefix(a.Hkv, a.P + a.C, a.hd, a.P, 0, device=dev)
        q, kn, vn = synth.canvas_qkv(a.C, a.Hq, a.Hkv, a.hd, 0, device=dev)
        ws = torch.empty(max(256, B.canvas_attn_workspace_size(a.C, a.Hq, a.Hkv, a.hd, a.P)), dtype=torch.uint8,
                         device=dev)
        out = torch.empty_like(q)
        lse = torch.empty((a.Hq, a.C), device=dev)
        if a.op == "attn":
            run = lambda: B.canvas_attn(q, k, v, a.P, kn, vn, out=out, lse=lse, workspace=ws, stream=s)
            flops = 4.0 * a.C * (a.P + a.C) * a.hd * a.Hq
        else:
            run = lambda: B.kv_append(k, v, a.P, kn, vn, stream=s)
            flops = 0.0
    else:
        tok = torch.zeros(a.C, dtype=torch.int32, device=dev)
        am = torch.zeros(a.C, dtype=torch.int32, device=dev)
        conf = torch.rand(a.C, device=dev)
        run = lambda: B.renoise(tok, am, conf, a.V, 0.3, 0, 1, a.P, stream=s)
        flops = 0.0
    with torch.cuda.stream(s):
        for _ in range(a.warmup):
            run()
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(a.iters):
            run()
        e1.record(s)
    s.synchronize()
    ms = e0.elapsed_time(e1) / a.iters
    st = B.device_status(s)
    print(json.dumps({"op": a.op, "ms": round(ms, 4), "tflops": round(flops / ms / 1e9, 1) if flops else None,
                      "status": st, "shape": vars(a)}))
    if st != 0:
        raise SystemExit(f"device status {st}")


if __name__ == "__main__":
    main()
