"""Calibrates the signal scale alpha of the synthetic hidden state so that
about half the canvas positions are confident (conf >= threshold).

H_i = alpha * E[t_i] + N(0, 1). At the scales first written for the two
bf16 workload sizes (8 and 6) the oracle finds no confident position at
all, so the workload would re-noise everything every step. This script
bisects alpha on the oracle's confidences (a row subset of seed 0, step 0)
and prints the result; the values are copied into configs.py.

Usage: python -m oracle.calibrate_alpha [workload ...]
"""
from __future__ import annotations

import sys

import numpy as np
import torch

from canvas_denoising_gb300 import synth
from canvas_denoising_gb300.configs import WORKLOADS

from .vocab import vocab_step


def confident_fraction(w, alpha, rows=64):
    emb = synth.embedding(w.V, w.d, w.seed, dtype=torch.bfloat16)
    tgt = synth.targets(w.C, w.V, w.seed)[:rows]
    h = synth.hidden(emb, tgt, alpha, w.seed)
    res = vocab_step(h.float().numpy(), emb.float().numpy(), want_top2=False)
    return float(np.mean(res["conf"] >= w.thresholds[0]))


def calibrate(name, target=0.5, lo=0.0, hi=64.0, iters=12):
    w = WORKLOADS[name]
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if confident_fraction(w, mid) < target:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


if __name__ == "__main__":
    names = sys.argv[1:] or ["v32k_d1024_p1k", "v262k_d2816_p4k"]
    for n in names:
        a = calibrate(n)
        print(f"{n}: alpha={a:.2f} confident={confident_fraction(WORKLOADS[n], round(a)):.3f} "
              f"(literal {WORKLOADS[n].alpha_literal}: {confident_fraction(WORKLOADS[n], WORKLOADS[n].alpha_literal):.3f})")
