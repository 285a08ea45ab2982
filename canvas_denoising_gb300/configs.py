"""Named workloads: shapes of the explainer's canvas workload (a 256-token
canvas, a large vocabulary, a long KV prefix) at five sizes.

`alpha` is the signal scale of the synthetic hidden state
H_i = alpha * E[t_i] + N(0, 1). `alpha_literal` is the value first written
for each workload; at those values no position reaches the threshold, so
`alpha` is re-calibrated (oracle/calibrate_alpha.py, bisection on the
oracle's confidences, seed 0) until about half the positions are confident.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    name: str
    C: int
    V: int
    d: int
    Hq: int
    Hkv: int
    hd: int
    prefix: int
    dtype: str            # "f32" or "bf16"
    thresholds: tuple
    steps: int
    alpha: float
    alpha_literal: float
    blocks: int = 1
    seed: int = 0
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def cap(self) -> int:
        """KV-cache capacity: the prefix plus every block this workload appends."""
        return self.prefix + self.blocks * self.C


WORKLOADS = {
    "tiny_f32": Workload(
        "tiny_f32", C=16, V=512, d=64, Hq=2, Hkv=1, hd=32, prefix=32, dtype="f32",
        thresholds=(0.5,), steps=4, alpha=0.0, alpha_literal=0.0,
        notes="H~N(0,1): every position is below the threshold and re-noised"),
    "v32k_d1024_p1k": Workload(
        "v32k_d1024_p1k", C=256, V=32768, d=1024, Hq=8, Hkv=4, hd=128, prefix=1024, dtype="bf16",
        thresholds=(0.5,), steps=8, alpha=26.0, alpha_literal=8.0),
    "v262k_d2816_p4k": Workload(
        "v262k_d2816_p4k", C=256, V=262144, d=2816, Hq=16, Hkv=8, hd=128, prefix=4096, dtype="bf16",
        thresholds=(0.3,), steps=16, alpha=11.0, alpha_literal=6.0),
    "v262k_d2816_p32k": Workload(
        "v262k_d2816_p32k", C=256, V=262144, d=2816, Hq=16, Hkv=8, hd=128, prefix=32768, dtype="bf16",
        thresholds=(0.1, 0.3, 0.5, 0.7), steps=32, alpha=11.0, alpha_literal=6.0,
        notes="long context; alpha fixed at the 4k workload's value for every threshold"),
    "multiblock_8x24": Workload(
        "multiblock_8x24", C=256, V=262144, d=2816, Hq=16, Hkv=8, hd=128, prefix=2048, dtype="bf16",
        thresholds=(0.3,), steps=24, alpha=11.0, alpha_literal=6.0, blocks=8,
        notes="8 canvases x 24 steps; each finalised canvas is appended (prefix 2048 -> 4096)"),
}

HEADLINE = "v262k_d2816_p4k"
