"""Seeded synthetic inputs for the canvas-denoising hot path.

This module only draws random tensors. It holds none of the method's
arithmetic (no attention, no softmax, no Philox re-noise), so that both
the CPU oracle and the CUDA path can consume the very same bytes without
sharing any code of the method.

Recipe (the pages give no distributions; these are the workload's):
  * embedding table E[V][d]      ~ N(0, 0.02^2), rounded to the compute dtype;
  * prefix K/V cache rows         ~ N(0, 1);
  * canvas Q, K_c, V_c            ~ N(0, 1), fresh per (block, step);
  * final hidden H[i] = alpha * E[t_i] + N(0, 1) noise, with target tokens
    t_i ~ U{0..V-1} fixed per canvas and the noise redrawn every step
    (alpha = 0 gives plain N(0, 1) hidden states).

Every draw comes from its own torch.Generator seeded by a stable hash of
(seed, purpose, block, step), so any tensor can be re-created alone.
"""
from __future__ import annotations

import hashlib

import torch

_PURPOSES = {
    "emb": 1, "k_prefix": 2, "v_prefix": 3, "q": 4, "k_canvas": 5, "v_canvas": 6,
    "h_noise": 7, "targets": 8, "tokens": 9, "misc": 10, "selfcond": 11, "h": 12,
}


def stream_seed(seed: int, purpose: str, block: int = 0, step: int = 0) -> int:
    """63-bit generator seed for one (seed, purpose, block, step) stream."""
    msg = f"{int(seed)}/{_PURPOSES[purpose]}/{int(block)}/{int(step)}".encode()
    return int.from_bytes(hashlib.blake2b(msg, digest_size=8).digest(), "little") >> 1


def _gen(seed, purpose, block, step, device):
    g = torch.Generator(device=device)
    g.manual_seed(stream_seed(seed, purpose, block, step))
    return g


def normal(shape, seed, purpose, block=0, step=0, std=1.0, dtype=torch.bfloat16, device="cpu"):
    """N(0, std^2) in fp32, rounded (round-to-nearest-even) to `dtype`."""
    g = _gen(seed, purpose, block, step, device)
    x = torch.randn(*shape, generator=g, dtype=torch.float32, device=device)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def randint(high, shape, seed, purpose, block=0, step=0, device="cpu"):
    g = _gen(seed, purpose, block, step, device)
    return torch.randint(0, high, shape, generator=g, dtype=torch.int64, device=device).to(torch.int32)


def embedding(V, d, seed, dtype=torch.bfloat16, device="cpu", std=0.02):
    """E[V][d] ~ N(0, std^2)."""
    return normal((V, d), seed, "emb", std=std, dtype=dtype, device=device)


def targets(C, V, seed, block=0, device="cpu"):
    """Target token ids t_i, fixed for one canvas."""
    return randint(V, (C,), seed, "targets", block=block, device=device)


def hidden(emb, tgt, alpha, seed, block=0, step=0, dtype=None):
    """H[i] = alpha * E[t_i] + N(0,1), built in fp32 and rounded once."""
    C = tgt.shape[0]
    d = emb.shape[1]
    dtype = dtype or emb.dtype
    noise = normal((C, d), seed, "h_noise", block, step, dtype=torch.float32, device=emb.device)
    if alpha != 0.0:
        noise.add_(emb.index_select(0, tgt.to(torch.int64)).to(torch.float32), alpha=float(alpha))
    return noise.to(dtype)


def kv_prefix(Hkv, cap, hd, prefix_len, seed, dtype=torch.bfloat16, device="cpu"):
    """K/V caches [Hkv][cap][hd]; rows [0, prefix_len) ~ N(0,1), the rest zero."""
    k = torch.zeros((Hkv, cap, hd), dtype=dtype, device=device)
    v = torch.zeros((Hkv, cap, hd), dtype=dtype, device=device)
    if prefix_len:
        k[:, :prefix_len] = normal((Hkv, prefix_len, hd), seed, "k_prefix", dtype=dtype, device=device)
        v[:, :prefix_len] = normal((Hkv, prefix_len, hd), seed, "v_prefix", dtype=dtype, device=device)
    return k, v


def canvas_qkv(C, Hq, Hkv, hd, seed, block=0, step=0, dtype=torch.bfloat16, device="cpu"):
    """Canvas Q [C][Hq][hd] and canvas K/V [Hkv][C][hd] for one (block, step)."""
    q = normal((C, Hq, hd), seed, "q", block, step, dtype=dtype, device=device)
    kc = normal((Hkv, C, hd), seed, "k_canvas", block, step, dtype=dtype, device=device)
    vc = normal((Hkv, C, hd), seed, "v_canvas", block, step, dtype=dtype, device=device)
    return q, kc, vc
