"""Block-diffusion driver over the C ABI (explainer, "Multi-canvas sampling"):
denoise a 256-token canvas for a fixed number of steps, append the finished
canvas to the KV cache by incremental causal prefill, start the next canvas.

Each step runs, on one stream and entirely in libdgcanvas kernels:
  dg_canvas_attn         bidirectional attention of the canvas over cache + canvas
  dg_vocab_step_renoise  logits, softmax, argmax, confidence, self-conditioning,
                         and the threshold re-noise of low-confidence positions
and each canvas starts with dg_canvas_init and ends with dg_kv_append.

The backbone that turns tokens into Q/K/V and the final hidden state is not
part of this path; `backbone(block, step, tokens, selfcond)` supplies them
(the tests and the benchmark use seeded synthetic tensors).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import binding as B


@dataclass
class StepOutputs:
    attn_out: torch.Tensor
    attn_lse: torch.Tensor
    argmax: torch.Tensor
    conf: torch.Tensor
    lse: torch.Tensor
    selfcond: torch.Tensor
    renoised: torch.Tensor


class CanvasDenoiser:
    """Owns the device buffers of one canvas stream (cache, canvas, outputs,
    workspaces) and issues the C-ABI calls of each step."""

    def __init__(self, emb, k_cache, v_cache, prefix_len, C, Hq, threshold, seed, stream=None):
        self.emb, self.k_cache, self.v_cache = emb, k_cache, v_cache
        self.Hkv, self.cap, self.hd = k_cache.shape
        self.V, self.d = emb.shape
        self.C, self.Hq = C, Hq
        self.len = int(prefix_len)
        self.threshold = float(threshold)
        self.seed = int(seed)
        self.stream = stream
        dev, dt = emb.device, emb.dtype
        code = B.DG_BF16 if dt == torch.bfloat16 else B.DG_F32
        self.tokens = torch.empty(C, dtype=torch.int32, device=dev)
        self.out = StepOutputs(
            attn_out=torch.empty((C, Hq, self.hd), dtype=dt, device=dev),
            attn_lse=torch.empty((Hq, C), dtype=torch.float32, device=dev),
            argmax=torch.empty(C, dtype=torch.int32, device=dev),
            conf=torch.empty(C, dtype=torch.float32, device=dev),
            lse=torch.empty(C, dtype=torch.float32, device=dev),
            selfcond=torch.empty((C, self.d), dtype=dt, device=dev),
            renoised=torch.empty(C, dtype=torch.uint8, device=dev))
        # workspaces sized for the longest prefix this cache can hold
        wa = max(B.canvas_attn_workspace_size(C, Hq, self.Hkv, self.hd, p, code)
                 for p in (self.len, max(self.len, self.cap - C)))
        self.ws_attn = torch.empty(max(wa, 256), dtype=torch.uint8, device=dev)
        self.ws_vocab = torch.empty(max(B.vocab_step_workspace_size(C, self.V, self.d, code), 256), dtype=torch.uint8,
                                    device=dev)

    def begin_canvas(self):
        """A fresh canvas of uniform random tokens at absolute positions [len, len + C)."""
        B.canvas_init(self.tokens, self.V, self.seed, self.len, stream=self.stream)

    def step(self, step, q, k_canvas, v_canvas, h):
        o = self.out
        B.canvas_attn(q, self.k_cache, self.v_cache, self.len, k_canvas, v_canvas, out=o.attn_out, lse=o.attn_lse,
                      workspace=self.ws_attn, stream=self.stream)
        # vocabulary step with the threshold re-noise fused into its last kernel
        B.vocab_step_renoise(h, self.emb, self.tokens, self.threshold, self.seed, step, self.len, argmax=o.argmax,
                             conf=o.conf, lse=o.lse, selfcond=o.selfcond, renoised=o.renoised,
                             workspace=self.ws_vocab, stream=self.stream)
        return o

    def end_canvas(self, k_final, v_final, q_final=None):
        """Incremental causal prefill of the finished canvas: append its K/V."""
        n, out, lse = B.kv_append(self.k_cache, self.v_cache, self.len, k_final, v_final, q_new=q_final,
                                  workspace=self.ws_attn if q_final is not None else None, stream=self.stream)
        self.len = n
        return out, lse


def generate(denoiser: CanvasDenoiser, n_blocks: int, steps: int, backbone, on_step=None):
    """Block diffusion: for each block, `steps` denoising steps then an append.
    Returns the finished canvases' tokens (list of int32 device tensors)."""
    finished = []
    for b in range(n_blocks):
        denoiser.begin_canvas()
        for s in range(steps):
            q, kc, vc, h = backbone(b, s, denoiser.tokens, denoiser.out.selfcond)
            denoiser.step(s, q, kc, vc, h)
            if on_step is not None:
                on_step(b, s, denoiser)
        finished.append(denoiser.tokens.clone())
        q, kc, vc, _ = backbone(b, steps, denoiser.tokens, denoiser.out.selfcond)
        denoiser.end_canvas(kc, vc)
    return finished
