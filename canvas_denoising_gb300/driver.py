"""Block-diffusion driver over the C ABI (explainer, "Multi-canvas sampling"):
denoise a 256-token canvas for a fixed number of steps, append the finished
canvas to the KV cache by incremental causal prefill, start the next canvas.

Each step runs, on one stream and entirely in libdgcanvas kernels:
  dg_canvas_attn         bidirectional attention of the canvas over cache + canvas
  dg_vocab_step_renoise  logits, softmax, argmax, confidence, self-conditioning,
                         and the threshold re-noise of low-confidence positions
and each canvas starts with dg_canvas_init and ends with dg_kv_append.

Variants (explainer, "1. Masked diffusion" and "Self-conditioning"):
  mask_id=...            masked diffusion: the canvas starts as [MASK]
                         (dg_canvas_fill) and each step unmasks confident
                         positions for good (dg_vocab_step + dg_unmask)
  next_input()           the next step's stand-in input E[token] + S
                         (dg_selfcond_input)
  generate(early_stop=True)  finish a canvas at the first step that re-noises
                         (or unmasks) nothing, counted on the device
                         (dg_count_flags)

The backbone that turns tokens into Q/K/V and the final hidden state is not
part of this path; `backbone(block, step, tokens, selfcond)` supplies them
(the tests and the benchmark use seeded synthetic tensors).
"""
from __future__ import annotations

import os
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

    def __init__(self, emb, k_cache, v_cache, prefix_len, C, Hq, threshold, seed, stream=None, mask_id=None):
        self.emb, self.k_cache, self.v_cache = emb, k_cache, v_cache
        self.Hkv, self.cap, self.hd = k_cache.shape
        self.V, self.d = emb.shape
        self.C, self.Hq = C, Hq
        self.len = int(prefix_len)
        self.threshold = float(threshold)
        self.seed = int(seed)
        self.stream = stream
        self.mask_id = mask_id
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
        self.count = torch.zeros(1, dtype=torch.int32, device=dev)
        self.x = torch.empty((C, self.d), dtype=dt, device=dev)
        # workspaces sized for the longest prefix this cache can hold
        wa = max(B.canvas_attn_workspace_size(C, Hq, self.Hkv, self.hd, p, code)
                 for p in (self.len, max(self.len, self.cap - C)))
        self.ws_attn = torch.empty(max(wa, 256), dtype=torch.uint8, device=dev)
        self.ws_vocab = torch.empty(max(B.vocab_step_workspace_size(C, self.V, self.d, code), 256), dtype=torch.uint8,
                                    device=dev)

    def begin_canvas(self):
        """A fresh canvas of uniform random tokens at absolute positions [len, len + C)
        (masked diffusion: every position [MASK])."""
        if self.mask_id is not None:
            B.canvas_fill(self.tokens, self.mask_id, stream=self.stream)
        else:
            B.canvas_init(self.tokens, self.V, self.seed, self.len, stream=self.stream)

    def step(self, step, q, k_canvas, v_canvas, h):
        o = self.out
        B.canvas_attn(q, self.k_cache, self.v_cache, self.len, k_canvas, v_canvas, out=o.attn_out, lse=o.attn_lse,
                      workspace=self.ws_attn, stream=self.stream)
        if self.mask_id is not None:
            B.vocab_step(h, self.emb, argmax=o.argmax, conf=o.conf, lse=o.lse, selfcond=o.selfcond,
                         workspace=self.ws_vocab, stream=self.stream)
            B.unmask(self.tokens, o.argmax, o.conf, self.mask_id, self.threshold, unmasked=o.renoised,
                     stream=self.stream)
            return o
        # vocabulary step with the threshold re-noise fused into its last kernel
        B.vocab_step_renoise(h, self.emb, self.tokens, self.threshold, self.seed, step, self.len, argmax=o.argmax,
                             conf=o.conf, lse=o.lse, selfcond=o.selfcond, renoised=o.renoised,
                             workspace=self.ws_vocab, stream=self.stream)
        return o

    def changed_positions(self) -> int:
        """Positions the last step re-noised (masked diffusion: unmasked),
        counted on the device; reading it synchronises the stream."""
        B.count_flags(self.out.renoised, count=self.count, stream=self.stream)
        return int(self.count.item())

    def next_input(self):
        """The next step's stand-in input x = E[token] + S (self-conditioning)."""
        return B.selfcond_input(self.tokens, self.emb, self.out.selfcond, x=self.x, stream=self.stream)

    def end_canvas(self, k_final, v_final, q_final=None):
        """Incremental causal prefill of the finished canvas: append its K/V."""
        n, out, lse = B.kv_append(self.k_cache, self.v_cache, self.len, k_final, v_final, q_new=q_final,
                                  workspace=self.ws_attn if q_final is not None else None, stream=self.stream)
        self.len = n
        return out, lse


def generate(denoiser: CanvasDenoiser, n_blocks: int, steps: int, backbone, on_step=None, early_stop=False):
    """Block diffusion: for each block, up to `steps` denoising steps then an
    append (early_stop: the canvas ends after the first step that changed no
    position). Returns the finished canvases' tokens (list of int32 device
    tensors); `denoiser.steps_taken` lists the steps each canvas ran."""
    finished = []
    denoiser.steps_taken = []
    for b in range(n_blocks):
        denoiser.begin_canvas()
        ran = 0
        for s in range(steps):
            q, kc, vc, h = backbone(b, s, denoiser.tokens, denoiser.out.selfcond)
            denoiser.step(s, q, kc, vc, h)
            ran = s + 1
            if on_step is not None:
                on_step(b, s, denoiser)
            if early_stop and denoiser.changed_positions() == 0:
                break
        denoiser.steps_taken.append(ran)
        finished.append(denoiser.tokens.clone())
        q, kc, vc, _ = backbone(b, steps, denoiser.tokens, denoiser.out.selfcond)
        denoiser.end_canvas(kc, vc)
    return finished


class GraphedBlockDiffusion:
    """Block diffusion with the cache length on the device: one CUDA graph per
    canvas (init, `steps` denoising steps, append), replayed for every block
    while the prefix grows (explainer, "Multi-canvas sampling (block
    diffusion)"). The backbone's per-step tensors are read from fixed buffers,
    which the caller fills before each replay (`load_block`)."""

    def __init__(self, emb, k_cache, v_cache, prefix_len, C, Hq, threshold, seed, steps, stream, events=None,
                 record=False):
        self.emb, self.k_cache, self.v_cache = emb, k_cache, v_cache
        self.Hkv, self.cap, self.hd = k_cache.shape
        self.V, self.d = emb.shape
        self.C, self.Hq, self.steps = C, Hq, steps
        self.threshold, self.seed, self.stream = float(threshold), int(seed), stream
        self.prefix_max = self.cap - C
        dev, dt = emb.device, emb.dtype
        self.len = int(prefix_len)
        self.len_dev = torch.tensor([self.len], dtype=torch.int64, device=dev)
        # zero-filled so that the warm-up canvas run by capture() reads finite values
        self.q = torch.zeros((steps, C, Hq, self.hd), dtype=dt, device=dev)
        self.kc = torch.zeros((steps + 1, self.Hkv, C, self.hd), dtype=dt, device=dev)  # [steps] = appended K
        self.vc = torch.zeros_like(self.kc)
        self.h = torch.zeros((steps, C, self.d), dtype=dt, device=dev)
        self.tokens = torch.empty(C, dtype=torch.int32, device=dev)
        self.out = StepOutputs(
            attn_out=torch.empty((C, Hq, self.hd), dtype=dt, device=dev),
            attn_lse=torch.empty((Hq, C), dtype=torch.float32, device=dev),
            argmax=torch.empty(C, dtype=torch.int32, device=dev),
            conf=torch.empty(C, dtype=torch.float32, device=dev),
            lse=torch.empty(C, dtype=torch.float32, device=dev),
            selfcond=torch.empty((C, self.d), dtype=dt, device=dev),
            renoised=torch.empty(C, dtype=torch.uint8, device=dev))
        wa = B.canvas_attn_workspace_size(C, Hq, self.Hkv, self.hd, self.prefix_max, B.DG_BF16)
        self.ws_attn = torch.empty(max(wa, 256), dtype=torch.uint8, device=dev)
        self.ws_vocab = torch.empty(max(B.vocab_step_workspace_size(C, self.V, self.d), 256), dtype=torch.uint8,
                                    device=dev)
        self.graph = None
        self.events = events  # optional per-step (attn start, attn end, vocab start, vocab end) timing events
        # kernels per canvas: init, steps x (attention 1-2 + vocab 2-3), append 2; attention with key
        # splits adds a counter reset kernel at head_dim 128 (DG_ATTN_COOP=1: a memset instead) and a
        # combine kernel at other head dims; the paired vocabulary form adds a flag reset kernel
        # (DG_VOCAB_COOP=1: a memset instead)
        split = self.ws_attn.numel() > 256
        n_attn = 2 if split and not (self.hd == 128 and os.environ.get("DG_ATTN_COOP") == "1") else 1
        pairs = B.vocab_step_plan(C, self.V, self.d)["cluster_pairs"] > 0
        n_vocab = 3 if pairs and os.environ.get("DG_VOCAB_COOP") != "1" else 2
        self.launches = 1 + (n_attn + n_vocab) * steps + 2
        # record=True: the initial canvas and every step's tokens, flags and statistics are copied
        # (device to device, inside the graph) into history buffers, so a whole canvas can be
        # inspected step by step
        self.history = None
        if record:
            self.history = {
                "init": torch.empty(C, dtype=torch.int32, device=dev),
                "tokens": torch.empty((steps, C), dtype=torch.int32, device=dev),
                "renoised": torch.empty((steps, C), dtype=torch.uint8, device=dev),
                "argmax": torch.empty((steps, C), dtype=torch.int32, device=dev),
                "conf": torch.empty((steps, C), dtype=torch.float32, device=dev),
                "lse": torch.empty((steps, C), dtype=torch.float32, device=dev),
                "attn_lse": torch.empty((steps, Hq, C), dtype=torch.float32, device=dev),
            }

    def _canvas(self):
        o, s_, ev = self.out, self.stream, self.events
        B.canvas_init_devpos(self.tokens, self.V, self.seed, self.len_dev, stream=s_)
        if self.history is not None:
            with torch.cuda.stream(s_):
                self.history["init"].copy_(self.tokens)
        for s in range(self.steps):
            if ev is not None:
                ev[s][0].record(s_)
            B.canvas_attn_devlen(self.q[s], self.k_cache, self.v_cache, self.len_dev, self.prefix_max, self.kc[s],
                                 self.vc[s], out=o.attn_out, lse=o.attn_lse, workspace=self.ws_attn, stream=s_)
            if ev is not None:
                ev[s][1].record(s_)
                ev[s][2].record(s_)
            B.vocab_step_renoise_devpos(self.h[s], self.emb, self.tokens, self.threshold, self.seed, s, self.len_dev,
                                        o.argmax, o.conf, o.lse, o.selfcond, o.renoised, self.ws_vocab, stream=s_)
            if ev is not None:
                ev[s][3].record(s_)
            if self.history is not None:
                hist = self.history
                with torch.cuda.stream(s_):
                    hist["tokens"][s].copy_(self.tokens)
                    hist["renoised"][s].copy_(o.renoised)
                    hist["argmax"][s].copy_(o.argmax)
                    hist["conf"][s].copy_(o.conf)
                    hist["lse"][s].copy_(o.lse)
                    hist["attn_lse"][s].copy_(o.attn_lse)
        B.kv_append_devlen(self.k_cache, self.v_cache, self.len_dev, self.kc[self.steps], self.vc[self.steps],
                           stream=s_)

    def capture(self):
        """Records one canvas as a CUDA graph (after one eager warm-up canvas,
        which the caller's first `run_block` replaces: the length is restored)."""
        saved = self.len_dev.clone()
        k0, v0 = self.k_cache.clone(), self.v_cache.clone()
        ev, self.events = self.events, None
        with torch.cuda.stream(self.stream):
            self._canvas()  # warm-up: kernel attributes and tensor maps set outside capture
        self.events = ev
        self.stream.synchronize()
        self.len_dev.copy_(saved)
        self.k_cache.copy_(k0)
        self.v_cache.copy_(v0)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self._canvas()
        return self.graph

    def load_block(self, q, kc, vc, h):
        """Per-step backbone tensors of the next block: q/kc/vc/h stacked over
        steps; kc/vc carry one more entry, the finished canvas's K/V."""
        with torch.cuda.stream(self.stream):
            self.q.copy_(q, non_blocking=True)
            self.kc.copy_(kc, non_blocking=True)
            self.vc.copy_(vc, non_blocking=True)
            self.h.copy_(h, non_blocking=True)

    def run_block(self):
        """One canvas: a graph replay; returns its final tokens (device)."""
        with torch.cuda.stream(self.stream):
            self.graph.replay()
        self.len += self.C
        return self.tokens
