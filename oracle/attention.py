"""Canvas attention, written out from its definition in float64.

Follows the explainer's "Architecture: incremental prefill and denoising"
section: in denoising mode every canvas query sees every canvas token and
the whole KV cache (bidirectional); in (incremental) prefill mode attention
is causal. Readings where the pages are silent: scale 1/sqrt(hd); Q and K
already carry any positional encoding; no soft-cap, no window; query head h
reads KV head floor(h / (Hq / Hkv)) (grouped-query attention).

Slow on purpose: one dense score matrix per head, no tiling, no online
softmax.
"""
from __future__ import annotations

import math

import numpy as np


def canvas_attention(q, k_cache, v_cache, prefix_len, k_canvas, v_canvas, scale=None, causal=False):
    """Attention of the C canvas queries over keys [cache rows 0..P-1 ; canvas rows 0..C-1].

    q:        [C][Hq][hd]
    k_cache:  [Hkv][cap][hd]   (rows [0, prefix_len) are used)
    v_cache:  [Hkv][cap][hd]
    k_canvas: [Hkv][C][hd]
    v_canvas: [Hkv][C][hd]
    causal:   False -> bidirectional (denoising); True -> query i (absolute
              position P+i) sees keys 0..P+i only (incremental causal prefill).
    Returns (out [C][Hq][hd] float64, lse [Hq][C] float64), lse = natural-log
    log-sum-exp of the scaled scores.
    """
    q = np.asarray(q, dtype=np.float64)
    C, Hq, hd = q.shape
    Hkv = k_canvas.shape[0]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    group = Hq // Hkv
    P = int(prefix_len)
    if scale is None or scale <= 0:
        scale = 1.0 / math.sqrt(hd)
    L = P + C
    out = np.empty((C, Hq, hd), dtype=np.float64)
    lse = np.empty((Hq, C), dtype=np.float64)
    if causal:
        key_pos = np.arange(L)[None, :]
        query_pos = (P + np.arange(C))[:, None]
        visible = key_pos <= query_pos
    for h in range(Hq):
        g = h // group
        keys = np.concatenate([np.asarray(k_cache[g, :P], np.float64), np.asarray(k_canvas[g], np.float64)], 0)
        vals = np.concatenate([np.asarray(v_cache[g, :P], np.float64), np.asarray(v_canvas[g], np.float64)], 0)
        s = (q[:, h, :] @ keys.T) * scale  # [C][L]
        if causal:
            s = np.where(visible, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        w = np.exp(s - m)
        z = w.sum(axis=1, keepdims=True)
        out[:, h, :] = (w @ vals) / z
        lse[h] = (m + np.log(z))[:, 0]
    return out, lse
