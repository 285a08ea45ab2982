"""Incremental prefill's cache write (explainer, "Architecture: incremental
prefill and denoising" and "Multi-canvas sampling"): a finalised canvas's
keys and values are appended to the KV cache after the current prefix.
"""
from __future__ import annotations

import numpy as np


def kv_append(k_cache, v_cache, prefix_len, k_new, v_new):
    """Returns (k_cache', v_cache', prefix_len + C); rows [P, P+C) replaced by
    the new block, every other row unchanged. Arrays are [Hkv][cap][hd] and
    [Hkv][C][hd]; copies are made, inputs are not modified."""
    P = int(prefix_len)
    C = k_new.shape[1]
    cap = k_cache.shape[1]
    if P + C > cap:
        raise ValueError("append would overflow the cache capacity")
    k = np.array(k_cache, copy=True)
    v = np.array(v_cache, copy=True)
    k[:, P:P + C] = k_new
    v[:, P:P + C] = v_new
    return k, v, P + C
