"""Threshold re-noising and canvas initialisation (integer work).

Explainer, "2. Uniform-state diffusion": there is no [MASK] token; noise is
a random vocabulary token; a token whose probability falls below a
threshold is re-noised with a new random token, a confident one is kept.
Explainer, "The problem with autoregressive models": the canvas starts as
256 random vocabulary tokens.

Readings (the pages leave these open):
  * "the token's probability" is the maximum softmax probability conf_i;
  * a kept (confident) position takes the argmax prediction;
  * re-noise iff conf < threshold (strict: conf == threshold is kept),
    compared in float32, the precision the kernels produce conf in;
  * the random token is uniform over all V ids (see philox.py).
"""
from __future__ import annotations

import numpy as np

from .philox import uniform_token, PHILOX_DOMAIN_RENOISE, PHILOX_DOMAIN_INIT


def renoise(argmax, conf, V, threshold, seed, step, abs_pos0):
    """Returns (tokens int32 [C], renoised uint8 [C])."""
    argmax = np.asarray(argmax, dtype=np.int64)
    conf32 = np.asarray(conf, dtype=np.float32)
    C = argmax.shape[0]
    draw = uniform_token(seed, step, int(abs_pos0) + np.arange(C, dtype=np.int64), PHILOX_DOMAIN_RENOISE, V)
    low = conf32 < np.float32(threshold)
    tokens = np.where(low, draw, argmax).astype(np.int32)
    return tokens, low.astype(np.uint8)


def canvas_init(C, V, seed, abs_pos0):
    """A fresh canvas: every position a uniform vocabulary token (domain 1, step 0)."""
    pos = int(abs_pos0) + np.arange(C, dtype=np.int64)
    return uniform_token(seed, 0, pos, PHILOX_DOMAIN_INIT, V).astype(np.int32)
