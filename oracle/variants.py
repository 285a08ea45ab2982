"""Rows next to the denoising step, written out from their definitions.

Test infrastructure only: the product path never imports this package.

Self-conditioning input (explainer, "Advanced inference frameworks" ->
"Self-conditioning"): after a step the probability matrix times the
token-embedding table is handed to the next step. The backbone layer that
receives it is not described on the pages; the stand-in here is the plainest
input that carries both the canvas and that vector:
    x_i = E[token_i] + S_i.

Probability of the current canvas token (explainer, "2. Uniform-state
diffusion", read the other way: "a token's probability" as the probability
the model gives to the token now on the canvas):
    p_i = softmax(l_i)[token_i] = exp(H_i . E[token_i] - lse_i).

Masked diffusion with lock-in (explainer, "1. Masked diffusion"): positions
start as a [MASK] id; a [MASK] is replaced by a word once the model is
confident, and a replaced token is never changed again. Reading: confident
means conf >= threshold (the complement of the re-noise rule), the word is
the argmax prediction, and non-[MASK] tokens are left as they are.

Early stop (the pages fix no stopping rule): a canvas is finished early when
a step re-noises no position.
"""
from __future__ import annotations

import numpy as np


def selfcond_input(tokens, emb, selfcond=None):
    """x [C][d] float64: the embedding row of each canvas token plus its
    self-conditioning vector (None: the embedding rows alone)."""
    tok = np.asarray(tokens, dtype=np.int64)
    x = np.asarray(emb)[tok].astype(np.float64)  # the C gathered rows, then widened
    if selfcond is not None:
        x += np.asarray(selfcond, dtype=np.float64)
    return x


def token_prob(h, emb, tokens, lse):
    """p [C] float64: the softmax probability of token_i in row i, given that
    row's log-sum-exp (natural log)."""
    H = np.asarray(h, dtype=np.float64)
    tok = np.asarray(tokens, dtype=np.int64)
    Et = np.asarray(emb)[tok].astype(np.float64)
    logit = np.einsum("ij,ij->i", H, Et)
    return np.exp(logit - np.asarray(lse, dtype=np.float64))


def unmask(tokens, argmax, conf, mask_id, threshold):
    """Masked-diffusion update. Returns (tokens int32 [C], unmasked uint8 [C]):
    a [MASK] position whose confidence (float32) is at least the threshold
    takes the argmax; every other position keeps its token."""
    tok = np.asarray(tokens, dtype=np.int64).copy()
    conf32 = np.asarray(conf, dtype=np.float32)
    take = (tok == int(mask_id)) & (conf32 >= np.float32(threshold))
    tok[take] = np.asarray(argmax, dtype=np.int64)[take]
    return tok.astype(np.int32), take.astype(np.uint8)


def canvas_fill(C, value):
    """A masked canvas: every position holds `value` (the [MASK] id)."""
    return np.full(C, int(value), dtype=np.int32)


def finished_early(renoised):
    """True when a step re-noised no position."""
    return not bool(np.asarray(renoised).any())
