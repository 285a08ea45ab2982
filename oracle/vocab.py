"""The vocabulary step, written out from its definition in float64.

Per canvas position i (row of H):
    l_i = H_i . E^T                 logits over the whole vocabulary
    m_i = max_v l_iv,  Z_i = sum_v exp(l_iv - m_i)
    p_i = exp(l_i - m_i) / Z_i      softmax over the vocabulary
    argmax_i = lowest v with l_iv == m_i
    conf_i = p_i[argmax_i] = 1 / Z_i     (the token's probability compared
                                          with the re-noise threshold)
    lse_i = m_i + ln Z_i
    S_i = p_i . E                   self-conditioning vector

Sources: the explainer's "Self-conditioning" section (the probability
matrix times the token-embedding table, handed to the next step) and
"2. Uniform-state diffusion" (a token's probability against a threshold).
The pages never write the LM head; logits = H . E^T with the embedding
table tied to the output is the reading taken here (no temperature, no
soft-cap, no scaling).

The logits and S are formed chunk by chunk over the vocabulary only to
bound host memory: each logit is still one independent float64 dot
product, and S is the same sum of float64 products taken chunk by chunk.
"""
from __future__ import annotations

import numpy as np


def vocab_step(h, emb, chunk=16384, want_top2=True):
    """Returns dict with argmax (int64 [C]), conf, lse, selfcond ([C][d]),
    and p2 (second-largest probability, [C]) all float64."""
    H = np.asarray(h, dtype=np.float64)
    C, d = H.shape
    V = emb.shape[0]
    logits = np.empty((C, V), dtype=np.float64)
    for v0 in range(0, V, chunk):
        v1 = min(V, v0 + chunk)
        logits[:, v0:v1] = H @ np.asarray(emb[v0:v1], dtype=np.float64).T
    m = logits.max(axis=1)
    amax = logits.argmax(axis=1)  # first index attaining the maximum
    w = np.exp(logits - m[:, None])
    Z = w.sum(axis=1)
    p = w / Z[:, None]
    del w
    S = np.zeros((C, d), dtype=np.float64)
    for v0 in range(0, V, chunk):
        v1 = min(V, v0 + chunk)
        S += p[:, v0:v1] @ np.asarray(emb[v0:v1], dtype=np.float64)
    res = {
        "argmax": amax.astype(np.int64),
        "conf": 1.0 / Z,
        "lse": m + np.log(Z),
        "selfcond": S,
        "max_logit": m,
    }
    if want_top2:
        if V >= 2:
            top2 = np.partition(p, V - 2, axis=1)[:, V - 2]
        else:
            top2 = np.zeros(C)
        res["p2"] = top2
        # second-largest logit, for the logit-gap diagnostic at re-noised rows
        res["l2"] = np.partition(logits, V - 2, axis=1)[:, V - 2] if V >= 2 else np.full(C, -np.inf)
    return res
