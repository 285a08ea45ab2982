"""Philox4x64-10 counter-based generator and the uniform vocabulary draw.

Philox is restated from its published definition (Salmon, Moraes, Dror,
Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11, section 3.2):
each of the 10 rounds multiplies counter words 0 and 2 by two fixed odd
constants, takes the 128-bit products' high and low halves, XORs the high
halves with the other two counter words and the round key, and permutes;
the key is bumped by two Weyl constants between rounds.

The explainer ("2. Uniform-state diffusion") says noise is a token drawn
at random from the vocabulary; the draw here is the Philox word mapped to
[0, V) by the multiply-shift of D. Lemire ("Fast random integer generation
in an interval", 2019) without rejection: exactly uniform when V is a power
of two, bias at most V / 2^32 otherwise.

Counter layout (a reading; the pages give no RNG):
    key     = (seed, 0)
    counter = (absolute sequence position, step, domain, 0)
    domain 0 = threshold re-noise, domain 1 = canvas initialisation.
"""
from __future__ import annotations

import numpy as np

_M0 = np.uint64(0xD2E7470EE14C6C93)
_M1 = np.uint64(0xCA5A826395121157)
_W0 = np.uint64(0x9E3779B97F4A7C15)  # golden ratio
_W1 = np.uint64(0xBB67AE8584CAA73B)  # sqrt(3) - 1
_LO32 = np.uint64(0xFFFFFFFF)
_S32 = np.uint64(32)

PHILOX_DOMAIN_RENOISE = 0
PHILOX_DOMAIN_INIT = 1


def _mulhilo(a, b):
    """128-bit product of uint64 arrays, returned as (hi, lo) uint64 halves."""
    a_lo, a_hi = a & _LO32, a >> _S32
    b_lo, b_hi = b & _LO32, b >> _S32
    ll = a_lo * b_lo
    lh = a_lo * b_hi
    hl = a_hi * b_lo
    hh = a_hi * b_hi
    mid = (ll >> _S32) + (lh & _LO32) + (hl & _LO32)
    hi = hh + (lh >> _S32) + (hl >> _S32) + (mid >> _S32)
    lo = a * b  # wraps mod 2^64
    return hi, lo


def philox4x64_10(ctr, key):
    """Philox4x64 with 10 rounds.

    ctr: uint64 array [..., 4]; key: uint64 array [..., 2] (broadcastable).
    Returns the four output words, uint64 [..., 4].
    """
    ctr = np.asarray(ctr, dtype=np.uint64)
    key = np.asarray(key, dtype=np.uint64)
    c0, c1, c2, c3 = (ctr[..., i].copy() for i in range(4))
    k0 = np.broadcast_to(key[..., 0], c0.shape).copy()
    k1 = np.broadcast_to(key[..., 1], c0.shape).copy()
    with np.errstate(over="ignore"):
        for r in range(10):
            if r:
                k0 = k0 + _W0
                k1 = k1 + _W1
            hi0, lo0 = _mulhilo(_M0, c0)
            hi1, lo1 = _mulhilo(_M1, c2)
            c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=-1)


def uniform_token(seed, step, abs_pos, domain, V):
    """Uniform vocabulary ids U(seed, step, abs_pos) in [0, V) (int64 array)."""
    abs_pos = np.asarray(abs_pos, dtype=np.int64)
    n = abs_pos.shape
    ctr = np.zeros(n + (4,), dtype=np.uint64)
    ctr[..., 0] = abs_pos.astype(np.uint64)
    ctr[..., 1] = np.uint64(step)
    ctr[..., 2] = np.uint64(domain)
    key = np.array([np.uint64(seed), np.uint64(0)], dtype=np.uint64)
    x0 = philox4x64_10(ctr, key)[..., 0]
    with np.errstate(over="ignore"):
        return (((x0 >> _S32) * np.uint64(V)) >> _S32).astype(np.int64)
