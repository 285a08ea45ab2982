"""Pins for the oracle's Philox4x64-10 and uniform vocabulary draw.

External pin: numpy.random.Philox is an independent implementation of the
same generator (4 words x 64 bits, 10 rounds). numpy advances its counter
by one before producing the first block, so the block for counter c is the
first four raw words of a numpy Philox started at c - 1.
"""
import numpy as np
import pytest
from scipy import stats

from oracle.philox import philox4x64_10, uniform_token, PHILOX_DOMAIN_INIT, PHILOX_DOMAIN_RENOISE

U64 = 2 ** 64


def _numpy_block(ctr, key):
    c = [int(x) for x in ctr]
    # subtract one with borrow across the four words
    for i in range(4):  # all-zero wraps to all-ones, as a 256-bit counter does
        if c[i] > 0:
            c[i] -= 1
            break
        c[i] = U64 - 1
    bg = np.random.Philox(counter=np.array(c, dtype=np.uint64), key=np.array(key, dtype=np.uint64))
    return [int(x) for x in bg.random_raw(4)]


@pytest.mark.parametrize("trial", range(40))
def test_philox_matches_numpy(trial):
    rng = np.random.default_rng(1000 + trial)
    ctr = rng.integers(0, U64, size=4, dtype=np.uint64, endpoint=False)
    if trial % 4 == 0:
        ctr[1:] = 0  # the layout the path uses: small words
        ctr[0] = trial
    key = rng.integers(0, U64, size=2, dtype=np.uint64, endpoint=False)
    mine = [int(x) for x in philox4x64_10(ctr, key)]
    assert mine == _numpy_block(ctr, key)


def test_philox_vectorised_equals_scalar():
    rng = np.random.default_rng(7)
    ctr = rng.integers(0, U64, size=(17, 4), dtype=np.uint64)
    key = np.array([12345, 678], dtype=np.uint64)
    batch = philox4x64_10(ctr, key)
    for i in range(17):
        assert [int(x) for x in batch[i]] == [int(x) for x in philox4x64_10(ctr[i], key)]


def test_lemire_map_closed_form():
    """token = floor(hi32(x0) * V / 2^32), checked with Python integers."""
    seed, step, V = 99, 3, 262144 + 7  # a non-power-of-two V too
    pos = np.arange(0, 64, dtype=np.int64) * 1013
    toks = uniform_token(seed, step, pos, PHILOX_DOMAIN_RENOISE, V)
    for p, t in zip(pos, toks):
        x0 = _numpy_block([int(p), step, PHILOX_DOMAIN_RENOISE, 0], [seed, 0])[0]
        assert int(t) == ((x0 >> 32) * V) >> 32
        assert 0 <= int(t) < V


@pytest.mark.parametrize("V", [1024, 1000])
def test_uniform_token_chi_square(V):
    n = 1 << 20
    toks = uniform_token(5, 2, np.arange(n, dtype=np.int64), PHILOX_DOMAIN_RENOISE, V)
    counts = np.bincount(toks, minlength=V)
    assert counts.shape[0] == V
    p = stats.chisquare(counts).pvalue
    assert 0.001 < p < 0.999, p


def test_streams_differ_by_step_domain_seed():
    pos = np.arange(4096, dtype=np.int64)
    a = uniform_token(1, 0, pos, PHILOX_DOMAIN_RENOISE, 1 << 18)
    b = uniform_token(1, 1, pos, PHILOX_DOMAIN_RENOISE, 1 << 18)
    c = uniform_token(1, 0, pos, PHILOX_DOMAIN_INIT, 1 << 18)
    d = uniform_token(2, 0, pos, PHILOX_DOMAIN_RENOISE, 1 << 18)
    for x in (b, c, d):
        assert np.mean(a == x) < 0.01
