"""Pins for the oracle's vocabulary step (logits, softmax, argmax,
confidence, log-sum-exp, self-conditioning)."""
import math

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle.vocab import vocab_step


def test_one_hot_probability_reproduces_an_embedding_row():
    rng = np.random.default_rng(0)
    V, d = 40, 16
    E = rng.standard_normal((V, d))
    t = np.array([3, 17, 39])
    H = 1e4 * E[t]  # the target logit wins by ~1e4 * d: every other p underflows to 0
    r = vocab_step(H, E)
    np.testing.assert_array_equal(r["argmax"], t)
    np.testing.assert_array_equal(r["conf"], 1.0)
    np.testing.assert_allclose(r["selfcond"], E[t], rtol=0, atol=0)
    np.testing.assert_allclose(r["lse"], (H * E[t]).sum(1), rtol=1e-15)


def test_uniform_probability_gives_column_mean():
    rng = np.random.default_rng(1)
    V, d = 33, 8
    E = rng.standard_normal((V, d))
    H = np.zeros((4, d))
    r = vocab_step(H, E)
    np.testing.assert_allclose(r["selfcond"], np.broadcast_to(E.mean(0), (4, d)), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(r["conf"], 1.0 / V, rtol=1e-14)
    np.testing.assert_allclose(r["lse"], math.log(V), rtol=1e-14)
    np.testing.assert_array_equal(r["argmax"], 0)  # all tied: the lowest index


def test_probability_rows_sum_to_one():
    """A column of ones in E makes that column of S equal to sum_v p_v."""
    rng = np.random.default_rng(2)
    V, d = 500, 12
    E = 0.3 * rng.standard_normal((V, d))
    E[:, 5] = 1.0
    H = 3.0 * rng.standard_normal((7, d))
    r = vocab_step(H, E, chunk=64)
    np.testing.assert_allclose(r["selfcond"][:, 5], 1.0, rtol=0, atol=1e-12)


def test_matches_scipy_softmax_and_logsumexp():
    rng = np.random.default_rng(3)
    V, d, C = 257, 24, 6
    E = rng.standard_normal((V, d)) * 0.5
    H = rng.standard_normal((C, d))
    r = vocab_step(H, E, chunk=50)
    L = H @ E.T
    p = softmax(L, axis=1)
    np.testing.assert_allclose(r["lse"], logsumexp(L, axis=1), rtol=1e-13)
    np.testing.assert_allclose(r["conf"], p.max(1), rtol=1e-12)
    np.testing.assert_allclose(r["selfcond"], p @ E, rtol=1e-11, atol=1e-14)
    np.testing.assert_array_equal(r["argmax"], L.argmax(1))
    np.testing.assert_allclose(r["p2"], np.sort(p, 1)[:, -2], rtol=1e-12)


def test_brute_force_loops_tiny():
    rng = np.random.default_rng(4)
    V, d, C = 9, 3, 2
    E = rng.standard_normal((V, d))
    H = rng.standard_normal((C, d))
    r = vocab_step(H, E, chunk=4)
    for i in range(C):
        l = [sum(H[i, k] * E[v, k] for k in range(d)) for v in range(V)]
        m = max(l)
        w = [math.exp(x - m) for x in l]
        Z = sum(w)
        s = [sum(w[v] / Z * E[v, k] for v in range(V)) for k in range(d)]
        assert r["argmax"][i] == l.index(m)
        assert abs(r["conf"][i] - max(w) / Z) < 1e-14
        assert abs(r["lse"][i] - (m + math.log(Z))) < 1e-13
        np.testing.assert_allclose(r["selfcond"][i], s, rtol=1e-12, atol=1e-14)


def test_argmax_ties_take_lowest_index():
    E = np.zeros((10, 2))
    E[4] = [1.0, 0.0]
    E[7] = [1.0, 0.0]
    E[9] = [1.0, 0.0]
    r = vocab_step(np.array([[5.0, 1.0]]), E, chunk=3)
    assert r["argmax"][0] == 4


@pytest.mark.parametrize("chunk", [1, 7, 64, 1 << 20])
def test_chunking_does_not_change_results(chunk):
    rng = np.random.default_rng(5)
    E = rng.standard_normal((130, 10))
    H = rng.standard_normal((3, 10))
    a = vocab_step(H, E, chunk=chunk)
    b = vocab_step(H, E, chunk=130)
    for k in ("conf", "lse", "selfcond"):
        np.testing.assert_allclose(a[k], b[k], rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(a["argmax"], b["argmax"])
