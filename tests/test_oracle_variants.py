"""Pins for the oracle's next-row functions (self-conditioning input,
probability of the current token, masked-diffusion unmasking, early stop),
each against something other than its own formula."""
import numpy as np
from scipy.special import softmax

from oracle.vocab import vocab_step
from oracle.variants import canvas_fill, finished_early, selfcond_input, token_prob, unmask


def test_selfcond_input_is_a_one_hot_product_plus_s():
    rng = np.random.default_rng(0)
    V, d, C = 50, 12, 9
    E = rng.standard_normal((V, d))
    S = rng.standard_normal((C, d))
    tok = rng.integers(0, V, C)
    onehot = np.zeros((C, V))
    onehot[np.arange(C), tok] = 1.0
    np.testing.assert_allclose(selfcond_input(tok, E, S), onehot @ E + S, rtol=0, atol=1e-15)
    # no self-conditioning vector: exactly the embedding rows, row by row
    x = selfcond_input(tok, E)
    for i in range(C):
        np.testing.assert_array_equal(x[i], E[tok[i]])


def test_selfcond_input_of_the_oracles_own_s_for_a_one_hot_step():
    """A confident step's S is an embedding row (one-hot P), so the next input
    is the sum of two embedding rows."""
    rng = np.random.default_rng(1)
    V, d = 40, 16
    E = rng.standard_normal((V, d))
    t = np.array([5, 11, 39])
    r = vocab_step(1e4 * E[t], E)
    tok = np.array([0, 11, 7])
    np.testing.assert_allclose(selfcond_input(tok, E, r["selfcond"]), E[tok] + E[t], rtol=0, atol=0)


def test_token_prob_matches_scipy_softmax_and_sums_to_one():
    rng = np.random.default_rng(2)
    V, d, C = 300, 10, 4
    E = rng.standard_normal((V, d))
    H = 2.0 * rng.standard_normal((C, d))
    r = vocab_step(H, E)
    p = softmax(H @ E.T, axis=1)
    for v in (0, 7, 299):
        tok = np.full(C, v)
        np.testing.assert_allclose(token_prob(H, E, tok, r["lse"]), p[:, v], rtol=1e-12)
    # enumerating every token of row 0 gives a distribution
    tot = sum(token_prob(H[:1], E, np.array([v]), r["lse"][:1])[0] for v in range(V))
    np.testing.assert_allclose(tot, 1.0, rtol=1e-12)


def test_token_prob_of_the_argmax_is_the_confidence():
    rng = np.random.default_rng(3)
    V, d, C = 200, 8, 6
    E = rng.standard_normal((V, d))
    H = 3.0 * rng.standard_normal((C, d))
    r = vocab_step(H, E)
    np.testing.assert_allclose(token_prob(H, E, r["argmax"], r["lse"]), r["conf"], rtol=1e-12)


def test_unmask_thresholds_and_lock_in():
    C, mask = 8, 99
    tok = np.array([99, 3, 99, 99, 5, 99, 99, 0], dtype=np.int32)
    am = np.array([1, 2, 3, 4, 5, 6, 7, 8], dtype=np.int32)
    conf = np.array([0.9, 0.9, 0.1, 0.5, 0.0, 0.49999, 0.5, 1.0], dtype=np.float32)
    out, flag = unmask(tok, am, conf, mask, 0.5)
    # masked and conf >= 0.5 -> argmax; masked and below -> still masked; unmasked positions never change
    np.testing.assert_array_equal(out, [1, 3, 99, 4, 5, 99, 7, 0])
    np.testing.assert_array_equal(flag, [1, 0, 0, 1, 0, 0, 1, 0])
    # threshold 0 unmasks every masked position; above 1 unmasks none
    np.testing.assert_array_equal(unmask(tok, am, conf, mask, 0.0)[0], np.where(tok == mask, am, tok))
    np.testing.assert_array_equal(unmask(tok, am, conf, mask, 1.5)[0], tok)
    # applying the same update twice changes nothing more (unmasked tokens are locked)
    np.testing.assert_array_equal(unmask(out, am + 10, conf, mask, 0.5)[0][tok != mask], tok[tok != mask])


def test_canvas_fill_and_early_stop():
    np.testing.assert_array_equal(canvas_fill(5, 7), [7] * 5)
    assert finished_early(np.zeros(4, np.uint8))
    assert not finished_early(np.array([0, 0, 1, 0], np.uint8))
