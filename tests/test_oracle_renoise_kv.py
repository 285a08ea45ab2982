"""Pins for threshold re-noising, canvas initialisation and the KV append."""
import numpy as np
import pytest
from scipy import stats

from oracle.kv import kv_append
from oracle.philox import uniform_token, PHILOX_DOMAIN_INIT, PHILOX_DOMAIN_RENOISE
from oracle.renoise import canvas_init, renoise


def _inputs(C=256, V=262144, seed=0):
    rng = np.random.default_rng(seed)
    return rng.integers(0, V, C), rng.random(C).astype(np.float32)


def test_threshold_zero_renoises_nothing():
    am, conf = _inputs()
    tok, rn = renoise(am, conf, 262144, 0.0, 1, 3, 4096)
    np.testing.assert_array_equal(tok, am)
    assert rn.sum() == 0


def test_threshold_one_renoises_everything_uniformly():
    C, V = 1 << 16, 1024
    am, conf = _inputs(C, V)
    conf = np.minimum(conf, np.float32(0.999))
    tok, rn = renoise(am, conf, V, 1.0, 11, 2, 0)
    assert rn.all()
    np.testing.assert_array_equal(tok, uniform_token(11, 2, np.arange(C), PHILOX_DOMAIN_RENOISE, V))
    p = stats.chisquare(np.bincount(tok, minlength=V)).pvalue
    assert 0.001 < p < 0.999


def test_renoised_set_is_exactly_below_threshold():
    am, conf = _inputs(4096, 32768, 3)
    conf[:10] = np.float32(0.3)  # equality is kept (strict comparison)
    tok, rn = renoise(am, conf, 32768, 0.3, 1, 0, 100)
    np.testing.assert_array_equal(rn.astype(bool), conf < np.float32(0.3))
    np.testing.assert_array_equal(tok[~rn.astype(bool)], am[~rn.astype(bool)])
    assert not rn[:10].any()


def test_absolute_position_keys_the_draw():
    """Two canvases at different prefix offsets never reuse draws; the same
    absolute position and step give the same draw."""
    am, conf = _inputs(256, 1 << 18)
    a, _ = renoise(am, np.zeros(256, np.float32), 1 << 18, 0.5, 9, 4, 2048)
    b, _ = renoise(am, np.zeros(256, np.float32), 1 << 18, 0.5, 9, 4, 2048 + 256)
    c, _ = renoise(am[128:], np.zeros(128, np.float32), 1 << 18, 0.5, 9, 4, 2048 + 128)
    assert np.mean(a == b) < 0.01
    np.testing.assert_array_equal(a[128:], c)


def test_canvas_init_uses_its_own_domain():
    t = canvas_init(256, 262144, 0, 0)
    assert t.dtype == np.int32 and t.min() >= 0 and t.max() < 262144
    np.testing.assert_array_equal(t, uniform_token(0, 0, np.arange(256), PHILOX_DOMAIN_INIT, 262144))
    r, _ = renoise(np.zeros(256), np.zeros(256, np.float32), 262144, 1.0, 0, 0, 0)
    assert np.mean(t == r) < 0.01


def test_kv_append_writes_rows_and_keeps_the_rest():
    rng = np.random.default_rng(0)
    Hkv, cap, hd, P, C = 2, 20, 4, 7, 5
    k = rng.standard_normal((Hkv, cap, hd)).astype(np.float32)
    v = rng.standard_normal((Hkv, cap, hd)).astype(np.float32)
    kn = rng.standard_normal((Hkv, C, hd)).astype(np.float32)
    vn = rng.standard_normal((Hkv, C, hd)).astype(np.float32)
    k2, v2, n = kv_append(k, v, P, kn, vn)
    assert n == P + C
    assert k2[:, P:P + C].tobytes() == kn.tobytes() and v2[:, P:P + C].tobytes() == vn.tobytes()
    for a, b in ((k2, k), (v2, v)):
        assert a[:, :P].tobytes() == b[:, :P].tobytes()
        assert a[:, P + C:].tobytes() == b[:, P + C:].tobytes()
    with pytest.raises(ValueError):
        kv_append(k, v, cap - C + 1, kn, vn)
