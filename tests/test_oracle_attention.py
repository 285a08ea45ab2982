"""Pins for the oracle's canvas attention (bidirectional denoising and
causal incremental prefill), against torch's float64 attention on CPU,
brute-force Python loops, closed forms and invariants."""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

from oracle.attention import canvas_attention


def _rand(shape, rng):
    return rng.standard_normal(shape)


def _case(rng, C=5, Hq=4, Hkv=2, hd=8, P=7, cap=None):
    cap = cap or P + C + 3
    q = _rand((C, Hq, hd), rng)
    kc = np.zeros((Hkv, cap, hd)); vc = np.zeros((Hkv, cap, hd))
    kc[:, :P] = _rand((Hkv, P, hd), rng); vc[:, :P] = _rand((Hkv, P, hd), rng)
    kcv = _rand((Hkv, C, hd), rng); vcv = _rand((Hkv, C, hd), rng)
    return q, kc, vc, P, kcv, vcv


def _torch_ref(q, kc, vc, P, kcv, vcv, causal):
    C, Hq, hd = q.shape
    Hkv = kcv.shape[0]
    K = torch.from_numpy(np.concatenate([kc[:, :P], kcv], 1))  # [Hkv][L][hd]
    Vv = torch.from_numpy(np.concatenate([vc[:, :P], vcv], 1))
    K = K.repeat_interleave(Hq // Hkv, 0)
    Vv = Vv.repeat_interleave(Hq // Hkv, 0)
    Q = torch.from_numpy(q).permute(1, 0, 2)  # [Hq][C][hd]
    mask = None
    if causal:
        L = P + C
        mask = torch.arange(L)[None, :] <= (P + torch.arange(C))[:, None]
    o = torch.nn.functional.scaled_dot_product_attention(Q[None], K[None], Vv[None], attn_mask=mask)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(5, 4, 2, 8, 7), (1, 2, 1, 4, 0), (9, 6, 3, 16, 20), (3, 2, 2, 4, 1)])
def test_matches_torch_float64(causal, shape):
    C, Hq, Hkv, hd, P = shape
    rng = np.random.default_rng(hash(shape) % 1000 + causal)
    q, kc, vc, P, kcv, vcv = _case(rng, C, Hq, Hkv, hd, P)
    out, lse = canvas_attention(q, kc, vc, P, kcv, vcv, causal=causal)
    ref = _torch_ref(q, kc, vc, P, kcv, vcv, causal)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_lse_matches_scipy_and_brute_force_loops():
    rng = np.random.default_rng(3)
    q, kc, vc, P, kcv, vcv = _case(rng, C=3, Hq=2, Hkv=1, hd=3, P=2)
    out, lse = canvas_attention(q, kc, vc, P, kcv, vcv)
    C, Hq, hd = q.shape
    scale = 1 / math.sqrt(hd)
    for h in range(Hq):
        keys = [kc[0, j] for j in range(P)] + [kcv[0, j] for j in range(C)]
        vals = [vc[0, j] for j in range(P)] + [vcv[0, j] for j in range(C)]
        for i in range(C):
            s = [sum(q[i, h, t] * k[t] for t in range(hd)) * scale for k in keys]
            assert abs(lse[h, i] - logsumexp(s)) < 1e-12
            mx = max(s)
            w = [math.exp(x - mx) for x in s]
            z = sum(w)
            o = [sum(w[j] * vals[j][t] for j in range(len(w))) / z for t in range(hd)]
            np.testing.assert_allclose(out[i, h], o, rtol=1e-12, atol=1e-13)


def test_single_key_returns_its_value():
    rng = np.random.default_rng(4)
    q, kc, vc, P, kcv, vcv = _case(rng, C=1, Hq=2, Hkv=1, hd=8, P=0)
    out, lse = canvas_attention(q, kc, vc, 0, kcv, vcv)
    for h in range(2):
        np.testing.assert_array_equal(out[0, h], vcv[0, 0])
        assert abs(lse[h, 0] - q[0, h] @ kcv[0, 0] / math.sqrt(8)) < 1e-12


def test_equal_keys_give_mean_value_and_log_length():
    rng = np.random.default_rng(5)
    C, Hq, Hkv, hd, P = 4, 2, 1, 8, 6
    q, kc, vc, P, kcv, vcv = _case(rng, C, Hq, Hkv, hd, P)
    k = rng.standard_normal(hd)
    kc[:, :P] = k
    kcv[:] = k
    out, lse = canvas_attention(q, kc, vc, P, kcv, vcv)
    allv = np.concatenate([vc[0, :P], vcv[0]], 0)
    for h in range(Hq):
        for i in range(C):
            np.testing.assert_allclose(out[i, h], allv.mean(0), rtol=1e-12, atol=1e-12)
            s = q[i, h] @ k / math.sqrt(hd)
            assert abs(lse[h, i] - (math.log(P + C) + s)) < 1e-12


def test_bidirectional_is_permutation_equivariant():
    rng = np.random.default_rng(6)
    q, kc, vc, P, kcv, vcv = _case(rng, C=8, Hq=4, Hkv=2, hd=8, P=5)
    out, lse = canvas_attention(q, kc, vc, P, kcv, vcv)
    perm = rng.permutation(8)
    out_p, lse_p = canvas_attention(q[perm], kc, vc, P, kcv[:, perm], vcv[:, perm])
    np.testing.assert_allclose(out_p, out[perm], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse_p, lse[:, perm], rtol=1e-12, atol=1e-12)


def test_causal_block_equals_full_causal_recompute():
    """Appending a block and running its causal attention equals rows
    [P, P+C) of causal attention over the whole sequence."""
    rng = np.random.default_rng(8)
    Hq, Hkv, hd, P, C = 4, 2, 8, 6, 5
    L = P + C
    Qall = rng.standard_normal((L, Hq, hd))
    Kall = rng.standard_normal((Hkv, L, hd))
    Vall = rng.standard_normal((Hkv, L, hd))
    cap = L + 2
    kc = np.zeros((Hkv, cap, hd)); vc = np.zeros((Hkv, cap, hd))
    kc[:, :P] = Kall[:, :P]; vc[:, :P] = Vall[:, :P]
    out, _ = canvas_attention(Qall[P:], kc, vc, P, Kall[:, P:], Vall[:, P:], causal=True)
    Q = torch.from_numpy(Qall).permute(1, 0, 2)[None]
    K = torch.from_numpy(Kall).repeat_interleave(Hq // Hkv, 0)[None]
    Vt = torch.from_numpy(Vall).repeat_interleave(Hq // Hkv, 0)[None]
    full = torch.nn.functional.scaled_dot_product_attention(Q, K, Vt, is_causal=True)[0].permute(1, 0, 2).numpy()
    np.testing.assert_allclose(out, full[P:], rtol=1e-12, atol=1e-12)


def test_causal_differs_from_bidirectional():
    rng = np.random.default_rng(9)
    q, kc, vc, P, kcv, vcv = _case(rng, C=4, Hq=2, Hkv=1, hd=8, P=3)
    a, _ = canvas_attention(q, kc, vc, P, kcv, vcv, causal=False)
    b, _ = canvas_attention(q, kc, vc, P, kcv, vcv, causal=True)
    np.testing.assert_allclose(a[-1], b[-1], rtol=1e-12)  # the last query sees everything either way
    assert np.abs(a[0] - b[0]).max() > 1e-3
