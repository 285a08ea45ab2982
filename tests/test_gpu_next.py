"""GPU parity for the rows next to the step (self-conditioning input,
probability of the current token, masked-diffusion unmasking, canvas fill,
flag count, early stop) and for prompt-prefill shapes of the causal append,
against the float64 oracle on the same seeded bytes."""
import numpy as np
import pytest
import torch

import oracle
from canvas_denoising_gb300 import binding as B
from canvas_denoising_gb300 import synth
from tests.parity import CONF_REL, LSE_ABS, assert_rows_close

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().float().cpu().numpy() if t.dtype in (torch.bfloat16, torch.float16) else t.detach().cpu().numpy()


def _bf16_of(x64):
    """float64 -> bf16 values (round to nearest even through float32, which is
    exact here: a sum of two bf16 numbers fits in float32)."""
    return torch.from_numpy(np.asarray(x64, np.float32)).to(torch.bfloat16).float().numpy()


# ------------------------------------------------------------------ self-conditioning input
@pytest.mark.parametrize("C,V,d", [(256, 32768, 2816), (100, 1000, 264), (1, 64, 8)])
def test_selfcond_input_bf16(lib, C, V, d):
    emb = synth.embedding(V, d, seed=1)
    sc = synth.normal((C, d), seed=1, purpose="selfcond", std=0.02)
    tok = synth.randint(V, (C,), seed=1, purpose="tokens").to(torch.int32)
    x = B.selfcond_input(tok.cuda(), emb.cuda(), sc.cuda())
    ref = oracle.selfcond_input(tok.numpy(), _np(emb), _np(sc))
    assert_rows_close(_np(x), ref, what="selfcond input")
    exact = (_np(x) == _bf16_of(ref)).mean()
    assert exact >= 0.999, f"only {exact:.4%} of elements equal the rounded oracle sum"
    # without S: the embedding rows, bytewise
    x0 = B.selfcond_input(tok.cuda(), emb.cuda())
    assert x0.cpu().view(torch.int16).numpy().tobytes() == emb[tok.long()].view(torch.int16).numpy().tobytes()
    assert B.device_status() == B.DG_OK


def test_selfcond_input_f32_and_bad_token(lib):
    C, V, d = 33, 500, 36
    emb = synth.embedding(V, d, seed=2, dtype=torch.float32)
    sc = synth.normal((C, d), seed=2, purpose="selfcond", dtype=torch.float32)
    tok = synth.randint(V, (C,), seed=2, purpose="tokens").to(torch.int32)
    x = B.selfcond_input(tok.cuda(), emb.cuda(), sc.cuda())
    np.testing.assert_allclose(_np(x), oracle.selfcond_input(tok.numpy(), _np(emb), _np(sc)), rtol=1e-6, atol=1e-7)
    assert B.device_status() == B.DG_OK
    tok[5] = V  # out of range: a zero row and a latched bounds error
    x = B.selfcond_input(tok.cuda(), emb.cuda(), sc.cuda())
    assert B.device_status() == B.DG_ERR_DEVICE_BOUNDS
    assert (_np(x)[5] == 0).all()


# ------------------------------------------------------------------ probability of the current token
@pytest.mark.parametrize("C,V,d,alpha", [(256, 32768, 1024, 26.0), (200, 9000, 320, 6.0)])
def test_token_prob_end_to_end(lib, C, V, d, alpha):
    emb = synth.embedding(V, d, seed=3)
    tgt = synth.targets(C, V, seed=3)
    h = synth.hidden(emb, tgt, alpha, seed=3)
    am, conf, lse, _ = B.vocab_step(h.cuda(), emb.cuda())
    tok = synth.randint(V, (C,), seed=3, purpose="tokens").to(torch.int32)
    tok[::3] = tgt[::3].to(torch.int32)  # some rows hold the likely token
    prob = B.token_prob(h.cuda(), emb.cuda(), tok.cuda(), lse)
    ref_v = oracle.vocab_step(_np(h), _np(emb), want_top2=False)
    ref = oracle.token_prob(_np(h), _np(emb), tok.numpy(), ref_v["lse"])
    # lse within 1e-2 absolute bounds the relative error of exp(logit - lse)
    np.testing.assert_allclose(_np(prob), ref, rtol=CONF_REL, atol=1e-30)
    # the argmax's probability is the confidence
    p_am = B.token_prob(h.cuda(), emb.cuda(), am, lse)
    np.testing.assert_allclose(_np(p_am), _np(conf), rtol=1e-4)
    assert B.device_status() == B.DG_OK


def test_token_prob_kernel_alone_f32(lib):
    C, V, d = 40, 700, 52
    emb = synth.embedding(V, d, seed=4, dtype=torch.float32, std=0.3)
    h = synth.normal((C, d), seed=4, purpose="h", dtype=torch.float32)
    tok = synth.randint(V, (C,), seed=4, purpose="tokens").to(torch.int32)
    ref_v = oracle.vocab_step(_np(h), _np(emb), want_top2=False)
    lse = torch.from_numpy(ref_v["lse"].astype(np.float32))
    prob = B.token_prob(h.cuda(), emb.cuda(), tok.cuda(), lse.cuda())
    np.testing.assert_allclose(_np(prob), oracle.token_prob(_np(h), _np(emb), tok.numpy(), lse.numpy()), rtol=1e-5)


# ------------------------------------------------------------------ masked diffusion, fill, count
@pytest.mark.parametrize("C,thr", [(256, 0.5), (1000, 0.3), (7, 0.0), (256, 1.5)])
def test_unmask_bit_exact(lib, C, thr):
    g = torch.Generator().manual_seed(C)
    mask_id = 262143
    tok = torch.randint(0, 1000, (C,), generator=g, dtype=torch.int32)
    tok[torch.rand(C, generator=g) < 0.6] = mask_id
    am = torch.randint(0, 1000, (C,), generator=g, dtype=torch.int32)
    conf = torch.rand(C, generator=g, dtype=torch.float32)
    conf[: min(5, C)] = thr if thr <= 1 else 0.5  # equality unmasks
    td = tok.cuda()
    flags = torch.zeros(C, dtype=torch.uint8, device="cuda")
    B.unmask(td, am.cuda(), conf.cuda(), mask_id, thr, unmasked=flags)
    ref_tok, ref_flag = oracle.unmask(tok.numpy(), am.numpy(), conf.numpy(), mask_id, thr)
    np.testing.assert_array_equal(_np(td), ref_tok)
    np.testing.assert_array_equal(_np(flags), ref_flag)
    cnt = B.count_flags(flags)
    assert int(cnt.item()) == int(ref_flag.sum())


def test_canvas_fill_and_count(lib):
    for C in (1, 256, 1000):
        tok = torch.empty(C, dtype=torch.int32, device="cuda")
        B.canvas_fill(tok, 262143)
        np.testing.assert_array_equal(_np(tok), oracle.canvas_fill(C, 262143))
        f = (torch.arange(C, device="cuda") % 3 == 0).to(torch.uint8)
        assert int(B.count_flags(f).item()) == (C + 2) // 3
        z = torch.zeros(C, dtype=torch.uint8, device="cuda")
        assert int(B.count_flags(z).item()) == 0 and oracle.finished_early(_np(z))


# ------------------------------------------------------------------ prompt prefill shapes
@pytest.mark.parametrize("P,C", [(0, 2048), (1024, 2048), (0, 520), (0, 4096)])
def test_prefill_shapes_causal_append(lib, P, C):
    """Incremental causal prefill of a whole prompt chunk (the step before the
    denoising loop): a C-row block appended at P, with its causal attention."""
    Hkv, Hq, hd = 8, 16, 128
    cap = P + C
    k, v = synth.kv_prefix(Hkv, cap, hd, P, seed=5)
    q, kn, vn = synth.canvas_qkv(C, Hq, Hkv, hd, seed=5)
    kd, vd = k.cuda(), v.cuda()
    n, out, lse = B.kv_append(kd, vd, P, kn.cuda(), vn.cuda(), q_new=q.cuda())
    assert n == P + C
    assert kd[:, P:P + C].cpu().view(torch.int16).numpy().tobytes() == kn.view(torch.int16).numpy().tobytes()
    ro, rl = oracle.canvas_attention(_np(q), _np(k), _np(v), P, _np(kn), _np(vn), causal=True)
    assert_rows_close(_np(out).reshape(C * Hq, hd), ro.reshape(C * Hq, hd), what="prefill out")
    assert np.abs(_np(lse) - rl).max() <= LSE_ABS
    assert B.device_status() == B.DG_OK


# ------------------------------------------------------------------ device-side cache length
def test_devlen_attention_matches_host_length(lib):
    """dg_canvas_attn_devlen at every prefix a growing cache passes through
    equals the oracle (rows past the prefix hold finite stale data)."""
    C, Hq, Hkv, hd, Pmax = 256, 16, 8, 128, 2048
    k, v = synth.kv_prefix(Hkv, Pmax + C, hd, Pmax, seed=41)
    q, kn, vn = synth.canvas_qkv(C, Hq, Hkv, hd, seed=41)
    kd, vd = k.cuda(), v.cuda()
    for P in (0, 512, 1300, Pmax):
        pdev = torch.tensor([P], dtype=torch.int64, device="cuda")
        for mask in (B.DG_MASK_BIDIR, B.DG_MASK_CAUSAL_BLOCK):
            out, lse = B.canvas_attn_devlen(q.cuda(), kd, vd, pdev, Pmax, kn.cuda(), vn.cuda(), mask=mask)
            ro, rl = oracle.canvas_attention(_np(q), _np(k), _np(v), P, _np(kn), _np(vn),
                                             causal=mask == B.DG_MASK_CAUSAL_BLOCK)
            assert_rows_close(_np(out).reshape(C * Hq, hd), ro.reshape(C * Hq, hd), what=f"devlen P={P} m={mask}")
            assert np.abs(_np(lse) - rl).max() <= LSE_ABS
    assert B.device_status() == B.DG_OK
    # a device prefix beyond the planned maximum is clamped and reported
    pdev = torch.tensor([Pmax + 7], dtype=torch.int64, device="cuda")
    B.canvas_attn_devlen(q.cuda(), kd, vd, pdev, Pmax, kn.cuda(), vn.cuda())
    assert B.device_status() == B.DG_ERR_DEVICE_BOUNDS


def test_devlen_append_and_bounds(lib):
    Hkv, hd, C, cap = 4, 128, 64, 200
    k = torch.zeros((Hkv, cap, hd), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    kn = synth.normal((Hkv, C, hd), seed=42, purpose="k_canvas").cuda()
    vn = synth.normal((Hkv, C, hd), seed=42, purpose="v_canvas").cuda()
    ln = torch.tensor([10], dtype=torch.int64, device="cuda")
    B.kv_append_devlen(k, v, ln, kn, vn)
    B.kv_append_devlen(k, v, ln, kn, vn)
    assert int(ln.item()) == 10 + 2 * C
    assert torch.equal(k[:, 10:10 + C], kn) and torch.equal(v[:, 10 + C:10 + 2 * C], vn)
    assert B.device_status() == B.DG_OK
    before = k.clone()
    B.kv_append_devlen(k, v, ln, kn, vn)  # 138 + 64 > 200: nothing written, length unchanged
    assert B.device_status() == B.DG_ERR_DEVICE_BOUNDS
    assert int(ln.item()) == 10 + 2 * C and torch.equal(k, before)


def test_large_prefill_chunk_is_causal(lib):
    """A 16384-row prompt chunk (2048 CTAs, more than fit at once): row i sees
    only keys 0..i, so its first 2048 rows equal the 2048-row chunk's, which
    the oracle test above checks; the lse agree as well."""
    Hkv, Hq, hd, C, Cs = 8, 16, 128, 16384, 2048
    k, v = synth.kv_prefix(Hkv, C, hd, 0, seed=43, device="cuda")
    q, kn, vn = synth.canvas_qkv(C, Hq, Hkv, hd, seed=43, device="cuda")
    _, out, lse = B.kv_append(k, v, 0, kn, vn, q_new=q)
    k2, v2 = synth.kv_prefix(Hkv, Cs, hd, 0, seed=43, device="cuda")
    _, out_s, lse_s = B.kv_append(k2, v2, 0, kn[:, :Cs].contiguous(), vn[:, :Cs].contiguous(),
                                  q_new=q[:Cs].contiguous())
    assert_rows_close(_np(out[:Cs]).reshape(Cs * Hq, hd), _np(out_s).reshape(Cs * Hq, hd), tol=1e-2,
                      what="prefix rows")
    assert np.abs(_np(lse[:, :Cs]) - _np(lse_s)).max() <= 1e-3
    assert np.isfinite(_np(out)).all() and np.isfinite(_np(lse)).all()
    assert B.device_status() == B.DG_OK
