"""Failure detection without a GPU fault: a launch whose cross-CTA handshake
is withheld (a flag nothing sets) runs into its bounded waits, latches
DG_ERR_TIMEOUT, returns, and leaves the context usable for the next call."""
import numpy as np
import pytest
import torch

import oracle
from canvas_denoising_gb300 import binding as B
from canvas_denoising_gb300 import synth
from tests.parity import LSE_ABS, assert_rows_close

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().float().cpu().numpy() if t.dtype == torch.bfloat16 else t.detach().cpu().numpy()


def test_attention_withheld_arrival_times_out_then_recovers(lib):
    C, Hq, Hkv, hd, P = 256, 16, 8, 128, 4096
    k, v = synth.kv_prefix(Hkv, P + C, hd, P, seed=31, device="cuda")
    q, kn, vn = synth.canvas_qkv(C, Hq, Hkv, hd, seed=31, device="cuda")
    assert B.device_status() == B.DG_OK
    B.debug_inject(B.INJECT_ATTN_ARRIVAL, wait_ms=100)
    B.canvas_attn(q, k, v, P, kn, vn)
    assert B.device_status() == B.DG_ERR_TIMEOUT
    # the injection applied to one launch only; the next call is correct
    out, lse = B.canvas_attn(q, k, v, P, kn, vn)
    assert B.device_status() == B.DG_OK
    ro, rl = oracle.canvas_attention(_np(q), _np(k), _np(v), P, _np(kn), _np(vn))
    assert_rows_close(_np(out).reshape(C * Hq, hd), ro.reshape(C * Hq, hd), what="after recovery")
    assert np.abs(_np(lse) - rl).max() <= LSE_ABS


def test_vocab_withheld_tile_flag_times_out_then_recovers(lib):
    C, V, d = 256, 40000, 256
    emb = synth.embedding(V, d, seed=32, std=0.1)
    h = synth.hidden(emb, synth.targets(C, V, seed=32), 4.0, seed=32)
    hd_, ed = h.cuda(), emb.cuda()
    B.debug_inject(B.INJECT_VOCAB_READY, wait_ms=100)
    B.vocab_step(hd_, ed)
    assert B.device_status() == B.DG_ERR_TIMEOUT
    am, conf, lse, sc = B.vocab_step(hd_, ed)
    assert B.device_status() == B.DG_OK
    ref = oracle.vocab_step(_np(h), _np(emb))
    assert np.abs(_np(lse) - ref["lse"]).max() <= LSE_ABS
    assert_rows_close(_np(sc), ref["selfcond"], what="selfcond after recovery")


def test_injection_is_cleared(lib):
    B.debug_inject(B.INJECT_ATTN_ARRIVAL, wait_ms=100)
    B.debug_inject(B.INJECT_NONE)
    C, Hq, Hkv, hd, P = 64, 4, 2, 128, 1024
    k, v = synth.kv_prefix(Hkv, P + C, hd, P, seed=33, device="cuda")
    q, kn, vn = synth.canvas_qkv(C, Hq, Hkv, hd, seed=33, device="cuda")
    B.canvas_attn(q, k, v, P, kn, vn)
    assert B.device_status() == B.DG_OK
