"""Whole-canvas parity at the full shapes of the 262144-id workloads
(d = 2816, 16 query / 8 KV heads, head_dim 128): every canvas row and every
head, in the launch configuration the benchmark times (dg_canvas_attn and
dg_vocab_step_renoise, or their device-length forms inside the per-canvas
CUDA graph), against the float64 oracle, step after step.

Decisions (argmax, conf < threshold, re-noised tokens) must be identical
except at positions the oracle flags (top-2 probability gap at a kept
position, or |conf - threshold|, below 1e-3); flagged positions must stay
below 0.5% of all positions x steps of the workload. argmax is also compared
where the token is a draw, flagged there by a relative logit gap below 1e-3,
and may differ at no more than 0.5% of positions. Philox draws are bit-exact at every re-noised
position, flagged or not. Floats: per-row relative 2e-2 (attention output,
self-conditioning), 1e-2 absolute (log-sum-exp), 1e-2 relative (conf).

Each whole oracle step costs a few seconds of host time (the vocabulary
step is two float64 products over the 1.5 GB table), so these tests take
minutes; the workloads' step counts are run in full except where noted.
"""
import numpy as np
import pytest
import torch

import oracle
from canvas_denoising_gb300 import binding as B
from canvas_denoising_gb300 import synth
from canvas_denoising_gb300.configs import WORKLOADS
from tests.parity import (CONF_REL, FLAG_BUDGET, LSE_ABS, assert_rows_close, decision_flags, logit_gap_flags)

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().float().cpu().numpy() if t.dtype == torch.bfloat16 else t.detach().cpu().numpy()


class Tally:
    """Flagged positions (decisions) and argmax differences over all positions
    x steps of one workload."""

    def __init__(self):
        self.flagged = 0
        self.am_diff = 0
        self.total = 0

    def add(self, flags, am_diff):
        self.flagged += int(np.count_nonzero(flags))
        self.am_diff += int(np.count_nonzero(am_diff))
        self.total += flags.size

    def check(self):
        assert self.total > 0
        assert self.flagged <= FLAG_BUDGET * self.total, f"{self.flagged}/{self.total} positions flagged"
        assert self.am_diff <= max(1, int(FLAG_BUDGET * self.total)), f"argmax differs at {self.am_diff} rows"


def check_decisions(rv, thr, V, seed, step, pos0, tok, rn, am, tally, what):
    """Tokens and re-noise flags of one step against the oracle's statistics
    `rv` (all host arrays). Returns nothing; asserts."""
    C = tok.shape[0]
    fl = decision_flags(rv, thr)
    ref_tok, ref_rn = oracle.renoise(rv["argmax"], rv["conf"].astype(np.float32), V, thr, seed, step, pos0)
    assert ((tok == ref_tok) | fl).all(), f"{what}: tokens differ at {np.nonzero((tok != ref_tok) & ~fl)[0][:8]}"
    assert ((rn == ref_rn) | fl).all(), f"{what}: re-noise flags differ"
    # every re-noised position holds exactly its Philox draw, every kept one the step's argmax
    draw = oracle.uniform_token(seed, step, pos0 + np.arange(C), oracle.PHILOX_DOMAIN_RENOISE, V)
    low = rn.astype(bool)
    np.testing.assert_array_equal(tok[low], draw[low], err_msg=f"{what}: Philox draws")
    np.testing.assert_array_equal(tok[~low], am[~low], err_msg=f"{what}: kept positions")
    gap = logit_gap_flags(rv)
    assert ((am == rv["argmax"]) | fl | gap).all(), f"{what}: argmax differs at an unflagged row"
    tally.add(fl, am != rv["argmax"])


def check_stats(rv, conf, lse, what, sc=None):
    np.testing.assert_allclose(conf, rv["conf"], rtol=CONF_REL, err_msg=f"{what}: conf")
    assert np.abs(lse - rv["lse"]).max() <= LSE_ABS, f"{what}: lse"
    if sc is not None:
        assert_rows_close(sc, rv["selfcond"], what=f"{what}: selfcond")


def check_attention(out, lse, ro, rl, hd, what):
    assert_rows_close(out.reshape(-1, hd), ro.reshape(-1, hd), what=f"{what}: attention out")
    assert np.abs(lse - rl).max() <= LSE_ABS, f"{what}: attention lse"


def _resident(w):
    emb = synth.embedding(w.V, w.d, w.seed, device="cuda")
    tgt = synth.targets(w.C, w.V, w.seed, device="cuda")
    k, v = synth.kv_prefix(w.Hkv, w.cap, w.hd, w.prefix, w.seed, device="cuda")
    return emb, tgt, k, v


def _workspaces(w, prefix):
    wa = B.canvas_attn_workspace_size(w.C, w.Hq, w.Hkv, w.hd, prefix)
    wv = B.vocab_step_workspace_size(w.C, w.V, w.d)
    return (torch.empty(max(wa, 256), dtype=torch.uint8, device="cuda"),
            torch.empty(max(wv, 256), dtype=torch.uint8, device="cuda"))


def test_headline_workload_every_step(lib):
    """The 4096-token prefix workload: init, all 16 steps (attention +
    fused vocabulary step and re-noise, every row), then the append."""
    w = WORKLOADS["v262k_d2816_p4k"]
    thr, P = w.thresholds[0], w.prefix
    emb, tgt, k, v = _resident(w)
    emb_np, k_np, v_np = _np(emb), _np(k), _np(v)
    ws_a, ws_v = _workspaces(w, P)
    tokens = torch.empty(w.C, dtype=torch.int32, device="cuda")
    rn = torch.empty(w.C, dtype=torch.uint8, device="cuda")
    B.canvas_init(tokens, w.V, w.seed, P)
    np.testing.assert_array_equal(_np(tokens), oracle.canvas_init(w.C, w.V, w.seed, P))
    tally = Tally()
    for step in range(w.steps):
        q, kn, vn = synth.canvas_qkv(w.C, w.Hq, w.Hkv, w.hd, w.seed, step=step, device="cuda")
        h = synth.hidden(emb, tgt, w.alpha, w.seed, step=step)
        out, alse = B.canvas_attn(q, k, v, P, kn, vn, workspace=ws_a)
        am, conf, lse, sc = B.vocab_step_renoise(h, emb, tokens, thr, w.seed, step, P, renoised=rn, workspace=ws_v)
        torch.cuda.synchronize()
        what = f"step {step}"
        ro, rl = oracle.canvas_attention(_np(q), k_np, v_np, P, _np(kn), _np(vn))
        check_attention(_np(out), _np(alse), ro, rl, w.hd, what)
        rv = oracle.vocab_step(_np(h), emb_np)
        check_stats(rv, _np(conf), _np(lse), what, sc=_np(sc))
        check_decisions(rv, thr, w.V, w.seed, step, P, _np(tokens), _np(rn), _np(am), tally, what)
    tally.check()
    # the finished canvas's K/V go to cache rows [P, P + C); nothing else changes
    n, _, _ = B.kv_append(k, v, P, kn, vn)
    assert n == P + w.C
    ref_k, ref_v, _ = oracle.kv_append(k_np, v_np, P, _np(kn), _np(vn))
    np.testing.assert_array_equal(_np(k), ref_k)
    np.testing.assert_array_equal(_np(v), ref_v)
    assert B.device_status() == B.DG_OK


def test_long_context_threshold_sweep(lib):
    """The 32768-token prefix workload: all 32 steps, attention on every row
    and head, and the fused vocabulary step + re-noise at each of the four
    thresholds (the oracle's statistics serve all four)."""
    w = WORKLOADS["v262k_d2816_p32k"]
    P = w.prefix
    emb, tgt, k, v = _resident(w)
    emb_np, k_np, v_np = _np(emb), _np(k), _np(v)
    ws_a, ws_v = _workspaces(w, P)
    toks = {thr: torch.empty(w.C, dtype=torch.int32, device="cuda") for thr in w.thresholds}
    rns = {thr: torch.empty(w.C, dtype=torch.uint8, device="cuda") for thr in w.thresholds}
    tallies = {thr: Tally() for thr in w.thresholds}
    for thr in w.thresholds:
        B.canvas_init(toks[thr], w.V, w.seed, P)
    for step in range(w.steps):
        q, kn, vn = synth.canvas_qkv(w.C, w.Hq, w.Hkv, w.hd, w.seed, step=step, device="cuda")
        h = synth.hidden(emb, tgt, w.alpha, w.seed, step=step)
        out, alse = B.canvas_attn(q, k, v, P, kn, vn, workspace=ws_a)
        res = {thr: [_np(x) for x in B.vocab_step_renoise(h, emb, toks[thr], thr, w.seed, step, P,
                                                           renoised=rns[thr], workspace=ws_v)]
               for thr in w.thresholds}
        torch.cuda.synchronize()
        ro, rl = oracle.canvas_attention(_np(q), k_np, v_np, P, _np(kn), _np(vn))
        check_attention(_np(out), _np(alse), ro, rl, w.hd, f"step {step}")
        rv = oracle.vocab_step(_np(h), emb_np)
        for thr in w.thresholds:
            am, conf, lse, sc = res[thr]
            what = f"step {step} thr {thr}"
            check_stats(rv, conf, lse, what, sc=sc if thr == w.thresholds[0] else None)
            check_decisions(rv, thr, w.V, w.seed, step, P, _np(toks[thr]), _np(rns[thr]), am, tallies[thr], what)
    for thr in w.thresholds:
        tallies[thr].check()
    assert B.device_status() == B.DG_OK


def test_multiblock_graphed_against_oracle(lib):
    """8 canvases x 24 steps from a 2048-token prefix through the per-canvas
    CUDA graph with the cache length on the device (prefix 2048 -> 4096).
    Every canvas's initial tokens (the device-position canvas init) against
    the oracle's draws. Every step of every canvas: the Philox draw at each
    re-noised position
    (bit-exact), the argmax at each kept one, and the flags equal conf <
    threshold. The first and last step of every canvas: tokens, flags, conf,
    lse and attention lse against the oracle over the cache as it stood; the
    last step also the attention output and the self-conditioning vector.
    After the last canvas: the cache bytes."""
    from canvas_denoising_gb300.driver import GraphedBlockDiffusion
    w = WORKLOADS["multiblock_8x24"]
    thr, steps, P0 = w.thresholds[0], w.steps, w.prefix
    emb, _, k, v = _resident(w)
    emb_np = _np(emb)
    mirror_k, mirror_v = _np(k), _np(v)  # host copy of the cache, appended as the graph appends
    stream = torch.cuda.Stream()
    gb = GraphedBlockDiffusion(emb, k, v, P0, w.C, w.Hq, thr, w.seed, steps, stream, record=True)
    gb.capture()
    tally = Tally()
    checked = (0, steps - 1)
    for b in range(w.blocks):
        tgt = synth.targets(w.C, w.V, w.seed, block=b, device="cuda")
        per = []
        for s in range(steps + 1):
            q, kc, vc = synth.canvas_qkv(w.C, w.Hq, w.Hkv, w.hd, w.seed, block=b, step=s, device="cuda")
            h = synth.hidden(emb, tgt, w.alpha, w.seed, block=b, step=s)
            per.append((q, kc, vc, h))
        gb.load_block(torch.stack([p[0] for p in per[:steps]]), torch.stack([p[1] for p in per]),
                      torch.stack([p[2] for p in per]), torch.stack([p[3] for p in per[:steps]]))
        gb.run_block()
        stream.synchronize()
        P = P0 + b * w.C
        hist = {key: _np(t) for key, t in gb.history.items()}
        np.testing.assert_array_equal(hist["init"], oracle.canvas_init(w.C, w.V, w.seed, P),
                                      err_msg=f"canvas {b}: initial tokens")
        for s in range(steps):
            what = f"canvas {b} step {s}"
            tok, rn, am, conf = hist["tokens"][s], hist["renoised"][s], hist["argmax"][s], hist["conf"][s]
            low = rn.astype(bool)
            draw = oracle.uniform_token(w.seed, s, P + np.arange(w.C), oracle.PHILOX_DOMAIN_RENOISE, w.V)
            np.testing.assert_array_equal(tok[low], draw[low], err_msg=f"{what}: Philox draws")
            np.testing.assert_array_equal(tok[~low], am[~low], err_msg=f"{what}: kept positions")
            np.testing.assert_array_equal(low, conf < np.float32(thr), err_msg=f"{what}: flags vs conf")
            if s not in checked:
                continue
            q, kc, vc, h = per[s]
            ro, rl = oracle.canvas_attention(_np(q), mirror_k, mirror_v, P, _np(kc), _np(vc))
            assert np.abs(hist["attn_lse"][s] - rl).max() <= LSE_ABS, f"{what}: attention lse"
            rv = oracle.vocab_step(_np(h), emb_np)
            last = s == steps - 1
            check_stats(rv, conf, hist["lse"][s], what, sc=_np(gb.out.selfcond) if last else None)
            if last:
                assert_rows_close(_np(gb.out.attn_out).reshape(-1, w.hd), ro.reshape(-1, w.hd),
                                  what=f"{what}: attention out")
            check_decisions(rv, thr, w.V, w.seed, s, P, tok, rn, am, tally, what)
        mirror_k, mirror_v, _ = oracle.kv_append(mirror_k, mirror_v, P, _np(per[steps][1]), _np(per[steps][2]))
    tally.check()
    assert int(gb.len_dev.item()) == P0 + w.blocks * w.C
    np.testing.assert_array_equal(_np(k), mirror_k)
    np.testing.assert_array_equal(_np(v), mirror_v)
    assert B.device_status() == B.DG_OK
