"""Block diffusion through the driver: several canvases, each denoised for a
few steps and then appended to the cache, checked step by step against the
oracle (teacher-forced: the oracle sees the same inputs and cache prefix)."""
import numpy as np
import pytest
import torch

import oracle
from canvas_denoising_gb300 import synth
from canvas_denoising_gb300.driver import CanvasDenoiser, generate
from tests.parity import FLAG_BUDGET, LSE_ABS, assert_rows_close, decision_flags

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().float().cpu().numpy() if t.dtype == torch.bfloat16 else t.detach().cpu().numpy()


@pytest.mark.parametrize("C,V,d,Hq,Hkv,P0,blocks,steps", [(128, 8192, 256, 4, 2, 256, 3, 2),
                                                          (256, 32768, 1024, 8, 4, 1024, 2, 2)])
def test_generate_matches_oracle_each_step(lib, C, V, d, Hq, Hkv, P0, blocks, steps):
    hd, thr, seed, alpha = 128, 0.3, 7, 6.0 if d == 256 else 26.0
    std = 0.1 if d == 256 else 0.02
    emb = synth.embedding(V, d, seed, std=std)
    k, v = synth.kv_prefix(Hkv, P0 + blocks * C, hd, P0, seed)
    emb_d, k_d, v_d = emb.cuda(), k.cuda(), v.cuda()
    mirror = {"k": _np(k), "v": _np(v), "blocks": 0}  # host copy of the cache, appended as the GPU appends
    den = CanvasDenoiser(emb_d, k_d, v_d, P0, C, Hq, thr, seed)
    inputs = {}

    def backbone(b, s, tokens, selfcond):
        q, kc, vc = synth.canvas_qkv(C, Hq, Hkv, hd, seed, block=b, step=s)
        h = synth.hidden(emb, synth.targets(C, V, seed, block=b), alpha, seed, block=b, step=s)
        inputs[(b, s)] = (q, kc, vc, h)
        return q.cuda(), kc.cuda(), vc.cuda(), h.cuda()

    stats = {"flagged": 0, "total": 0}

    def sync_mirror(upto):
        while mirror["blocks"] < upto:
            b0 = mirror["blocks"]
            _, kc0, vc0, _ = inputs[(b0, steps)]
            mirror["k"], mirror["v"], _ = oracle.kv_append(mirror["k"], mirror["v"], P0 + b0 * C, _np(kc0), _np(vc0))
            mirror["blocks"] += 1

    def on_step(b, s, dn):
        sync_mirror(b)
        assert dn.len == P0 + b * C
        q, kc, vc, h = inputs[(b, s)]
        o = dn.out
        ro, rl = oracle.canvas_attention(_np(q), mirror["k"], mirror["v"], dn.len, _np(kc), _np(vc))
        assert_rows_close(_np(o.attn_out).reshape(-1, hd), ro.reshape(-1, hd), what=f"attn b{b}s{s}")
        assert np.abs(_np(o.attn_lse) - rl).max() <= LSE_ABS
        rv = oracle.vocab_step(_np(h), _np(emb))
        assert_rows_close(_np(o.selfcond), rv["selfcond"], what=f"selfcond b{b}s{s}")
        tok, _ = oracle.renoise(rv["argmax"], rv["conf"].astype(np.float32), V, thr, seed, s, dn.len)
        fl = decision_flags(rv, thr)
        assert ((_np(dn.tokens) == tok) | fl).all(), f"tokens b{b}s{s}"
        stats["flagged"] += int(fl.sum())
        stats["total"] += C

    finished = generate(den, blocks, steps, backbone, on_step=on_step)
    torch.cuda.synchronize()
    assert len(finished) == blocks and den.len == P0 + blocks * C
    # the cache holds the prefix and every finished canvas's K/V, in order
    sync_mirror(blocks)
    np.testing.assert_array_equal(_np(k_d), mirror["k"])
    np.testing.assert_array_equal(_np(v_d), mirror["v"])
    assert stats["flagged"] <= FLAG_BUDGET * stats["total"]


def test_masked_diffusion_steps_match_oracle(lib):
    """Masked diffusion through the driver: a [MASK] canvas, each step unmasks
    the confident positions for good; checked step by step (teacher-forced)."""
    C, V, d, Hq, Hkv, hd, P0, steps = 128, 8192, 256, 4, 2, 128, 256, 4
    thr, seed, alpha, mask_id = 0.3, 11, 6.0, V - 1
    emb = synth.embedding(V, d, seed, std=0.1)
    k, v = synth.kv_prefix(Hkv, P0 + C, hd, P0, seed)
    den = CanvasDenoiser(emb.cuda(), k.cuda(), v.cuda(), P0, C, Hq, thr, seed, mask_id=mask_id)
    state = {"tok": np.full(C, mask_id, np.int32)}
    inputs = {}

    def backbone(b, s, tokens, selfcond):
        q, kc, vc = synth.canvas_qkv(C, Hq, Hkv, hd, seed, block=b, step=s)
        h = synth.hidden(emb, synth.targets(C, V, seed, block=b), alpha * (s + 1) / steps, seed, block=b, step=s)
        inputs[(b, s)] = h
        return q.cuda(), kc.cuda(), vc.cuda(), h.cuda()

    def on_step(b, s, dn):
        rv = oracle.vocab_step(_np(inputs[(b, s)]), _np(emb))
        ref, _ = oracle.unmask(state["tok"], rv["argmax"], rv["conf"].astype(np.float32), mask_id, thr)
        got = _np(dn.tokens)
        fl = decision_flags(rv, thr)
        assert ((got == ref) | fl).all(), f"masked tokens step {s}"
        # locked: a position that held a word keeps it
        held = state["tok"] != mask_id
        np.testing.assert_array_equal(got[held], state["tok"][held])
        state["tok"] = got  # teacher-forced: the oracle continues from the GPU's canvas

    generate(den, 1, steps, backbone, on_step=on_step)
    assert (state["tok"] != mask_id).sum() > 0


def test_early_stop_and_next_input(lib):
    """A canvas whose positions are all confident re-noises nothing at its
    first step, so early stop finishes it after one step; the next input is
    E[token] + S."""
    C, V, d, Hq, Hkv, hd, P0 = 64, 4096, 128, 4, 2, 128, 128
    thr, seed = 0.3, 3
    emb = synth.embedding(V, d, seed, std=0.3)
    k, v = synth.kv_prefix(Hkv, P0 + 2 * C, hd, P0, seed)
    den = CanvasDenoiser(emb.cuda(), k.cuda(), v.cuda(), P0, C, Hq, thr, seed)
    seen = {}

    def backbone(b, s, tokens, selfcond):
        q, kc, vc = synth.canvas_qkv(C, Hq, Hkv, hd, seed, block=b, step=s)
        alpha = 200.0 if b == 0 else 0.0  # block 0 certain, block 1 uniform
        h = synth.hidden(emb, synth.targets(C, V, seed, block=b), alpha, seed, block=b, step=s)
        seen[(b, s)] = h
        return q.cuda(), kc.cuda(), vc.cuda(), h.cuda()

    def on_step(b, s, dn):
        rv = oracle.vocab_step(_np(seen[(b, s)]), _np(emb))
        _, rn = oracle.renoise(rv["argmax"], rv["conf"].astype(np.float32), V, thr, seed, s, dn.len)
        assert dn.changed_positions() == int(rn.sum())
        x = dn.next_input()
        ref = oracle.selfcond_input(_np(dn.tokens), _np(emb), _np(dn.out.selfcond))
        assert_rows_close(_np(x), ref, what="next input")

    generate(den, 2, 3, backbone, on_step=on_step, early_stop=True)
    assert den.steps_taken == [1, 3]


def test_graphed_block_diffusion_matches_eager(lib):
    """One CUDA graph per canvas with the cache length on the device, replayed
    for every block, gives the eager host-length run's tokens and cache
    bytes, and attention within tolerance of the oracle."""
    from canvas_denoising_gb300.driver import GraphedBlockDiffusion
    C, V, d, Hq, Hkv, hd, P0, blocks, steps = 256, 8192, 256, 16, 8, 128, 512, 3, 3
    thr, seed, alpha = 0.3, 21, 6.0
    emb = synth.embedding(V, d, seed, std=0.1)
    cap = P0 + blocks * C
    k, v = synth.kv_prefix(Hkv, cap, hd, P0, seed)
    k[:, P0:] = 0  # rows past the prefix: finite (the device-length attention reads and masks them)
    v[:, P0:] = 0

    def inputs(b, s):
        q, kc, vc = synth.canvas_qkv(C, Hq, Hkv, hd, seed, block=b, step=s)
        h = synth.hidden(emb, synth.targets(C, V, seed, block=b), alpha, seed, block=b, step=s)
        return q, kc, vc, h

    # eager, host length
    ke, ve = k.cuda(), v.cuda()
    den = CanvasDenoiser(emb.cuda(), ke, ve, P0, C, Hq, thr, seed)

    def backbone(b, s, tokens, selfcond):
        return tuple(x.cuda() for x in inputs(b, s))

    eager = [t.cpu() for t in generate(den, blocks, steps, backbone)]
    # graphed, device length
    kg, vg = k.cuda(), v.cuda()
    stream = torch.cuda.Stream()
    gb = GraphedBlockDiffusion(emb.cuda(), kg, vg, P0, C, Hq, thr, seed, steps, stream)
    gb.capture()
    for b in range(blocks):
        per = [inputs(b, s) for s in range(steps + 1)]
        gb.load_block(torch.stack([p[0] for p in per[:steps]]).cuda(), torch.stack([p[1] for p in per]).cuda(),
                      torch.stack([p[2] for p in per]).cuda(), torch.stack([p[3] for p in per[:steps]]).cuda())
        tok = gb.run_block()
        stream.synchronize()
        np.testing.assert_array_equal(_np(tok), eager[b].numpy(), err_msg=f"block {b}")
        # the last step's attention, against the oracle over the cache as it stood
        q, kc, vc, _ = per[steps - 1]
        P = P0 + b * C
        ro, rl = oracle.canvas_attention(_np(q), _np(kg.cpu())[:, :P], _np(vg.cpu())[:, :P], P, _np(kc), _np(vc))
        assert_rows_close(_np(gb.out.attn_out).reshape(-1, hd), ro.reshape(-1, hd), what=f"graphed attn b{b}")
        assert np.abs(_np(gb.out.attn_lse) - rl).max() <= LSE_ABS
    assert int(gb.len_dev.item()) == P0 + blocks * C == den.len
    np.testing.assert_array_equal(_np(kg), _np(ke))
    np.testing.assert_array_equal(_np(vg), _np(ve))
    from canvas_denoising_gb300 import binding as B
    assert B.device_status() == B.DG_OK
