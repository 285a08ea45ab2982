"""Vocabulary steps and attention calls launched at once on separate
streams. The paired vocabulary kernel and the split attention kernel need all
of their CTAs resident together and are launched without the cooperative
attribute by default, so several such grids in flight must still each run to
completion (the grid dispatched first takes the SMs, the others follow) with
the results of a lone call and no expired wait."""
import pytest
import torch

from canvas_denoising_gb300 import binding as B
from canvas_denoising_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("V,d", [(65536, 2816), (32768, 1024)])
@pytest.mark.parametrize("n_streams", [2, 3])
def test_concurrent_vocab_steps_on_separate_streams(lib, V, d, n_streams):
    C, dev = 256, torch.device("cuda", 0)
    emb = synth.embedding(V, d, 4, device=dev)
    h = synth.hidden(emb, synth.targets(C, V, 4, device=dev), 11.0, 4)
    ref = [x.clone() for x in B.vocab_step(h, emb)]
    torch.cuda.synchronize()
    ws = [torch.empty(B.vocab_step_workspace_size(C, V, d), dtype=torch.uint8, device=dev) for _ in range(n_streams)]
    outs = [[torch.empty(C, dtype=torch.int32, device=dev), torch.empty(C, device=dev), torch.empty(C, device=dev),
             torch.empty((C, d), dtype=torch.bfloat16, device=dev)] for _ in range(n_streams)]
    streams = [torch.cuda.Stream() for _ in range(n_streams)]
    for _ in range(10):
        for k in range(n_streams):
            with torch.cuda.stream(streams[k]):
                B.vocab_step(h, emb, *outs[k], workspace=ws[k], stream=streams[k])
        torch.cuda.synchronize()
        assert B.device_status() == B.DG_OK
        for k in range(n_streams):
            for got, want in zip(outs[k], ref):
                assert torch.equal(got.view(torch.uint8) if got.dtype != torch.int32 else got,
                                   want.view(torch.uint8) if want.dtype != torch.int32 else want)


def _attn_inputs(P, seed, dev):
    C, Hq, Hkv, hd = 256, 16, 8, 128
    k, v = synth.kv_prefix(Hkv, P + C, hd, P, seed, device=dev)
    q, kn, vn = synth.canvas_qkv(C, Hq, Hkv, hd, seed, device=dev)
    return (q, k, v, P, kn, vn), torch.empty(max(256, B.canvas_attn_workspace_size(C, Hq, Hkv, hd, P)),
                                             dtype=torch.uint8, device=dev)


@pytest.mark.parametrize("mix", ["attn+attn", "attn+vocab"])
def test_concurrent_attention_on_separate_streams(lib, mix):
    dev = torch.device("cuda", 0)
    jobs = []  # (launch(stream), outputs, lone-call reference)
    for k in range(2):
        if mix == "attn+attn" or k == 0:
            args, ws = _attn_inputs(4096 if k == 0 else 2048, 7 + k, dev)
            ref = [x.clone() for x in B.canvas_attn(*args, workspace=ws)]
            out = [torch.empty_like(ref[0]), torch.empty_like(ref[1])]
            jobs.append((lambda st, a=args, w=ws, o=out: B.canvas_attn(*a, out=o[0], lse=o[1], workspace=w, stream=st),
                         out, ref))
        else:
            C, V, d = 256, 65536, 2816
            emb = synth.embedding(V, d, 4, device=dev)
            h = synth.hidden(emb, synth.targets(C, V, 4, device=dev), 11.0, 4)
            ref = [x.clone() for x in B.vocab_step(h, emb)]
            ws = torch.empty(B.vocab_step_workspace_size(C, V, d), dtype=torch.uint8, device=dev)
            out = [torch.empty(C, dtype=torch.int32, device=dev), torch.empty(C, device=dev),
                   torch.empty(C, device=dev), torch.empty((C, d), dtype=torch.bfloat16, device=dev)]
            jobs.append((lambda st, w=ws, o=out, hh=h, e=emb: B.vocab_step(hh, e, *o, workspace=w, stream=st), out, ref))
    torch.cuda.synchronize()
    assert B.device_status() == B.DG_OK
    streams = [torch.cuda.Stream() for _ in jobs]
    for _ in range(10):
        for (launch, _, _), st in zip(jobs, streams):
            with torch.cuda.stream(st):
                for _ in range(3):
                    launch(st)
        torch.cuda.synchronize()
        assert B.device_status() == B.DG_OK
        for _, out, ref in jobs:
            for got, want in zip(out, ref):
                assert torch.equal(got.view(torch.uint8) if got.dtype != torch.int32 else got,
                                   want.view(torch.uint8) if want.dtype != torch.int32 else want)
