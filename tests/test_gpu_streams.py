"""Vocabulary steps launched at once on separate streams. The paired kernel
needs all of its CTAs resident together and is launched without the
cooperative attribute by default, so two or three such grids in flight must
still each run to completion (the grid dispatched first takes the SMs, the
others follow) with the results of a lone call and no expired wait."""
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
